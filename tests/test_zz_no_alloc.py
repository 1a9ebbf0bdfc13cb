"""The scratch-free decode entry point, checked against the regular one.

compkv_decode_static is for callers that cannot allocate device memory when
they decode (for example an engine that handed the whole GPU to its cache pool
at start-up and gives plug-ins no allocator).  It runs the same decode step
as compkv_decode but keeps its scratch in a fixed device array inside the
library.  Two identical caches are advanced by two decode steps in a row, one
through each entry point, and must agree: identical selections, outputs
within the 2e-3 tolerance the parity tests use, the same lengths afterwards.
This file is collected last so that a failure here cannot hide another test.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import block_sparse_kv_summary_gb300 as P
    P.build()
    P.lib()


def _cache_pair(wl):
    from block_sparse_kv_summary_gb300.cache import CompKVCache
    lens, caps = synth.sequence_lengths(wl), synth.capacity_tokens(wl)
    caches, future = [], {}
    for _ in range(2):
        c = CompKVCache(num_layers=1, batch=wl.batch, num_kv_heads=wl.num_kv_heads, group_size=wl.group_size,
                        head_dim=wl.head_dim, r=wl.r, budget_tokens=wl.budget_tokens, capacity_tokens=caps,
                        device="cuda")
        for s in range(wl.batch):
            K, V = synth.sequence_tokens(wl, 0, s, caps[s], lens[s], device="cuda")
            for h in range(wl.num_kv_heads):
                kv, vv = c.token_view(0, s, h)
                kv[:lens[s]] = K[h, :lens[s]]
                vv[:lens[s]] = V[h, :lens[s]]
            future[s] = (K[:, lens[s]:lens[s] + wl.steps], V[:, lens[s]:lens[s] + wl.steps])
        c.prefill(0, lens)
        caches.append(c)
    torch.cuda.synchronize()
    return caches, future


def test_static_scratch_matches_regular_decode_twice():
    from block_sparse_kv_summary_gb300 import compkv as C
    wl = synth.Workload("static", 1, 3, 2, 4, 128, 4, 0, 128, 2, lengths=(37, 2049, 4100))
    (reg, sta), future = _cache_pair(wl)
    stream = torch.cuda.current_stream().cuda_stream
    for step in range(2):
        q = torch.from_numpy(synth.step_queries(wl, 0, step)).cuda()
        k_new = torch.stack([future[s][0][:, step] for s in range(wl.batch)]).contiguous()
        v_new = torch.stack([future[s][1][:, step] for s in range(wl.batch)]).contiguous()
        out_r, sel_r = reg.new_out(), reg.new_sel()
        reg.decode(0, q, k_new, v_new, out=out_r, sel=sel_r)
        out_s = torch.full_like(out_r, float("nan"))
        sel_s = torch.full_like(sel_r, -7)
        C.compkv_decode_static(sta.cfg, sta.bufs, 0, q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                               out_s.data_ptr(), sel_s.data_ptr(), stream)
        torch.cuda.synchronize()
        assert torch.equal(sel_r, sel_s), f"step {step}: selections differ"
        err = (out_r.double() - out_s.double()).abs().max().item()
        assert np.isfinite(err) and err <= 2e-3, f"step {step}: outputs differ by {err}"
        assert torch.equal(reg.seq_len, sta.seq_len)
    assert reg.device_status() == 0


def test_static_scratch_rejects_a_configuration_that_does_not_fit():
    from block_sparse_kv_summary_gb300 import compkv as C
    cfg = C.make_config(1, 16, 8, 4, 128, 4, 1024, max_tokens=131088)
    assert C.compkv_scratch_bytes(cfg) > C.COMPKV_STATIC_SCRATCH_BYTES
    bufs = C.compkv_buffers(256, 256, 256, 256, 256, 256, 0, 0)
    with pytest.raises(C.CompKVError, match="static scratch holds"):
        C.compkv_decode_static(cfg, bufs, 0, 256, 256, 256, 256, 0, None)


_FRESH = r'''
import sys, torch
sys.path.insert(0, sys.argv[1])
import block_sparse_kv_summary_gb300 as P
from block_sparse_kv_summary_gb300 import compkv as C
P.lib()
# no context is ever initialised in this process: the entry point sets up the kernels itself
d, G = 128, 4
cfg = C.make_config(1, 1, 1, G, d, 4, 2048, capacity_tokens=[4096])
rows = C.compkv_rows_per_layer(cfg)
dev = torch.device("cuda", 0)
k = torch.zeros((rows, 16, d), dtype=torch.bfloat16, device=dev)
v = torch.zeros((rows, 16, d), dtype=torch.bfloat16, device=dev)
kbar = torch.zeros((rows, d), dtype=torch.float32, device=dev)
vbar = torch.zeros((rows, d), dtype=torch.float32, device=dev)
dbar = torch.zeros((rows, 4), dtype=torch.float32, device=dev)
seq_len = torch.zeros((1, 1), dtype=torch.int32, device=dev)
bufs = C.compkv_buffers(k.data_ptr(), v.data_ptr(), kbar.data_ptr(), vbar.data_ptr(), dbar.data_ptr(),
                        seq_len.data_ptr(), 0, 0)
g = torch.Generator().manual_seed(7)
q = torch.randn((1, G, d), generator=g).to(dev)
k_new = torch.randn((1, 1, d), generator=g).to(torch.bfloat16).to(dev)
v_new = torch.randn((1, 1, d), generator=g).to(torch.bfloat16).to(dev)
out = torch.full((1, G, d), float("nan"), device=dev)
sel = torch.full((1, 1, 128), -7, dtype=torch.int32, device=dev)
C.compkv_decode_static(cfg, bufs, 0, q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), out.data_ptr(),
                       sel.data_ptr(), torch.cuda.current_stream().cuda_stream)
torch.cuda.synchronize()
# one token in the cache: softmax over it is 1, so every head's output is its value row
want = v_new[0, 0].float().expand(G, d)
assert torch.equal(out[0], want), (out[0] - want).abs().max().item()
assert sel[0, 0, 0].item() == 0 and bool((sel[0, 0, 1:] == -1).all())
assert seq_len.item() == 1
print("fresh process ok")
'''


def test_static_scratch_in_a_process_without_a_context():
    # compkv_decode_static must work as the first and only call of a process: it sets the
    # kernels' shared-memory limits itself (compkv_init does this for the other entry points)
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH, root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "fresh process ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
