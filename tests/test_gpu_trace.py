"""The work-item trace: a traced decode call computes exactly what an untraced one does.

With a trace buffer set, both decode kernels run as their traced instances
(separate compiled code that also records timestamps).  Two identical caches
take the same two decode steps, one traced and one not.  The traced cache
must give identical selections and bit-identical outputs, and its records
must follow the layout include/compkv.h documents:
- one record per stream CTA, with its start <= plan <= end;
- one per CTA of the second kernel, with every unit present at every cluster
  rank 0..C-1, its start <= wait end <= attention done <= end;
- the unit's selected block count, min(K, N).
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


def test_traced_decode_matches_untraced():
    from block_sparse_kv_summary_gb300 import compkv as C
    # ragged lengths: a sequence with N <= K, partial blocks, several segments per unit
    wl = synth.Workload("trace", 1, 3, 2, 4, 128, 4, 0, 512, 2, lengths=(37, 2049, 9000))
    (plain, traced), future = _cache_pair(wl)
    units = wl.batch * wl.num_kv_heads
    K = wl.budget_tokens // 16
    buf = torch.zeros(1 + 8 * 8192, dtype=torch.int64, device="cuda")
    C.compkv_trace(traced.ctx, buf.data_ptr(), buf.numel() * 8)
    try:
        for step in range(2):
            q = torch.from_numpy(synth.step_queries(wl, 0, step)).cuda()
            k_new = torch.stack([future[s][0][:, step] for s in range(wl.batch)]).contiguous()
            v_new = torch.stack([future[s][1][:, step] for s in range(wl.batch)]).contiguous()
            buf.zero_()
            out_p, sel_p = plain.new_out(), plain.new_sel()
            out_t, sel_t = traced.new_out(), traced.new_sel()
            plain.decode(0, q, k_new, v_new, out=out_p, sel=sel_p)
            traced.decode(0, q, k_new, v_new, out=out_t, sel=sel_t)
            torch.cuda.synchronize()
            assert torch.equal(sel_p, sel_t), f"step {step}: selections differ"
            assert torch.equal(out_p, out_t), f"step {step}: outputs differ"
            assert torch.equal(plain.seq_len, traced.seq_len)

            tr = buf.cpu().numpy()[1:].reshape(-1, 8).astype(np.int64)
            used = tr[:, 2] != 0
            kind = (tr[:, 0] >> 24) & 0xFF
            srec, prec = tr[used & (kind == 0)], tr[used & (kind == 1)]
            assert len(srec) > 0
            assert (srec[:, 2] <= srec[:, 3]).all() and (srec[:, 3] <= srec[:, 5]).all()
            # every unit at every rank 0..C-1, once
            unit, rank = prec[:, 1], prec[:, 0] & 0xFFFFFF
            C_ = len(prec) // units
            assert len(prec) == units * C_ and C_ >= 1
            pairs = set(zip(unit.tolist(), rank.tolist()))
            assert pairs == {(u, p) for u in range(units) for p in range(C_)}
            assert (prec[:, 2] <= prec[:, 3]).all() and (prec[:, 3] <= prec[:, 4]).all()
            assert (prec[:, 4] <= prec[:, 6]).all()
            L = plain.seq_len.cpu().numpy()[0]
            for u, cnt in zip(unit.tolist(), prec[:, 7].tolist()):
                N = (int(L[u // wl.num_kv_heads]) + 15) // 16
                assert cnt == min(K, N), (u, cnt, N)
    finally:
        C.compkv_trace(traced.ctx, 0, 0)
    assert plain.device_status() == 0 and traced.device_status() == 0
