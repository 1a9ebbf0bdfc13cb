"""Parity of the decode step with the K and V rows in page-locked host memory.

The CompKV page keeps the KV cache and the block summaries in pinned CPU
memory and moves the selected blocks to the GPU each step (section "어떻게
쓰나").  On a GB300 the GPU reads host memory directly over its chip-to-chip
link, so this variant keeps only the bf16 K/V rows in host memory: the
summaries, the scratch and everything the summary stream reads stay in GPU
memory, and the post kernel copies each selected block over the link.  The
library recognises host K/V from the pointers at init.  Same oracle, same
tolerances as the device-memory tests.
"""
import numpy as np
import pytest
import torch

import synth
from harness import Run, check_step, check_summaries

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import block_sparse_kv_summary_gb300 as P
    P.build()
    P.lib()


def _ragged(shape, lengths, budget, steps):
    return synth.Workload("ragged-host", 1, len(lengths), shape["num_kv_heads"], shape["group_size"],
                          shape["head_dim"], shape["r"], 0, budget, steps, lengths=tuple(lengths))


def test_tiny_workload_host_kv():
    wl = synth.WORKLOADS["tiny"]
    run = Run(wl, kv_memory="host")
    assert run.cache.k.device.type == "cpu" and run.cache.k.is_pinned()
    q, sel, out, res = run.decode_step(0)
    check_step(run, 0, sel, out, res)
    for (l, s, h) in run.heads:
        check_summaries(run, l, s, h)
    assert run.cache.device_status() == 0


@pytest.mark.parametrize("shape", [dict(head_dim=128, group_size=4, r=4, num_kv_heads=2),
                                   dict(head_dim=64, group_size=8, r=64, num_kv_heads=1),
                                   dict(head_dim=128, group_size=1, r=1, num_kv_heads=2)],
                         ids=lambda s: f"d{s['head_dim']}G{s['group_size']}r{s['r']}")
def test_ragged_steps_host_kv(shape):
    # partial blocks, N <= K, several attention rounds (budget 4096: K = 256)
    wl = _ragged(shape, lengths=(1, 37, 2049, 9000), budget=4096 if shape["group_size"] == 4 else 128, steps=18)
    run = Run(wl, kv_memory="host")
    for step in range(wl.steps):
        q, sel, out, res = run.decode_step(0)
        check_step(run, 0, sel, out, res)
    for (l, s, h) in run.heads:
        check_summaries(run, l, s, h)
    assert run.cache.seq_len.cpu().tolist() == [[L + wl.steps for L in wl.lengths]]
    assert run.cache.device_status() == 0


def test_host_kv_matches_device_kv():
    # the same cache and queries in both placements: identical selections, outputs within 1e-5
    wl = _ragged(dict(head_dim=128, group_size=4, r=4, num_kv_heads=3), lengths=(300, 5000, 20000), budget=512,
                 steps=4)
    dev = Run(wl)
    host = Run(wl, kv_memory="host")
    for step in range(wl.steps):
        qd, seld, outd, resd = dev.decode_step(0)
        qh, selh, outh, resh = host.decode_step(0)
        assert torch.equal(qd, qh)
        assert torch.equal(seld, selh)
        assert (outd - outh).abs().max().item() <= 1e-5
        check_step(host, 0, selh, outh, resh)
    assert dev.cache.device_status() == 0 and host.cache.device_status() == 0
