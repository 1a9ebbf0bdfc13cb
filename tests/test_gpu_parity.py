"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, small sizes.

Selections must match bit for bit (inputs carry the 1e-4 score-gap
guarantee), summaries and scores within 1e-4 relative, attention outputs
within 2e-3 absolute.  Sizes span several 64-block scoring items with a
ragged tail, partial last blocks, N <= K, N < 3, and every (d, G, r) family.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from harness import (TOL_OUT, Run, check_scores, check_step, check_summaries, f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import block_sparse_kv_summary_gb300 as P
    P.build()
    P.lib()


def test_tiny_workload_decode():
    wl = synth.WORKLOADS["tiny"]
    run = Run(wl)
    for (l, s, h) in run.heads:
        check_summaries(run, l, s, h)
    q, sel, out, res = run.decode_step(0)
    check_step(run, 0, sel, out, res)
    for (l, s, h) in run.heads:
        check_summaries(run, l, s, h)
    assert run.cache.seq_len.cpu().tolist() == [[1025]]
    assert run.cache.device_status() == 0
    # the planted needles (soft check: reported, not pinned)
    hits = 0
    for h in range(wl.num_kv_heads):
        pos = synth.workloads.needle_positions(wl, 0, 0, h, 1024)
        hits += sum(p // 16 in set(res[(0, h)].sel.tolist()) for p in pos)
    print(f"needle blocks selected: {hits} of {3 * wl.num_kv_heads}")


SHAPES = [
    dict(head_dim=64, group_size=4, r=4, num_kv_heads=2),
    dict(head_dim=128, group_size=4, r=4, num_kv_heads=3),
    dict(head_dim=128, group_size=8, r=128, num_kv_heads=2),
    dict(head_dim=128, group_size=1, r=1, num_kv_heads=2),
    dict(head_dim=128, group_size=2, r=2, num_kv_heads=1),
    dict(head_dim=64, group_size=8, r=64, num_kv_heads=1),
    dict(head_dim=128, group_size=4, r=16, num_kv_heads=2),
    dict(head_dim=128, group_size=4, r=64, num_kv_heads=2),  # long Dbar rows, two coordinates per lane
]


def _ragged(shape, lengths=(1, 37, 2049, 4100), budget=128, steps=18):
    return synth.Workload("ragged", 1, len(lengths), shape["num_kv_heads"], shape["group_size"],
                          shape["head_dim"], shape["r"], 0, budget, steps, lengths=tuple(lengths))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"d{s['head_dim']}G{s['group_size']}r{s['r']}")
def test_decode_ragged_steps(shape):
    wl = _ragged(shape)
    run = Run(wl)
    for (l, s, h) in run.heads:
        check_summaries(run, l, s, h)
    for step in range(wl.steps):
        q, sel, out, res = run.decode_step(0)
        check_step(run, 0, sel, out, res)
    for (l, s, h) in run.heads:
        check_summaries(run, l, s, h)
    assert run.cache.seq_len.cpu().tolist() == [[L + wl.steps for L in wl.lengths]]
    assert run.cache.device_status() == 0


@pytest.mark.parametrize("budget", [48, 64, 256])
def test_budgets_and_forced_only(budget):
    # K = 3 selects only the forced blocks; larger budgets span several attention items
    wl = _ragged(SHAPES[1], lengths=(5, 600, 1800), budget=budget, steps=3)
    run = Run(wl)
    for step in range(wl.steps):
        q, sel, out, res = run.decode_step(0)
        check_step(run, 0, sel, out, res)


def test_budget_above_one_round():
    # K = 256 blocks: 16 CTAs per unit, each attends two rounds of 8 blocks
    wl = _ragged(SHAPES[1], lengths=(5, 1800, 9000), budget=4096, steps=3)
    run = Run(wl)
    for step in range(wl.steps):
        q, sel, out, res = run.decode_step(0)
        check_step(run, 0, sel, out, res)
    assert run.cache.device_status() == 0


def test_score_select_api_scores():
    wl = _ragged(SHAPES[1], lengths=(70, 3000, 5000), budget=256, steps=2)
    run = Run(wl)
    run.decode_step(0)
    # score the current cache with fresh queries through compkv_score_select
    k_new, v_new = run.new_tokens(0, 1)
    run.oracle_append(0, k_new, v_new)
    run.cache.append(0, k_new, v_new)
    q, results = run.choose_queries(0, 1)
    scores = torch.zeros((wl.batch, wl.num_kv_heads, run.cache.max_cap_blocks), device="cuda")
    sel = run.cache.score_select(0, q, scores=scores)
    S = f64(scores)
    for (s, h), res in results.items():
        N = len(res.scores.S)
        check_scores(S[s, h, :N], res.scores.S)
        exp = np.full(wl.K_blocks, -1)
        exp[:len(res.sel)] = res.sel
        assert np.array_equal(sel[s, h].cpu().numpy(), exp)
    assert run.cache.device_status() == 0


def test_attend_api_arbitrary_selections():
    wl = _ragged(SHAPES[2], lengths=(3, 200, 1000, 3000), budget=160, steps=1)
    run = Run(wl)
    rng = np.random.default_rng(5)
    K = wl.K_blocks
    for trial in range(4):
        q = torch.from_numpy(synth.step_queries(wl, 0, 100 + trial)).cuda()
        sel = np.full((wl.batch, wl.num_kv_heads, K), -1, dtype=np.int32)
        for (l, s, h), st in run.states.items():
            N = O.num_blocks(st.L)
            cnt = [0, min(N, K), min(N, 1), int(rng.integers(0, min(N, K) + 1))][trial]
            pick = np.sort(rng.choice(N, size=cnt, replace=False))
            sel[s, h, :cnt] = pick
        sel_t = torch.from_numpy(sel).cuda()
        out = f64(run.cache.attend(0, q, sel_t))
        qh = q.cpu().numpy().astype(np.float64)
        G = wl.group_size
        for (l, s, h), st in run.states.items():
            chosen = [b for b in sel[s, h] if b >= 0]
            ref = O.compkv_attend(qh[s, h * G:(h + 1) * G], st.K[:st.L], st.V[:st.L], chosen, st.n, st.kbar, st.vbar)
            assert np.abs(out[s, h * G:(h + 1) * G] - ref).max() <= TOL_OUT
    assert run.cache.device_status() == 0


def test_append_api_matches_oracle():
    wl = _ragged(SHAPES[0], lengths=(14, 16, 31), budget=64, steps=20)
    run = Run(wl)
    for step in range(wl.steps):
        k_new, v_new = run.new_tokens(0, step)
        run.oracle_append(0, k_new, v_new)
        run.cache.append(0, k_new, v_new)
        torch.cuda.synchronize()
        for (l, s, h), st in run.states.items():
            N = O.num_blocks(st.L)
            check_summaries(run, l, s, h, blocks=[N - 1])
            kv, vv = run.cache.token_view(l, s, h)
            assert np.array_equal(f64(kv[st.L - 1]), st.K[st.L - 1])
            assert np.array_equal(f64(vv[st.L - 1]), st.V[st.L - 1])
    assert run.cache.seq_len.cpu().tolist() == [[14 + 20, 16 + 20, 31 + 20]]


def test_device_errors_are_reported():
    import block_sparse_kv_summary_gb300 as P
    wl = _ragged(SHAPES[0], lengths=(30, 32), budget=64, steps=1)
    run = Run(wl)
    # capacities are 32 and 48 tokens: fill sequence 0 to capacity, then overflow it
    k_new, v_new = run.new_tokens(0, 0)
    run.cache.append(0, k_new, v_new)
    run.cache.append(0, k_new, v_new)
    assert run.cache.device_status() == 0
    run.cache.append(0, k_new, v_new)                # sequence 0 is full: left unchanged
    assert run.cache.device_status() == 3            # COMPKV_ERR_CAPACITY
    assert run.cache.device_status() == 0            # the read cleared it
    assert run.cache.seq_len.cpu().tolist() == [[32, 35]]
    # a selection that is not ascending
    q = torch.zeros((wl.batch, wl.num_kv_heads * wl.group_size, wl.head_dim), device="cuda")
    sel = torch.full((wl.batch, wl.num_kv_heads, wl.K_blocks), -1, dtype=torch.int32, device="cuda")
    sel[0, 0, 0] = 1
    sel[0, 0, 1] = 0
    run.cache.attend(0, q, sel)
    assert run.cache.device_status() == 6            # COMPKV_ERR_BAD_SELECTION
    # host-side validation: nothing is enqueued
    with pytest.raises(P.CompKVError):
        run.cache.attend(5, q, sel)
    with pytest.raises(ValueError):
        run.cache.attend(0, q[:, :1], sel)


def test_bounded_wait_timeout_is_reported():
    """A device wait that nothing completes gives up after its poll cap: the
    context's status word reads COMPKV_ERR_TIMEOUT (5), the read clears it, and
    the context keeps working."""
    import time
    wl = _ragged(SHAPES[0], lengths=(30, 40), budget=64, steps=1)
    run = Run(wl)
    t0 = time.perf_counter()
    run.cache.selftest_wait_timeout()
    assert run.cache.device_status() == 5
    waited = time.perf_counter() - t0
    assert run.cache.device_status() == 0
    q, sel, out, res = run.decode_step(0)
    check_step(run, 0, sel, out, res)
    assert run.cache.device_status() == 0
    print(f"bounded wait gave up after {waited:.3f} s")


@pytest.mark.parametrize("pattern", ["all_equal", "two_kinds"])
def test_selection_ties_go_to_the_lower_index(pattern):
    """Blocks with identical tokens have identical summaries and scores (on both
    sides: the same operations on the same bytes), so the Top-K boundary falls
    inside a run of exactly tied keys and only the lower-index rule decides.
    all_equal: every block the same (4000 blocks: more tied candidates than the
    fast path lists, so the general radix path runs); two_kinds: block b holds
    pattern A when b % 5 == 0, else pattern B, every 64-block chunk holding both."""
    from block_sparse_kv_summary_gb300.cache import CompKVCache
    Hkv, G, d, r, budget = 2, 4, 128, 4, 1024
    lens = [16 * 4000, 16 * 200, 16 * 641]
    cache = CompKVCache(num_layers=1, batch=len(lens), num_kv_heads=Hkv, group_size=G, head_dim=d, r=r,
                        budget_tokens=budget, capacity_tokens=[L + 16 for L in lens])
    gen = torch.Generator().manual_seed(11)
    states = {}
    for s, L in enumerate(lens):
        for h in range(Hkv):
            A = (torch.randn(1, d, generator=gen) + 0.7 * torch.randn(16, d, generator=gen)).to(torch.bfloat16)
            B = (torch.randn(1, d, generator=gen) + 0.3 * torch.randn(16, d, generator=gen)).to(torch.bfloat16)
            nb = L // 16
            blocks = [A if (pattern == "all_equal" or b % 5 == 0) else B for b in range(nb)]
            K = torch.cat(blocks)
            V = torch.randn(L, d, generator=gen).to(torch.bfloat16)
            kv, vv = cache.token_view(0, s, h)
            kv[:L] = K.cuda()
            vv[:L] = V.cuda()
            states[(s, h)] = O.HeadState(K=f64(K), V=f64(V), L=L, r=r).summarise()
    cache.prefill(0, lens)
    q = torch.randn(len(lens), Hkv * G, d, generator=gen)
    sel = cache.score_select(0, q.cuda()).cpu().numpy()
    Kb = budget // 16
    q64 = q.numpy().astype(np.float64)
    for (s, h), st in states.items():
        S = O.block_scores(q64[s, h * G:(h + 1) * G], st.n, st.kbar, st.Dbar).S
        N = len(S)
        # a library matrix product may round identical columns differently in its
        # edge tiles: give every block its pattern's score so the ties are exact
        kind = np.array([0 if (pattern == "all_equal" or b % 5 == 0) else 1 for b in range(N)])
        first = [int(np.nonzero(kind == k)[0][0]) for k in (0, 1) if (kind == k).any()]
        assert all(np.abs(S[kind == kind[f]] - S[f]).max() <= 1e-12 * S[f] for f in first)
        S = np.array([S[first[k]] for k in kind])
        ref = O.select_blocks(S, Kb)
        if pattern == "all_equal":
            assert ref.tolist() == list(range(Kb - 2)) + [N - 2, N - 1]
        exp = np.full(Kb, -1)
        exp[:len(ref)] = ref
        assert np.array_equal(sel[s, h], exp), f"unit {(s, h)}:\n gpu {sel[s, h]}\n ref {exp}"
    assert cache.device_status() == 0


@pytest.mark.parametrize("pinned", [True, False], ids=["page-locked", "pageable"])
def test_decode_host_buffers(pinned):
    # compkv_decode_host: host inputs to host outputs (page-locked buffers are read and written
    # by the kernels directly, pageable ones are copied); the oracle decides, and the outputs equal
    # those of compkv_decode on device buffers of the same cache
    wl = _ragged(SHAPES[1], lengths=(5, 600, 1800), budget=256, steps=3)
    dev, host = Run(wl), Run(wl)
    for step in range(wl.steps):
        qd, seld, outd, resd = dev.decode_step(0)
        k_new, v_new = host.new_tokens(0, step)
        host.oracle_append(0, k_new, v_new)
        q, res = host.choose_queries(0, step)
        mk = (lambda t: t.cpu().pin_memory()) if pinned else (lambda t: t.cpu().clone())
        hq, hk, hv = mk(q), mk(k_new), mk(v_new)
        hout = mk(torch.zeros_like(outd))
        hsel = mk(torch.zeros_like(seld))
        host.cache.decode_host(0, hq, hk, hv, hout, sel=hsel)
        host.step_no[0] += 1
        check_step(host, 0, hsel, hout, res)
        assert torch.equal(hsel, seld.cpu())
        assert (hout - outd.cpu()).abs().max().item() <= 1e-6
    assert host.cache.device_status() == 0
