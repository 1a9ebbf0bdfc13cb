"""GPU parity of the ablation variants and of a compensation-dominated cache.

The ablations of section "전제와 한계" of the CompKV page (first-order mass,
no external variance factor, no Mean compensation) are compile-free switches
of compkv_config.variant; each is checked against the oracle's own switches
under the same rules as the method itself: selections identical, outputs
within 2e-3.  With G = 1, no compensation and no variance factor the selection
is Top-K by the estimated mass (the appendix case of "어떻게 동작하나").

The compensation-dominated case follows the kernels' design: the stream adds
the Mean-compensation term of every block and the attention removes the
selected blocks' own terms.  When the selected blocks carry nearly all of
that mass, the difference is small next to the terms removed; the output must
still match the oracle far inside the 2e-3 tolerance.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from harness import (VARIANT_FIRST_ORDER_MASS, VARIANT_NO_COMPENSATION, VARIANT_NO_VARIANCE_FACTOR, Run,
                     check_step, check_summaries, f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import block_sparse_kv_summary_gb300 as P
    P.build()
    P.lib()


VARIANTS = [VARIANT_FIRST_ORDER_MASS, VARIANT_NO_VARIANCE_FACTOR, VARIANT_NO_COMPENSATION,
            VARIANT_FIRST_ORDER_MASS | VARIANT_NO_VARIANCE_FACTOR,
            VARIANT_FIRST_ORDER_MASS | VARIANT_NO_VARIANCE_FACTOR | VARIANT_NO_COMPENSATION]
SHAPES = [dict(head_dim=128, group_size=4, r=4, num_kv_heads=2),
          dict(head_dim=64, group_size=8, r=64, num_kv_heads=1)]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SHAPES, ids=["d128g4r4", "d64g8r64"])
def test_variant_matches_oracle(variant, shape):
    wl = synth.Workload("variant", 1, 2, shape["num_kv_heads"], shape["group_size"], shape["head_dim"],
                        shape["r"], 0, 256, 3, lengths=(2049, 700))
    run = Run(wl, variant=variant)
    for _ in range(wl.steps):
        q, sel, out, res = run.decode_step(0)
        check_step(run, 0, sel, out, res)
    for (l, s, h) in run.heads:
        check_summaries(run, l, s, h)
    assert run.cache.device_status() == 0


def test_no_compensation_g1_selects_top_k_by_estimated_mass():
    wl = synth.Workload("mass", 1, 1, 2, 1, 128, 4, 0, 160, 2, lengths=(3000,))
    run = Run(wl, variant=VARIANT_NO_COMPENSATION | VARIANT_NO_VARIANCE_FACTOR)
    for _ in range(wl.steps):
        q, sel, out, res = run.decode_step(0)
        check_step(run, 0, sel, out, res)
        for (s, h), r in res.items():
            # the selection is the forced set plus the largest estimated masses phat
            phat = r.scores.phat[0]
            N = len(phat)
            F = O.forced_blocks(N)
            rest = sorted((b for b in range(N) if b not in F), key=lambda b: (-phat[b], b))
            want = sorted(F + rest[:wl.K_blocks - len(F)])
            assert list(r.sel) == want
            # and the output is softmax attention over the selected tokens alone
            st = run.states[(0, s, h)]
            tok = np.concatenate([np.arange(16 * b, min(16 * b + 16, st.L)) for b in r.sel])
            qh = f64(q)[s, h:h + 1]
            np.testing.assert_allclose(r.out, O.dense_attention(qh, st.K[tok], st.V[tok]), rtol=1e-12, atol=1e-13)
    assert run.cache.device_status() == 0


def _dominated_cache(rng, N, d, G, needles, zero_selected_values):
    """Keys N(0, 0.3^2) except whole needle blocks aimed at the mean query with
    logits near +20 (and within-block spread); values N(0, 1)."""
    q = rng.standard_normal((G, d)).astype(np.float32)
    u = q.astype(np.float64).mean(axis=0)
    u /= np.linalg.norm(u)
    qn = float(np.linalg.norm(q.astype(np.float64).mean(axis=0)))
    L = 16 * N
    K = 0.3 * rng.standard_normal((L, d))
    for b in needles:
        K[16 * b:16 * b + 16] = (20.0 * math.sqrt(d) / qn) * u + rng.standard_normal((16, d))
    V = rng.standard_normal((L, d))
    if zero_selected_values:
        for b in needles:
            V[16 * b:16 * b + 16] = 0.0
    Kb = torch.from_numpy(K.astype(np.float32)).to(torch.bfloat16)
    Vb = torch.from_numpy(V.astype(np.float32)).to(torch.bfloat16)
    return q, Kb, Vb


@pytest.mark.parametrize("zero_selected_values", [False, True])
def test_compensation_dominated_by_selected_blocks(zero_selected_values):
    from block_sparse_kv_summary_gb300.cache import CompKVCache
    rng = np.random.default_rng(91 + int(zero_selected_values))
    N, d, G, r = 600, 128, 4, 4
    needles = [37, 211, 400, 512]
    q, Kb, Vb = _dominated_cache(rng, N, d, G, needles, zero_selected_values)
    cache = CompKVCache(num_layers=1, batch=1, num_kv_heads=1, group_size=G, head_dim=d, r=r,
                        budget_tokens=16 * 16, capacity_tokens=16 * N, device="cuda")
    kv, vv = cache.token_view(0, 0, 0)
    kv[:] = Kb.cuda()
    vv[:] = Vb.cuda()
    cache.prefill(0, [16 * N])
    sel_blocks = sorted(set([0, N - 2, N - 1] + needles))
    sel = torch.full((1, 1, cache.K), -1, dtype=torch.int32, device="cuda")
    sel[0, 0, :len(sel_blocks)] = torch.tensor(sel_blocks, dtype=torch.int32)
    qt = torch.from_numpy(q).reshape(1, G, d).cuda()
    out = f64(cache.attend(0, qt, sel))[0]
    assert cache.device_status() == 0
    K64, V64 = f64(Kb), f64(Vb)
    n, kbar, Dbar, vbar = O.block_summaries(K64, V64, r)
    ref = O.compkv_attend(q.astype(np.float64), K64, V64, sel_blocks, n, kbar, vbar)
    # the selected blocks' mean terms dwarf the compensation of all the others
    zb = (kbar @ q.astype(np.float64).T).T / math.sqrt(d)
    w = n[None, :] * np.exp(zb - zb.max())
    unsel = [b for b in range(N) if b not in sel_blocks]
    assert (w[:, needles].sum(axis=1) / w[:, unsel].sum(axis=1)).min() > 1e4
    err = np.abs(out - ref).max()
    if zero_selected_values:
        # the output is the compensation part alone over the joint denominator
        assert np.abs(ref).max() > 0
        assert err <= 1e-6 + 1e-3 * np.abs(ref).max(), err
    else:
        assert err <= 5e-5, err
