"""Pins of the fp64 oracle to facts the CompKV page and mathematics fix.

Each test checks the oracle against something other than itself: a library
routine (numpy mean/var, scipy softmax/logsumexp), a closed form, a special
case that reduces to dense attention, brute force over all admissible sets,
or the asymptotics of the page's second-order Taylor argument.  Sections
cited are those of the CompKV page (onedev.kr/papers/157).
"""
import itertools
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp as sp_logsumexp
from scipy.special import softmax as sp_softmax

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_exact(x):
    """Round float64 values to the nearest bf16 (ties to even) and return float64."""
    a = np.asarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def rand_cache(rng, L, d, scale=0.5):
    N = O.num_blocks(L)
    centre = rng.standard_normal((N, d))
    K = np.repeat(centre, 16, axis=0)[:L] + scale * rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    return bf16_exact(K), bf16_exact(V)


# ---------------------------------------------------------------------------
# Golden: hand-worked closed forms ("무엇과 다른가", "어떻게 동작하나")
# ---------------------------------------------------------------------------
def _load_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = line.split(":", 1)
            vals.setdefault(k.strip(), []).append(v.split())
    return vals


def _ev(tokens):
    ns = {"exp": math.exp, "log": math.log, "e": math.e}
    return np.array([float(eval(t, {"__builtins__": {}}, ns)) for t in tokens])


def test_golden_hand_two_blocks():
    g = _load_golden("hand_two_blocks.txt")
    d, r = int(g["d"][0][0]), int(g["r"][0][0])
    q = _ev(g["q"][0])[None, :]
    keys = [_ev(k) for k in g["key"]]
    vals = [_ev(v) for v in g["value"]]
    K = np.array([keys[j % 4] for j in range(16)] + [_ev(k) for k in g["tail_key"]])
    V = np.array([vals[j % 4] for j in range(16)] + [_ev(v) for v in g["tail_value"]])
    n, kbar, Dbar, vbar = O.block_summaries(K, V, r)
    assert list(n) == [int(x) for x in g["expect_n"][0]]
    for b in range(2):
        np.testing.assert_allclose(kbar[b], _ev(g[f"expect_kbar{b}"][0]), atol=1e-15)
        np.testing.assert_allclose(Dbar[b], _ev(g[f"expect_Dbar{b}"][0]), atol=1e-15)
        np.testing.assert_allclose(vbar[b], _ev(g[f"expect_vbar{b}"][0]), atol=1e-15)
    sc = O.block_scores(q, n, kbar, Dbar)
    np.testing.assert_allclose(sc.zbar[0], _ev(g["expect_zbar"][0]), atol=1e-15)
    np.testing.assert_allclose(sc.sigma2[0], _ev(g["expect_sigma2"][0]), atol=1e-15)
    np.testing.assert_allclose(sc.phat[0], _ev(g["expect_phat"][0]), rtol=1e-14)
    np.testing.assert_allclose(sc.S, _ev(g["expect_S"][0]), rtol=1e-14, atol=1e-300)
    dense = O.compkv_attend(q, K, V, [0, 1], n, kbar, vbar)
    np.testing.assert_allclose(dense[0], _ev(g["expect_dense_out"][0]), rtol=1e-14)
    out1 = O.compkv_attend(q, K, V, [1], n, kbar, vbar)
    np.testing.assert_allclose(out1[0], _ev(g["expect_sel1_out"][0]), rtol=1e-14)
    kl = O.selection_loss_closed_form(q[0], K, len(K), [1])
    np.testing.assert_allclose(kl, _ev(g["expect_sel1_kl"][0])[0], rtol=1e-13)


# ---------------------------------------------------------------------------
# P1 summaries == numpy mean / population var, grouped ("무엇과 다른가")
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L,d,r", [(37, 8, 2), (16, 8, 8), (50, 16, 4), (1, 4, 1), (33, 64, 4)])
def test_summaries_match_numpy(L, d, r):
    rng = np.random.default_rng(L * 100 + d + r)
    K, V = rand_cache(rng, L, d)
    n, kbar, Dbar, vbar = O.block_summaries(K, V, r)
    N = (L + 15) // 16
    assert len(n) == N and n.sum() == L
    gs = d // r
    for b in range(N):
        blk = slice(16 * b, min(16 * b + 16, L))
        assert n[b] == len(range(L)[blk])
        np.testing.assert_allclose(kbar[b], np.mean(K[blk], axis=0), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(vbar[b], np.mean(V[blk], axis=0), rtol=1e-13, atol=1e-14)
        var = np.var(K[blk], axis=0, ddof=0)
        for t in range(r):
            np.testing.assert_allclose(Dbar[b, t], np.mean(var[t * gs:(t + 1) * gs]),
                                       rtol=1e-12, atol=1e-14)


def test_summary_hand_alternating():
    # keys alternating 0 / 2 in one coordinate: mean 1, population variance 1
    K = np.zeros((16, 4))
    K[1::2, 2] = 2.0
    n, kbar, Dbar, vbar = O.block_summaries(K, K, 4)
    assert kbar[0, 2] == 1.0 and Dbar[0, 2] == 1.0 and Dbar[0, [0, 1, 3]].sum() == 0.0


def test_append_matches_full_recompute():
    rng = np.random.default_rng(5)
    L0, d, r, steps = 45, 16, 4, 20
    K, V = rand_cache(rng, L0 + steps, d)
    st = O.HeadState(K=K.copy(), V=V.copy(), L=L0, r=r).summarise()
    st.K[L0:] = np.nan   # the appended tokens must come from the append call
    for i in range(steps):
        st.append(K[L0 + i], V[L0 + i])
        n, kbar, Dbar, vbar = O.block_summaries(K[: L0 + i + 1], V[: L0 + i + 1], r)
        assert np.array_equal(st.n, n)
        np.testing.assert_allclose(st.kbar, kbar, rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(st.Dbar, Dbar, rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(st.vbar, vbar, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------------------
# zbar is the exact block-mean logit (linearity)
# ---------------------------------------------------------------------------
def test_zbar_is_mean_token_logit():
    rng = np.random.default_rng(7)
    L, d, r, G = 70, 32, 4, 3
    K, V = rand_cache(rng, L, d)
    q = rng.standard_normal((G, d))
    n, kbar, Dbar, vbar = O.block_summaries(K, V, r)
    sc = O.block_scores(q, n, kbar, Dbar)
    for g in range(G):
        z = K @ q[g] / math.sqrt(d)
        for b in range(len(n)):
            np.testing.assert_allclose(sc.zbar[g, b], np.mean(z[16 * b:16 * b + n[b]]), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# P2 constant-key block: Dbar = 0, sigma2 = 0, S_b = 0 ("어떻게 동작하나")
# ---------------------------------------------------------------------------
def test_constant_key_block_scores_zero():
    rng = np.random.default_rng(11)
    L, d, r, G = 80, 16, 4, 4
    K, V = rand_cache(rng, L, d)
    K[16:32] = K[16]            # block 1 constant
    K[64:80] = K[70]            # block 4 constant
    q = rng.standard_normal((G, d))
    n, kbar, Dbar, vbar = O.block_summaries(K, V, r)
    sc = O.block_scores(q, n, kbar, Dbar)
    for b in (1, 4):
        assert np.all(Dbar[b] == 0.0) and np.all(sc.sigma2[:, b] == 0.0) and sc.S[b] == 0.0
        assert sc.phat[:, b].min() > 0.0        # it may still carry mass
    assert np.all(sc.S[[0, 2, 3]] > 0.0)


# ---------------------------------------------------------------------------
# P3 identical keys within every block => compensation exact for any selection
# ---------------------------------------------------------------------------
def test_identical_keys_compensation_exact():
    rng = np.random.default_rng(13)
    L, d, r, G = 90, 16, 4, 4
    N = O.num_blocks(L)
    centre = bf16_exact(rng.standard_normal((N, d)))
    K = np.repeat(centre, 16, axis=0)[:L]
    V = bf16_exact(rng.standard_normal((L, d)))
    q = rng.standard_normal((G, d))
    n, kbar, Dbar, vbar = O.block_summaries(K, V, r)
    dense = sp_softmax(q @ K.T / math.sqrt(d), axis=1) @ V
    for sel in ([0], [2, 5], [0, 1, 2, 3, 4, 5], [], [5], [1, 3]):
        out = O.compkv_attend(q, K, V, sel, n, kbar, vbar) if sel else None
        if sel:
            np.testing.assert_allclose(out, dense, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# P4 r = d: sigma2_hat equals the exact within-block logit variance when the
# block's key covariance is diagonal, or when q has one non-zero coordinate
# ---------------------------------------------------------------------------
def test_r_equals_d_variance_diagonal_covariance():
    rng = np.random.default_rng(17)
    d, G, N = 16, 4, 5
    blocks = []
    for b in range(N):
        c = np.round(rng.standard_normal(d) * 8) / 8
        toks = []
        for p in range(8):                     # 8 antithetic pairs: mean c, diagonal covariance
            i = rng.integers(d)
            a = rng.choice([0.5, 1.0, 1.5, 2.0])
            e = np.zeros(d); e[i] = a
            toks += [c + e, c - e]
        blocks.append(np.array(toks))
    K = np.concatenate(blocks)
    V = bf16_exact(rng.standard_normal(K.shape))
    assert np.array_equal(K, bf16_exact(K))
    q = rng.standard_normal((G, d))
    n, kbar, Dbar, vbar = O.block_summaries(K, V, d)
    sc = O.block_scores(q, n, kbar, Dbar)
    for g in range(G):
        z = K @ q[g] / math.sqrt(d)
        for b in range(N):
            np.testing.assert_allclose(sc.sigma2[g, b], np.var(z[16 * b:16 * b + 16]), rtol=1e-12)


def test_r_equals_d_variance_one_hot_query():
    rng = np.random.default_rng(19)
    L, d = 64, 16
    K, V = rand_cache(rng, L, d, scale=1.0)
    q = np.zeros((d, d))
    q[np.arange(d), np.arange(d)] = rng.uniform(0.5, 3.0, d)     # G = d one-hot queries
    n, kbar, Dbar, vbar = O.block_summaries(K, V, d)
    sc = O.block_scores(q, n, kbar, Dbar)
    for g in range(d):
        z = K @ q[g] / math.sqrt(d)
        for b in range(len(n)):
            np.testing.assert_allclose(sc.sigma2[g, b], np.var(z[16 * b:16 * b + 16]), rtol=1e-12, atol=1e-15)


def test_grouped_variance_is_group_pooled():
    # r < d: sigma2_hat = (1/d) sum_t Qsq_t Dbar_t; with q constant inside each
    # group it equals (1/d) sum_i q_i^2 var_i exactly (pooling loses nothing)
    rng = np.random.default_rng(23)
    L, d, r = 48, 16, 4
    K, V = rand_cache(rng, L, d, scale=1.0)
    qg = np.repeat(rng.standard_normal(r), d // r)[None, :]
    n, kbar, Dbar, vbar = O.block_summaries(K, V, r)
    sc = O.block_scores(qg, n, kbar, Dbar)
    for b in range(len(n)):
        var = np.var(K[16 * b:16 * b + 16], axis=0)
        np.testing.assert_allclose(sc.sigma2[0, b], np.sum(qg[0] ** 2 * var) / d, rtol=1e-12)


# ---------------------------------------------------------------------------
# P5 select-all: output == dense softmax attention
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L", [1, 15, 16, 17, 50, 130])
def test_select_all_is_dense(L):
    rng = np.random.default_rng(L)
    d, r, G = 32, 4, 4
    K, V = rand_cache(rng, L, d)
    q = rng.standard_normal((G, d)) * 2
    st = O.HeadState(K=K, V=V, L=L, r=r).summarise()
    N = O.num_blocks(L)
    res = O.decode_head(st, q, max(N, 3))
    assert list(res.sel) == list(range(N))
    dense = sp_softmax(q @ K.T / math.sqrt(d), axis=1) @ V
    np.testing.assert_allclose(res.out, dense, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# P6 mass estimate: sums to one; exact for constant-key blocks
# ---------------------------------------------------------------------------
def test_phat_normalised_and_exact_for_constant_blocks():
    rng = np.random.default_rng(29)
    L, d, r, G = 100, 16, 4, 4
    N = O.num_blocks(L)
    K = np.repeat(bf16_exact(rng.standard_normal((N, d)) * 2), 16, axis=0)[:L]
    V = bf16_exact(rng.standard_normal((L, d)))
    q = rng.standard_normal((G, d))
    n, kbar, Dbar, vbar = O.block_summaries(K, V, r)
    sc = O.block_scores(q, n, kbar, Dbar)
    np.testing.assert_allclose(sc.phat.sum(axis=1), 1.0, rtol=1e-13)
    for g in range(G):
        z = K @ q[g] / math.sqrt(d)
        logZ = np.array([sp_logsumexp(z[16 * b:16 * b + n[b]]) for b in range(N)])
        np.testing.assert_allclose(sc.phat[g], np.exp(logZ - sp_logsumexp(logZ)), rtol=1e-12)
    # random blocks: still a distribution
    K2, V2 = rand_cache(rng, L, d)
    sc2 = O.block_scores(q, *O.block_summaries(K2, V2, r)[:2], O.block_summaries(K2, V2, r)[2])
    np.testing.assert_allclose(sc2.phat.sum(axis=1), 1.0, rtol=1e-13)


def test_phat_lognormal_exact_for_gaussian_logits():
    # For a block whose logits are (nearly) normally distributed, the log-normal
    # mass |b| e^{zbar + sigma2/2} approaches the block partition function.
    rng = np.random.default_rng(31)
    from scipy.stats import norm
    d, n = 16, 16
    qg = np.zeros(d); qg[0] = math.sqrt(d)               # logit = k_0
    for s in (0.05, 0.2):
        z = norm.ppf((np.arange(n) + 0.5) / n) * s         # quantiles of N(0, s^2)
        z = (z - z.mean())
        K = np.zeros((n, d)); K[:, 0] = z
        nb, kbar, Dbar, vbar = O.block_summaries(K, K, d)
        sc = O.block_scores(qg[None], nb, kbar, Dbar)
        logZ = sp_logsumexp(z)
        assert abs(sc.a[0, 0] - logZ) < s ** 4         # error of the second-order log-partition


# ---------------------------------------------------------------------------
# P7 Taylor ("어떻게 동작하나"): per-block loss term / (p sigma^2 / 2) -> 1
# ---------------------------------------------------------------------------
def test_taylor_second_order():
    rng = np.random.default_rng(37)
    d, L = 8, 64
    N = O.num_blocks(L)
    base_c = rng.standard_normal((N, d))
    base_e = rng.standard_normal((L, d))
    qg = rng.standard_normal(d)
    errs = []
    for s in (1e-1, 1e-2, 1e-3):
        K = np.repeat(base_c, 16, axis=0) + s * base_e
        logZ, zmean, zvar, p = O.exact_block_stats(qg, K, L)
        n = O.block_counts(L)
        ratios = [O.block_loss_term(p[b], n[b], zmean[b], logZ[b]) / (0.5 * p[b] * zvar[b]) for b in range(N)]
        errs.append(max(abs(x - 1) for x in ratios))
    assert errs[0] < 0.2
    assert errs[1] < errs[0] / 5 and errs[2] < errs[1] / 5       # O(sigma) error shrinks ~linearly in s
    assert errs[2] < 1e-2


# ---------------------------------------------------------------------------
# KL closed form == KL of the token-level distributions, built independently
# ---------------------------------------------------------------------------
def _token_level_compensated(qg, K, L, sel, compensate=True):
    z = K[:L] @ qg / math.sqrt(len(qg))
    zz = z.copy()
    keep = np.ones(L, dtype=bool)
    for b in range(O.num_blocks(L)):
        if b in set(sel):
            continue
        blk = slice(16 * b, min(16 * b + 16, L))
        if compensate:
            zz[blk] = np.mean(z[blk])
        else:
            keep[blk] = False
    p = np.zeros(L)
    p[keep] = sp_softmax(zz[keep])
    return p, sp_softmax(z)


@pytest.mark.parametrize("sel", [[0, 3], [1], [0, 2, 4], [4]])
def test_kl_closed_form_matches_token_level(sel):
    rng = np.random.default_rng(41)
    L, d = 75, 8
    K, V = rand_cache(rng, L, d, scale=0.7)
    qg = rng.standard_normal(d) * 1.5
    p_tilde, p = _token_level_compensated(qg, K, L, sel)
    kl_tok = float(np.sum(p_tilde * np.log(p_tilde / p)))
    np.testing.assert_allclose(O.selection_loss_closed_form(qg, K, L, sel), kl_tok, rtol=1e-10)
    np.testing.assert_allclose(O.kl_divergence(p_tilde, p), kl_tok, rtol=1e-12)


@pytest.mark.parametrize("sel", [[0, 3], [1], [0, 2, 4], [4], [0, 1, 2, 3, 4]])
def test_attend_matches_token_level_mean_replacement(sel):
    # Mean compensation = every logit of an unselected block replaced by the
    # block mean, then ordinary softmax attention over the original values.
    rng = np.random.default_rng(43)
    L, d, r, G = 75, 16, 4, 3
    K, V = rand_cache(rng, L, d, scale=0.7)
    q = rng.standard_normal((G, d)) * 1.5
    n, kbar, Dbar, vbar = O.block_summaries(K, V, r)
    out = O.compkv_attend(q, K, V, sel, n, kbar, vbar)
    for g in range(G):
        p_tilde, _ = _token_level_compensated(q[g], K, L, sel)
        np.testing.assert_allclose(out[g], p_tilde @ V, rtol=1e-12, atol=1e-13)
    out_nc = O.compkv_attend(q, K, V, sel, n, kbar, vbar, compensate=False)
    for g in range(G):
        p_nc, _ = _token_level_compensated(q[g], K, L, sel, compensate=False)
        np.testing.assert_allclose(out_nc[g], p_nc @ V, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# P8 appendix ("어떻게 동작하나"): without compensation and G = 1, the loss is
# -ln sum_{b in S} p_b, minimised by Top-K on the exact mass.  Brute force.
# ---------------------------------------------------------------------------
def test_no_compensation_g1_is_topk_by_mass():
    rng = np.random.default_rng(47)
    d, r = 8, 2
    for trial in range(6):
        N = int(rng.integers(8, 12))
        L = 16 * (N - 1) + int(rng.integers(1, 17))
        Kblk = 3
        N = O.num_blocks(L)
        centre = bf16_exact(rng.standard_normal((N, d)) * 0.5)
        K = np.repeat(centre, 16, axis=0)[:L]         # constant-key blocks: mass estimate exact
        V = bf16_exact(rng.standard_normal((L, d)))
        qg = rng.standard_normal(d)
        F = O.forced_blocks(N)
        Kb = len(F) + Kblk
        best, best_set = None, None
        for extra in itertools.combinations([b for b in range(N) if b not in F], Kblk):
            sel = sorted(F + list(extra))
            p_nc, p = _token_level_compensated(qg, K, L, sel, compensate=False)
            kl = float(np.sum(p_nc[p_nc > 0] * np.log(p_nc[p_nc > 0] / p[p_nc > 0])))
            if best is None or kl < best - 1e-12:
                best, best_set = kl, sel
        n, kbar, Dbar, vbar = O.block_summaries(K, V, r)
        sc = O.block_scores(qg[None], n, kbar, Dbar, second_order_mass=False, variance_factor=False)
        assert list(O.select_blocks(sc.S, Kb)) == best_set
        # and the loss itself is -ln(selected exact mass)
        logZ, _, _, pm = O.exact_block_stats(qg, K, L)
        np.testing.assert_allclose(best, -math.log(pm[best_set].sum()), rtol=1e-10, atol=1e-13)
        assert best > 1e-3          # a non-trivial instance


# ---------------------------------------------------------------------------
# P9 selection: brute force over admissible sets; lower index wins ties
# ---------------------------------------------------------------------------
def test_selection_brute_force_and_tie_break():
    rng = np.random.default_rng(53)
    for trial in range(60):
        N = int(rng.integers(1, 11))
        K = int(rng.integers(3, 8))
        S = rng.choice([0.0, 0.25, 0.5, 1.0, 2.0, 3.0], size=N)      # many ties
        sel = list(O.select_blocks(S, K))
        if N <= K:
            assert sel == list(range(N))
            continue
        F = O.forced_blocks(N)
        assert set(F) <= set(sel) and len(sel) == K and sel == sorted(sel)
        best = max(sum(S[list(F) + list(c)]) for c in
                   itertools.combinations([b for b in range(N) if b not in F], K - len(F)))
        assert abs(sum(S[sel]) - best) < 1e-12
        chosen = [b for b in sel if b not in F]
        for b in range(N):
            if b in sel or b in F:
                continue
            for c in chosen:     # no rejected block precedes a chosen one in (S desc, index asc)
                assert S[b] < S[c] or (S[b] == S[c] and b > c)


def test_selection_small_N_edge_cases():
    assert list(O.select_blocks(np.array([5.0]), 8)) == [0]
    assert list(O.select_blocks(np.array([1.0, 2.0]), 8)) == [0, 1]
    assert list(O.select_blocks(np.arange(4.0), 3)) == [0, 2, 3]          # forced fill the budget
    assert list(O.select_blocks(np.array([0, 9, 9, 9, 0, 0.0]), 4)) == [0, 1, 4, 5]
    assert O.forced_blocks(1) == [0] and O.forced_blocks(2) == [0, 1] and O.forced_blocks(3) == [0, 1, 2]


def test_boundary_gap():
    S = np.array([0.0, 4.0, 3.0, 2.0, 1.0, 0.0, 0.0])     # forced {0, 5, 6}
    assert O.boundary_gap(S, 4) == pytest.approx(0.25)      # 4 selected, 3 first rejected
    assert O.boundary_gap(S, 5) == pytest.approx(1 / 3)
    assert O.boundary_gap(S, 7) == math.inf


# ---------------------------------------------------------------------------
# The two reference helpers of "어떻게 동작하나": dense softmax attention and
# the token-level distribution of Mean compensation.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L", [1, 16, 40, 130])
def test_dense_attention_pins(L):
    rng = np.random.default_rng(100 + L)
    d, G = 16, 3
    K, V = rand_cache(rng, L, d)
    q = rng.standard_normal((G, d)) * 2
    # a library routine: scipy's softmax over the scaled logits
    ref = sp_softmax(q @ K.T / math.sqrt(d), axis=1) @ V
    np.testing.assert_allclose(O.dense_attention(q, K, V), ref, rtol=1e-12, atol=1e-13)
    # identical keys: every weight is 1/L, the output is the mean value
    Kc = np.repeat(K[:1], L, axis=0)
    np.testing.assert_allclose(O.dense_attention(q, Kc, V), np.repeat(V.mean(axis=0)[None], G, axis=0),
                               rtol=1e-12, atol=1e-13)
    # one key far ahead of the others: the output is that key's value
    if L > 1:
        j = L // 2
        Kp = K.copy()
        Kp[j] = q[0] / np.linalg.norm(q[0]) * 200 * math.sqrt(d)
        np.testing.assert_allclose(O.dense_attention(q[:1], Kp, V)[0], V[j], rtol=0, atol=1e-12)


@pytest.mark.parametrize("sel", [[0, 3], [1], [0, 2, 4], [4], [0, 1, 2, 3, 4]])
def test_compensated_token_distribution_pins(sel):
    rng = np.random.default_rng(47)
    L, d, r = 75, 8, 2
    K, V = rand_cache(rng, L, d, scale=0.7)
    qg = rng.standard_normal(d) * 1.5
    p_ref, p = _token_level_compensated(qg, K, L, sel)
    pc = O.compensated_token_distribution(qg, K, L, sel)
    # an independent construction through scipy's softmax
    np.testing.assert_allclose(pc, p_ref, rtol=1e-12, atol=1e-15)
    assert abs(pc.sum() - 1.0) < 1e-12
    # its KL divergence from the token softmax is the closed-form selection loss
    np.testing.assert_allclose(O.kl_divergence(pc, p), O.selection_loss_closed_form(qg, K, L, sel), rtol=1e-10)
    # its expectation of the values is the compensated attention output
    n, kbar, Dbar, vbar = O.block_summaries(K, V, r)
    out = O.compkv_attend(qg[None], K, V, sel, n, kbar, vbar)[0]
    np.testing.assert_allclose(pc @ V, out, rtol=1e-12, atol=1e-13)
    # without compensation: the softmax restricted to the selected blocks, and
    # KL = -ln (exact mass of the selected blocks)
    pn = O.compensated_token_distribution(qg, K, L, sel, compensate=False)
    logZ, _, _, pm = O.exact_block_stats(qg, K, L)
    np.testing.assert_allclose(O.kl_divergence(pn, p), -math.log(sum(pm[b] for b in sel)), rtol=1e-10, atol=1e-14)
    nb = O.block_counts(L)
    outside = np.ones(L, dtype=bool)
    for b in sel:
        outside[16 * b:16 * b + nb[b]] = False
    assert np.all(pn[outside] == 0.0)
