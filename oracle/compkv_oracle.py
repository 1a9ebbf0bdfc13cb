"""fp64 CPU oracle for the CompKV decode step.

TEST INFRASTRUCTURE ONLY.  This module is the checker for the CUDA path: only
the test-suite, the package smoke check and the benchmark's CPU-baseline leg
may import it.  The product path (the C-ABI library and its Python binding)
never imports, links or calls anything here, and this module imports nothing
from the product path.  It shares no code, tables or helpers with the CUDA
kernels.

Source of every definition: the CompKV page (onedev.kr/papers/157).  Its
sections are cited by their headings:
  * "무엇과 다른가" (how it differs)  -- block summaries, estimators, score,
    forced set, Top-K, joint normalisation;
  * "어떻게 동작하나" (how it works) -- Mean compensation, the KL selection
    loss, its second-order Taylor form, the no-compensation special case;
  * "전제와 한계" (assumptions and limits) -- block size 16, r = 4, and the
    ablation switches (first-order mass, external variance factor, Mean
    compensation).

Everything is computed in float64 from the exact values the GPU holds (bf16
keys/values and fp32 queries upcast without rounding).  The code follows the
definitions term by term, with numpy primitives (mean, matmul, exp, log, sort)
as its only building blocks.

Readings taken where the page is silent (each is pinned by a test):
  * within-block variance is the population variance (1/|b|);
  * the r coordinate groups are contiguous runs of d/r coordinates;
  * the normaliser of the mass estimate runs over all blocks, forced ones and
    the partial last block included;
  * the last block may be partial; it counts |b| = its token count, is one of
    the two most recent (forced) blocks and costs one block of budget;
  * ties in the Top-K are broken towards the lower block index;
  * if the cache holds no more blocks than the budget, every block is
    selected (the step is then dense attention);
  * the garbled per-block loss term in "how it works" is read with Z the
    block's own partition function, Z_b = sum_{j in b} exp(z_j).

Parity pins: every public function below is pinned by tests in
tests/test_oracle_pins.py against library routines, closed forms, special
cases or brute force.  The quality of the synthetic needle construction is
the one item left "parity unpinned" (it is input generation, not method).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK = 16  # tokens per KV block ("전제와 한계": block size 16)


# --------------------------------------------------------------------------
# 1. Block summaries {|b|, kbar_b, Dbar_b, vbar_b}   ("무엇과 다른가")
# --------------------------------------------------------------------------
def num_blocks(L: int, block: int = BLOCK) -> int:
    """Number of blocks covering L tokens; the last one may be partial."""
    return (L + block - 1) // block


def block_counts(L: int, block: int = BLOCK) -> np.ndarray:
    """|b| for every block of a length-L sequence."""
    N = num_blocks(L, block)
    n = np.full(N, block, dtype=np.int64)
    if N:
        n[-1] = L - block * (N - 1)
    return n


def block_summaries(K: np.ndarray, V: np.ndarray, r: int, block: int = BLOCK):
    """Per-block summaries of one (sequence, KV head).

    K, V: [L, d] float64 (the stored bf16 values, upcast exactly).
    Returns n [N] (int), kbar [N, d], Dbar [N, r], vbar [N, d] (float64).

    kbar_b = mean of the block's keys; vbar_b = mean of its values;
    (Dbar_b)_t = mean over the coordinates i of group t of the within-block
    population variance of coordinate i.  Groups are contiguous: group t holds
    coordinates [t*d/r, (t+1)*d/r).
    """
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    L, d = K.shape
    if d % r:
        raise ValueError("r must divide d")
    n = block_counts(L, block)
    N = len(n)
    kbar = np.zeros((N, d))
    vbar = np.zeros((N, d))
    Dbar = np.zeros((N, r))
    for b in range(N):
        kb = K[block * b: block * b + n[b]]
        vb = V[block * b: block * b + n[b]]
        kbar[b] = kb.mean(axis=0)
        vbar[b] = vb.mean(axis=0)
        var = ((kb - kbar[b]) ** 2).mean(axis=0)          # population variance
        Dbar[b] = var.reshape(r, d // r).mean(axis=1)     # grouped mean
    return n, kbar, Dbar, vbar


# --------------------------------------------------------------------------
# 2. Scoring estimators   ("무엇과 다른가")
# --------------------------------------------------------------------------
def _logsumexp(a: np.ndarray, axis: int = -1) -> np.ndarray:
    m = np.max(a, axis=axis, keepdims=True)
    return (m + np.log(np.sum(np.exp(a - m), axis=axis, keepdims=True))).squeeze(axis)


@dataclass
class Scores:
    zbar: np.ndarray      # [G, N]  q_g . kbar_b / sqrt(d)
    sigma2: np.ndarray    # [G, N]  (1/d) sum_t (sum_{i in G_t} q_{g,i}^2) (Dbar_b)_t
    a: np.ndarray         # [G, N]  ln|b| + zbar + 1/2 sigma2   (log of the unnormalised mass)
    lse: np.ndarray       # [G]     logsumexp_b a_{g,b}
    phat: np.ndarray      # [G, N]  exp(a - lse)
    S: np.ndarray         # [N]     sum_g phat * sigma2


def block_scores(q: np.ndarray, n: np.ndarray, kbar: np.ndarray, Dbar: np.ndarray,
                 second_order_mass: bool = True, variance_factor: bool = True) -> Scores:
    """Estimated logit variance, estimated block mass and the block score.

    q: [G, d] float64, the G query heads that share this KV head.

    sigma2_{g,b} = (1/d) sum_t (sum_{i in G_t} q_{g,i}^2) (Dbar_b)_t
    phat_{g,b}   = |b| exp(zbar + sigma2/2) / sum_c |c| exp(zbar_c + sigma2_c/2)
    S_b          = sum_g phat_{g,b} sigma2_{g,b}

    The two switches restate the ablations of "전제와 한계": with
    second_order_mass=False the 1/2 sigma2 term is dropped from the mass
    (first-order mass); with variance_factor=False the score is the summed
    mass alone, S_b = sum_g phat_{g,b} (no external variance factor).
    """
    q = np.asarray(q, dtype=np.float64)
    G, d = q.shape
    r = Dbar.shape[1]
    zbar = (q @ kbar.T) / math.sqrt(d)
    Qsq = (q ** 2).reshape(G, r, d // r).sum(axis=2)      # [G, r]
    sigma2 = (Qsq @ Dbar.T) / d
    a = np.log(n.astype(np.float64))[None, :] + zbar
    if second_order_mass:
        a = a + 0.5 * sigma2
    lse = _logsumexp(a, axis=1)
    phat = np.exp(a - lse[:, None])
    S = (phat * sigma2).sum(axis=0) if variance_factor else phat.sum(axis=0)
    return Scores(zbar=zbar, sigma2=sigma2, a=a, lse=lse, phat=phat, S=S)


# --------------------------------------------------------------------------
# 3. Forced set + Top-K   ("무엇과 다른가")
# --------------------------------------------------------------------------
def forced_blocks(N: int) -> list[int]:
    """F = {sink block 0, the two most recent blocks N-2, N-1}, clipped to [0, N)."""
    return sorted({b for b in (0, N - 2, N - 1) if 0 <= b < N})


def select_blocks(S: np.ndarray, K: int) -> np.ndarray:
    """Selected block indices, ascending.

    F is always selected and counts against the K-block budget; the remaining
    K - |F| slots go to the other blocks with the largest S_b, ties to the
    lower index.  With N <= K every block is selected.
    """
    N = len(S)
    if N <= K:
        return np.arange(N, dtype=np.int64)
    F = forced_blocks(N)
    if K < len(F):
        raise ValueError("budget smaller than the forced set")
    rest = [b for b in range(N) if b not in F]
    rest.sort(key=lambda b: (-S[b], b))
    return np.array(sorted(F + rest[: K - len(F)]), dtype=np.int64)


def boundary_gap(S: np.ndarray, K: int) -> float:
    """Relative gap (S_(K') - S_(K'+1)) / S_(K') between the last selected and
    the first rejected non-forced score; +inf when no block is rejected."""
    N = len(S)
    if N <= K:
        return math.inf
    F = forced_blocks(N)
    rest = np.sort(np.array([S[b] for b in range(N) if b not in F]))[::-1]
    kp = K - len(F)
    if kp <= 0 or kp >= len(rest):
        return math.inf
    top, nxt = rest[kp - 1], rest[kp]
    if top <= 0.0:
        return 0.0
    return float((top - nxt) / top)


# --------------------------------------------------------------------------
# 4+5. Exact attention on the selected blocks + Mean compensation,
#      normalised jointly   ("무엇과 다른가", "어떻게 동작하나")
# --------------------------------------------------------------------------
def compkv_attend(q: np.ndarray, Ktok: np.ndarray, Vtok: np.ndarray, sel,
                  n: np.ndarray, kbar: np.ndarray, vbar: np.ndarray,
                  compensate: bool = True) -> np.ndarray:
    """Output [G, d] of one (sequence, KV head).

    Ktok, Vtok: [L, d] float64 tokens.  Selected blocks use their original
    tokens: logit z_j = q . k_j / sqrt(d).  Each unselected block b adds
    |b| exp(zbar_b) vbar_b to the numerator and |b| exp(zbar_b) to the
    denominator.  Both parts share one normaliser.  compensate=False drops
    the unselected blocks altogether (the no-compensation ablation).
    """
    q = np.asarray(q, dtype=np.float64)
    G, d = q.shape
    N = len(n)
    sel = np.asarray(sel, dtype=np.int64)
    selset = set(int(b) for b in sel)
    tok = np.concatenate([np.arange(BLOCK * b, BLOCK * b + n[b]) for b in sel]) \
        if len(sel) else np.zeros(0, dtype=np.int64)
    unsel = np.array([b for b in range(N) if b not in selset], dtype=np.int64)
    out = np.zeros((G, d))
    for g in range(G):
        z = (Ktok[tok] @ q[g]) / math.sqrt(d)                          # exact logits
        terms = [z]
        if compensate and len(unsel):
            zb = (kbar[unsel] @ q[g]) / math.sqrt(d)
            terms.append(np.log(n[unsel].astype(np.float64)) + zb)     # ln(|b| e^zbar)
        m = max(t.max() for t in terms if len(t))
        w_exact = np.exp(z - m)
        num = w_exact @ Vtok[tok]
        den = w_exact.sum()
        if compensate and len(unsel):
            w_mean = np.exp(terms[1] - m)
            num = num + w_mean @ vbar[unsel]
            den = den + w_mean.sum()
        out[g] = num / den
    return out


# --------------------------------------------------------------------------
# Whole decode step for one (sequence, KV head)
# --------------------------------------------------------------------------
@dataclass
class HeadState:
    """Cache of one (sequence, KV head): raw tokens plus maintained summaries."""
    K: np.ndarray                      # [capacity, d] float64 token keys
    V: np.ndarray                      # [capacity, d] float64 token values
    L: int                             # tokens held
    r: int
    n: np.ndarray = field(default=None)
    kbar: np.ndarray = field(default=None)
    Dbar: np.ndarray = field(default=None)
    vbar: np.ndarray = field(default=None)

    def summarise(self):
        self.n, self.kbar, self.Dbar, self.vbar = block_summaries(self.K[: self.L], self.V[: self.L], self.r)
        return self

    def append(self, k_new: np.ndarray, v_new: np.ndarray):
        """Write token L and recompute the (open) block that holds it from its tokens."""
        self.K[self.L] = k_new
        self.V[self.L] = v_new
        self.L += 1
        N = num_blocks(self.L)
        b = N - 1
        s = BLOCK * b
        nb, kb, Db, vb = block_summaries(self.K[s: self.L], self.V[s: self.L], self.r)
        if len(self.n) < N:
            d = self.K.shape[1]
            self.n = np.concatenate([self.n, [0]])
            self.kbar = np.vstack([self.kbar, np.zeros((1, d))])
            self.vbar = np.vstack([self.vbar, np.zeros((1, d))])
            self.Dbar = np.vstack([self.Dbar, np.zeros((1, self.r))])
        self.n[b], self.kbar[b], self.Dbar[b], self.vbar[b] = nb[0], kb[0], Db[0], vb[0]
        return self


@dataclass
class StepResult:
    scores: Scores
    sel: np.ndarray
    out: np.ndarray
    gap: float


def decode_head(state: HeadState, q: np.ndarray, K_blocks: int,
                second_order_mass: bool = True, variance_factor: bool = True,
                compensate: bool = True) -> StepResult:
    """Score, select and attend for one (sequence, KV head) whose cache (and
    summaries) already hold the current token."""
    sc = block_scores(q, state.n, state.kbar, state.Dbar, second_order_mass, variance_factor)
    sel = select_blocks(sc.S, K_blocks)
    out = compkv_attend(q, state.K[: state.L], state.V[: state.L], sel,
                        state.n, state.kbar, state.vbar, compensate)
    return StepResult(scores=sc, sel=sel, out=out, gap=boundary_gap(sc.S, K_blocks))


# --------------------------------------------------------------------------
# Definitions used by the theory checks   ("어떻게 동작하나")
# --------------------------------------------------------------------------
def dense_attention(q: np.ndarray, Ktok: np.ndarray, Vtok: np.ndarray) -> np.ndarray:
    """Textbook softmax(q K^T / sqrt(d)) V, [G, d]."""
    d = q.shape[1]
    z = (q @ Ktok.T) / math.sqrt(d)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    return p @ Vtok


def token_logits(qg: np.ndarray, Ktok: np.ndarray) -> np.ndarray:
    return (Ktok @ qg) / math.sqrt(len(qg))


def exact_block_stats(qg: np.ndarray, Ktok: np.ndarray, L: int):
    """Per block, from the tokens: log Z_b = log sum_{j in b} e^{z_j}, the exact
    mean logit, the exact population logit variance, and the exact mass p_b."""
    z = token_logits(qg, Ktok[:L])
    n = block_counts(L)
    N = len(n)
    logZ = np.zeros(N)
    zmean = np.zeros(N)
    zvar = np.zeros(N)
    for b in range(N):
        zb = z[BLOCK * b: BLOCK * b + n[b]]
        mb = zb.max()
        logZ[b] = mb + math.log(np.exp(zb - mb).sum())
        zmean[b] = zb.mean()
        zvar[b] = ((zb - zmean[b]) ** 2).mean()
    p = np.exp(logZ - _logsumexp(logZ, axis=0))
    return logZ, zmean, zvar, p


def compensated_token_distribution(qg: np.ndarray, Ktok: np.ndarray, L: int, sel,
                                   compensate: bool = True) -> np.ndarray:
    """Token-level distribution of Mean compensation: every logit of an
    unselected block replaced by that block's mean logit (compensate=True), or
    unselected blocks removed (compensate=False).  Length L, sums to 1."""
    z = token_logits(qg, Ktok[:L]).copy()
    n = block_counts(L)
    selset = set(int(b) for b in sel)
    keep = np.ones(L, dtype=bool)
    for b in range(len(n)):
        if b in selset:
            continue
        s, e = BLOCK * b, BLOCK * b + n[b]
        if compensate:
            z[s:e] = z[s:e].mean()
        else:
            keep[s:e] = False
    zz = np.where(keep, z, -np.inf)
    m = zz[keep].max()
    p = np.where(keep, np.exp(zz - m), 0.0)
    return p / p.sum()


def kl_divergence(p: np.ndarray, pref: np.ndarray) -> float:
    """KL(p || pref) = sum_j p_j ln(p_j / pref_j) over the support of p."""
    m = p > 0
    return float(np.sum(p[m] * (np.log(p[m]) - np.log(pref[m]))))


def selection_loss_closed_form(qg: np.ndarray, Ktok: np.ndarray, L: int, sel) -> float:
    """KL(compensated || original) for one query head, from block quantities:
    -ln(1 - sum_{b not in S} p_b (1 - |b| e^{zbar_b} / Z_b))."""
    logZ, zmean, _, p = exact_block_stats(qg, Ktok, L)
    n = block_counts(L)
    selset = set(int(b) for b in sel)
    acc = 0.0
    for b in range(len(n)):
        if b not in selset:
            acc += p[b] * (1.0 - math.exp(math.log(n[b]) + zmean[b] - logZ[b]))
    return -math.log1p(-acc)


def block_loss_term(p_b: float, n_b: int, zmean_b: float, logZ_b: float) -> float:
    """Per-block term p_b (1 - |b| e^{zbar_b} / Z_b) of the selection loss."""
    return p_b * (1.0 - math.exp(math.log(n_b) + zmean_b - logZ_b))
