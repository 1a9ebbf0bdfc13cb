"""Drives a synthetic workload through the CUDA path and the fp64 oracle side by side.

Inputs come from `synth` (seeded draws only).  The oracle receives the exact
bytes the GPU holds (bf16 tokens and fp32 queries, upcast), never anything the
CUDA path computed.  Before each decode step, every (sequence, head) the
oracle follows gets the gap guarantee: if its relative score gap at the
Top-K boundary is <= 1e-4, that GQA group's queries are redrawn (a new attempt
counter) so fp32-vs-fp64 rounding cannot flip the selection.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import synth

GAP = 1e-4
TOL_SUMMARY = 1e-4      # per row, ||delta||_inf / ||ref||_inf
TOL_SCORE = 1e-4        # per element, relative, with a floor of 1e-30 * max S
TOL_OUT = 2e-3          # max abs on the attention output


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


# compkv_config.variant bits and the oracle switches they correspond to
VARIANT_FIRST_ORDER_MASS = 1
VARIANT_NO_VARIANCE_FACTOR = 2
VARIANT_NO_COMPENSATION = 4


def oracle_flags(variant: int) -> dict:
    return dict(second_order_mass=not (variant & VARIANT_FIRST_ORDER_MASS),
                variance_factor=not (variant & VARIANT_NO_VARIANCE_FACTOR),
                compensate=not (variant & VARIANT_NO_COMPENSATION))


class Run:
    """One workload: the GPU cache (prefilled) and oracle states for `heads`.

    heads: iterable of (layer, seq, head) the oracle follows, or "all".
    variant: compkv_config.variant of the cache; the oracle runs the same ablation.
    """

    def __init__(self, wl: synth.Workload, heads="all", device="cuda", variant=0, kv_memory="device"):
        from block_sparse_kv_summary_gb300.cache import CompKVCache
        self.wl = wl
        self.variant = variant
        self.flags = oracle_flags(variant)
        self.lens = synth.sequence_lengths(wl)
        self.caps = synth.capacity_tokens(wl)
        self.cache = CompKVCache(num_layers=wl.layers, batch=wl.batch, num_kv_heads=wl.num_kv_heads,
                                 group_size=wl.group_size, head_dim=wl.head_dim, r=wl.r,
                                 budget_tokens=wl.budget_tokens, capacity_tokens=self.caps, device=device,
                                 variant=variant, kv_memory=kv_memory)
        if heads == "all":
            heads = [(l, s, h) for l in range(wl.layers) for s in range(wl.batch) for h in range(wl.num_kv_heads)]
        self.heads = sorted(set(heads))
        self.future = {}
        self.states = {}
        self.step_no = [0] * wl.layers
        for layer in range(wl.layers):
            for s in range(wl.batch):
                K, V = synth.sequence_tokens(wl, layer, s, self.caps[s], self.lens[s], device=device)
                L = self.lens[s]
                for h in range(wl.num_kv_heads):
                    kv, vv = self.cache.token_view(layer, s, h)
                    kv[:L] = K[h, :L]
                    vv[:L] = V[h, :L]
                    if (layer, s, h) in self.heads:
                        Kh, Vh = f64(K[h]), f64(V[h])
                        Kh[L:] = np.nan   # appended tokens reach the oracle only through append
                        Vh[L:] = np.nan
                        self.states[(layer, s, h)] = O.HeadState(K=Kh, V=Vh, L=L, r=wl.r).summarise()
                self.future[(layer, s)] = (K[:, L:L + wl.steps].contiguous(), V[:, L:L + wl.steps].contiguous())
                del K, V
            self.cache.prefill(layer, self.lens)
        torch.cuda.synchronize()

    # ------------------------------------------------------------------
    def new_tokens(self, layer, step):
        k = torch.stack([self.future[(layer, s)][0][:, step] for s in range(self.wl.batch)]).contiguous()
        v = torch.stack([self.future[(layer, s)][1][:, step] for s in range(self.wl.batch)]).contiguous()
        return k, v

    def oracle_append(self, layer, k_new, v_new):
        kn, vn = f64(k_new), f64(v_new)
        for (l, s, h), st in self.states.items():
            if l == layer:
                st.append(kn[s, h], vn[s, h])

    def choose_queries(self, layer, step):
        """Queries for this step with the gap guarantee on every followed head.
        Returns (q tensor on device, {(s, h): oracle StepResult})."""
        wl = self.wl
        attempts, results = {}, {}
        for (l, s, h), st in self.states.items():
            if l != layer:
                continue
            att = 0
            while True:
                q = synth.queries(wl, layer, s, h, step, att).astype(np.float64)
                sc = O.block_scores(q, st.n, st.kbar, st.Dbar, self.flags["second_order_mass"],
                                    self.flags["variance_factor"])
                if O.boundary_gap(sc.S, wl.K_blocks) > GAP:
                    break
                att += 1
                assert att < 50, "gap guarantee did not converge"
            attempts[(s, h)] = att
            results[(s, h)] = O.decode_head(st, q, wl.K_blocks, **self.flags)
        q = torch.from_numpy(synth.step_queries(wl, layer, step, attempts)).to(self.cache.device)
        return q, results

    def decode_step(self, layer):
        """Append + oracle + GPU decode for the next step of `layer`."""
        step = self.step_no[layer]
        k_new, v_new = self.new_tokens(layer, step)
        self.oracle_append(layer, k_new, v_new)
        q, results = self.choose_queries(layer, step)
        sel = self.cache.new_sel()
        out = self.cache.decode(layer, q, k_new, v_new, sel=sel)
        self.step_no[layer] += 1
        return q, sel, out, results


# ---------------------------------------------------------------------- checks
def check_summaries(run: Run, layer, s, h, blocks=None):
    """Every summary row (or the rows in `blocks`) of kbar, Dbar and vbar within
    TOL_SUMMARY of the oracle, relative to the row's largest magnitude."""
    st = run.states[(layer, s, h)]
    kbar, dbar, vbar = run.cache.summary_view(layer, s, h)
    N = O.num_blocks(st.L)
    idx = np.arange(N) if blocks is None else np.asarray(blocks)
    worst = 0.0
    for name, got, ref in (("kbar", kbar, st.kbar), ("Dbar", dbar, st.Dbar), ("vbar", vbar, st.vbar)):
        g = f64(got[:N])[idx]
        r = ref[idx]
        den = np.maximum(np.abs(r).max(axis=1), 1e-30)
        err = np.abs(g - r).max(axis=1) / den
        b = int(np.argmax(err))
        assert err[b] <= TOL_SUMMARY, f"{name} row {int(idx[b])} of {(layer, s, h)}: rel err {err[b]:.3e}"
        worst = max(worst, float(err[b]))
    return worst


def check_scores(S_gpu: np.ndarray, S_ref: np.ndarray):
    tol = TOL_SCORE * np.abs(S_ref) + 1e-30 * np.abs(S_ref).max()
    err = np.abs(S_gpu - S_ref)
    bad = np.nonzero(err > tol)[0]
    assert len(bad) == 0, f"{len(bad)} scores off, worst rel {(err / np.maximum(np.abs(S_ref), 1e-300)).max():.3e}"
    return float((err / np.maximum(np.abs(S_ref), 1e-30 * np.abs(S_ref).max())).max())


def check_step(run: Run, layer, sel, out, results):
    """Selection bit-exact, output within 2e-3, for every followed (seq, head)."""
    wl = run.wl
    sel_h = sel.cpu().numpy()
    out_h = f64(out)
    G = wl.group_size
    worst = 0.0
    for (s, h), res in results.items():
        K = wl.K_blocks
        exp_sel = np.full(K, -1, dtype=np.int64)
        exp_sel[:len(res.sel)] = res.sel
        assert np.array_equal(sel_h[s, h], exp_sel), \
            f"selection differs at {(layer, s, h)}:\n gpu {sel_h[s, h]}\n ref {exp_sel}"
        err = np.abs(out_h[s, h * G:(h + 1) * G] - res.out).max()
        worst = max(worst, err)
        assert err <= TOL_OUT, f"output of {(layer, s, h)} off by {err:.3e}"
    return worst
