"""Seeded synthetic inputs for the CompKV decode step.

This module only draws random numbers: it holds none of the method's
arithmetic (no summaries, scores, selection or attention), so both the CUDA
path's tests and the fp64 oracle can take their inputs from it.

Recipe (stand-in for the long-context suites the CompKV page evaluates on,
"전제와 한계": 32K-128K contexts, block size 16, r = 4):
  * keys, per (layer, sequence, KV head, 16-token block): a centre c_b ~ N(0, I_d)
    plus within-block noise N(0, s_b^2 I) with s_b ~ LogUniform(s_lo, s_hi);
  * two outlier channels per (layer, sequence, head), centre and noise times 5;
  * values N(0, 1); everything cast to bf16;
  * queries N(0, 1) fp32, drawn afresh for every decode step, one seed per
    (layer, sequence, KV head, step, attempt) so that one GQA group's queries
    can be redrawn without touching the others;
  * three needle tokens per (sequence, head) in distinct non-forced blocks,
    whose key is gamma * u, u the unit direction of the group's mean step-0
    query and gamma chosen so that the mean step-0 query gives it logit +6;
  * the token stream is drawn for the whole capacity up front, so appended
    tokens continue their block's centre and scale, and a new centre starts
    with every new block;
  * the batched workload draws every sequence length from U[8192, 131072].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch

BLOCK = 16


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    batch: int
    num_kv_heads: int
    group_size: int
    head_dim: int
    r: int
    context: int                 # uniform prefill length (ignored when ragged)
    budget_tokens: int
    steps: int                   # decode steps, one appended token each
    s_lo: float = 0.05
    s_hi: float = 1.0
    ragged: tuple | None = None  # (lo, hi) for per-sequence lengths
    lengths: tuple | None = None # explicit per-sequence lengths (test edge cases)
    needles: int = 3
    seed: int = 20261202

    @property
    def num_q_heads(self) -> int:
        return self.num_kv_heads * self.group_size

    @property
    def K_blocks(self) -> int:
        return self.budget_tokens // BLOCK


WORKLOADS = {
    # d 64, 2 KV heads x G 4, ctx 1024 -> 1025 tokens after the append (65 blocks), K 8
    "tiny": Workload("tiny", 1, 1, 2, 4, 64, 4, 1024, 128, 1),
    # Llama-3.1-8B-shaped layer, 32K context, 512-token budget
    "llama8b_32k": Workload("llama8b_32k", 1, 1, 8, 4, 128, 4, 32768, 512, 1),
    # Qwen3-8B-shaped layer, 128K context, 2048-token budget, 64 decode steps
    "qwen8b_128k": Workload("qwen8b_128k", 1, 1, 8, 4, 128, 4, 131072, 2048, 64),
    # Qwen3-32B-shaped layer, 64K context, 1024-token budget, r = d
    "qwen32b_64k": Workload("qwen32b_64k", 1, 1, 8, 8, 128, 128, 65536, 1024, 1,
                            s_lo=0.01, s_hi=2.0),
    # 32 Llama-3.1-8B-shaped layers x 16 ragged sequences, 16 steps
    "batched": Workload("batched", 32, 16, 8, 4, 128, 4, 0, 1024, 16,
                        ragged=(8192, 131072)),
}


def seed_for(base: int, *counters: int) -> int:
    """A 63-bit seed derived from a base seed and a tuple of counters."""
    ss = np.random.SeedSequence([int(base) & 0xFFFFFFFF, *[int(c) & 0xFFFFFFFF for c in counters]])
    st = ss.generate_state(2, dtype=np.uint32)
    return ((int(st[0]) << 32) | int(st[1])) & ((1 << 63) - 1)


def sequence_lengths(wl: Workload) -> list[int]:
    """Prefill length of every sequence (shared by all layers)."""
    if wl.lengths is not None:
        return [int(x) for x in wl.lengths]
    if wl.ragged is None:
        return [wl.context] * wl.batch
    rng = np.random.Generator(np.random.PCG64(seed_for(wl.seed, 7)))
    lo, hi = wl.ragged
    return [int(x) for x in rng.integers(lo, hi + 1, size=wl.batch)]


def capacity_tokens(wl: Workload) -> list[int]:
    """Per-sequence capacity: prefill + steps, rounded up to whole blocks."""
    return [((L + wl.steps + BLOCK - 1) // BLOCK) * BLOCK for L in sequence_lengths(wl)]


def queries(wl: Workload, layer: int, seq: int, head: int, step: int, attempt: int = 0) -> np.ndarray:
    """fp32 [G, d] queries of one GQA group for one decode step."""
    rng = np.random.Generator(np.random.PCG64(seed_for(wl.seed, 11, layer, seq, head, step, attempt)))
    return rng.standard_normal((wl.group_size, wl.head_dim)).astype(np.float32)


def step_queries(wl: Workload, layer: int, step: int, attempts=None) -> np.ndarray:
    """fp32 [B, Hq, d] for one layer and step; query head j belongs to KV head j // G.
    attempts: optional {(seq, head): attempt} for groups that were redrawn."""
    attempts = attempts or {}
    out = np.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=np.float32)
    G = wl.group_size
    for s in range(wl.batch):
        for h in range(wl.num_kv_heads):
            out[s, h * G:(h + 1) * G] = queries(wl, layer, s, h, step, attempts.get((s, h), 0))
    return out


def needle_positions(wl: Workload, layer: int, seq: int, head: int, prefill_len: int) -> list[int]:
    """Token positions of the needles: distinct blocks in [1, N0 - 3), N0 the
    prefill block count, so no needle block is ever forced."""
    N0 = (prefill_len + BLOCK - 1) // BLOCK
    hi = N0 - 3
    if hi - 1 < wl.needles:
        return []
    rng = np.random.Generator(np.random.PCG64(seed_for(wl.seed, 13, layer, seq, head)))
    blocks = rng.choice(np.arange(1, hi), size=wl.needles, replace=False)
    offs = rng.integers(0, BLOCK, size=wl.needles)
    return sorted(int(b) * BLOCK + int(o) for b, o in zip(blocks, offs))


def sequence_tokens(wl: Workload, layer: int, seq: int, cap_tokens: int, prefill_len: int,
                    device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """bf16 keys and values [Hkv, cap_tokens, d] for one (layer, sequence):
    the prefill tokens followed by the tokens the decode steps will append."""
    Hkv, d = wl.num_kv_heads, wl.head_dim
    nb = cap_tokens // BLOCK
    gen = torch.Generator(device=device)
    gen.manual_seed(seed_for(wl.seed, 3, layer, seq))
    f32 = dict(dtype=torch.float32, device=device, generator=gen)
    centre = torch.randn(Hkv, nb, 1, d, **f32)
    u = torch.rand(Hkv, nb, 1, 1, **f32)
    scale = torch.exp(math.log(wl.s_lo) + u * (math.log(wl.s_hi) - math.log(wl.s_lo)))
    K = torch.randn(Hkv, nb, BLOCK, d, **f32)
    K.mul_(scale).add_(centre)
    del centre, u, scale
    # two outlier channels per head
    rng = np.random.Generator(np.random.PCG64(seed_for(wl.seed, 5, layer, seq)))
    for h in range(Hkv):
        ch = torch.as_tensor(rng.choice(d, size=2, replace=False), device=device)
        K[h, :, :, ch] *= 5.0
    K = K.reshape(Hkv, cap_tokens, d)
    # needles, aimed at the group's mean step-0 query
    for h in range(Hkv):
        pos = needle_positions(wl, layer, seq, h, prefill_len)
        if not pos:
            continue
        qm = queries(wl, layer, seq, h, 0).astype(np.float64).mean(axis=0)
        nrm = float(np.linalg.norm(qm))
        gamma = 6.0 * math.sqrt(d) / nrm
        key = torch.from_numpy((gamma * qm / nrm).astype(np.float32)).to(device)
        for p in pos:
            K[h, p] = key
    Kb = K.to(torch.bfloat16)
    del K
    V = torch.randn(Hkv, cap_tokens, d, **f32).to(torch.bfloat16)
    return Kb, V


def small_variant(name: str, **changes) -> Workload:
    """A copy of a named workload with some fields changed (test sizes)."""
    return replace(WORKLOADS[name], **changes)
