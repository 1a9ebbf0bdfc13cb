#!/usr/bin/env python3
"""Benchmark of the CompKV decode step on one GB300 (replicas on N GPUs).

Workload: a Qwen3-8B-shaped layer (32 query / 8 KV heads, d 128), 131072-token
context, 2048-token budget (K = 128 blocks), r = 4, bf16 K/V and fp32
summaries in HBM, 64 consecutive decode steps each appending one token.  A
step = one compkv_decode: append + score + select + attend with Mean
compensation.  R independent layer caches are rotated so that ~R x 77 MB is
touched between two visits of the same data (larger than the 129 MB L2); after
64 steps a layer's seq_len is rewound, which replays the same 64 steps exactly
(the append recomputes the open block from its tokens).

Prints one JSON line.  `--impl reference` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode-step µs and achieved HBM GB/s (% of GB300 peak), 32K–128K ctx"
UNIT = "us/step"
WORKLOAD = "qwen8b_128k"
FALLBACK_HBM_GBS = 6800.0
BLOCK = 16


# ----------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel_file: str, kernel: str):
    """DRAM bytes per launch of `kernel` (full-size workload) from the committed ncu
    summary, or None if absent or taken on a different version of the kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(os.path.basename(kernel_file), {})
    src = os.path.join(ROOT, "block_sparse_kv_summary_gb300", "csrc", os.path.basename(kernel_file))
    if rec.get("source_sha") != source_sha(src):
        return None
    return rec.get("kernels", {}).get(kernel, {}).get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- workload
class QwenLayers:
    """R independent Qwen3-8B-shaped layer caches on one GPU, with staged step inputs."""

    def __init__(self, R: int, device):
        from block_sparse_kv_summary_gb300.cache import CompKVCache
        wl = synth.WORKLOADS[WORKLOAD]
        self.wl, self.R, self.device = wl, R, device
        self.L0 = wl.context
        self.cap = synth.capacity_tokens(wl)[0]
        self.cache = CompKVCache(num_layers=R, batch=1, num_kv_heads=wl.num_kv_heads, group_size=wl.group_size,
                                 head_dim=wl.head_dim, r=wl.r, budget_tokens=wl.budget_tokens,
                                 capacity_tokens=self.cap, device=device)
        S, H, G, d = wl.steps, wl.num_kv_heads, wl.group_size, wl.head_dim
        self.k_new = torch.empty((R, S, 1, H, d), dtype=torch.bfloat16, device=device)
        self.v_new = torch.empty_like(self.k_new)
        self.q = torch.empty((R, S, 1, H * G, d), dtype=torch.float32, device=device)
        for layer in range(R):
            K, V = synth.sequence_tokens(wl, layer, 0, self.cap, self.L0, device=device)
            for h in range(H):
                kv, vv = self.cache.token_view(layer, 0, h)
                kv[:self.L0] = K[h, :self.L0]
                vv[:self.L0] = V[h, :self.L0]
            self.k_new[layer, :, 0] = K[:, self.L0:self.L0 + S].transpose(0, 1)
            self.v_new[layer, :, 0] = V[:, self.L0:self.L0 + S].transpose(0, 1)
            for c in range(S):
                self.q[layer, c] = torch.from_numpy(synth.step_queries(wl, layer, c)).to(device)
            del K, V
            self.cache.prefill(layer, [self.L0])
        self.out = self.cache.new_out()
        self.sel = self.cache.new_sel()
        self.i = 0
        torch.cuda.synchronize(device)

    def step(self):
        layer = self.i % self.R
        c = (self.i // self.R) % self.wl.steps
        if c == 0 and self.i >= self.R:
            self.cache.seq_len[layer].fill_(self.L0)   # replay the same 64 steps
        self.cache.decode(layer, self.q[layer, c], self.k_new[layer, c], self.v_new[layer, c],
                          out=self.out, sel=self.sel)
        self.i += 1

    # algorithmic bytes, averaged over the 64-step cycle
    def bytes_per_step(self):
        wl = self.wl
        d, r, H, G, K = wl.head_dim, wl.r, wl.num_kv_heads, wl.group_size, wl.K_blocks
        summ, sel_kv, score = 0.0, 0.0, 0.0
        for c in range(wl.steps):
            L = self.L0 + c + 1
            N = (L + BLOCK - 1) // BLOCK
            n_last = L - BLOCK * (N - 1)
            summ += H * N * (2 * d + r + 1) * 4
            score += H * N * (2 * d + r) * 4
            sel_tok = min(N, K) * BLOCK - (BLOCK - n_last)
            sel_kv += H * sel_tok * d * 2 * 2
        S = wl.steps
        qo = 2 * H * G * d * 4
        return {"summary": summ / S, "selected_kv": sel_kv / S, "q_out": qo,
                "total": summ / S + sel_kv / S + qo, "score_kernel": score / S}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_baseline(budget_s: float = 12.0, heads=(0, 1)):
    """The fp64 oracle timed on the host on a bounded sample of the same workload:
    decode steps of `heads` of layer 0, until `budget_s` of CPU time is spent.
    Returns (us per full decode step, sample description, steps timed)."""
    import oracle as O
    wl = synth.WORKLOADS[WORKLOAD]
    L0, cap = wl.context, synth.capacity_tokens(wl)[0]
    K, V = synth.sequence_tokens(wl, 0, 0, cap, L0, device="cpu")
    states = {}
    for h in heads:
        Kh = K[h].float().numpy().astype(np.float64)
        Vh = V[h].float().numpy().astype(np.float64)
        states[h] = (O.HeadState(K=Kh.copy(), V=Vh.copy(), L=L0, r=wl.r).summarise(), Kh, Vh)
    done, t_total = 0, 0.0
    for c in range(wl.steps):
        for h in heads:
            st, Kh, Vh = states[h]
            q = synth.queries(wl, 0, 0, h, c).astype(np.float64)
            t0 = time.perf_counter()
            st.append(Kh[L0 + c], Vh[L0 + c])
            O.decode_head(st, q, wl.K_blocks)
            t_total += time.perf_counter() - t0
            done += 1
        if t_total > budget_s:
            break
    per_head = t_total / done
    us = per_head * wl.num_kv_heads * 1e6
    sample = (f"fp64 numpy oracle, {done} (head, step) decode steps of layer 0 (heads {list(heads)}, "
              f"steps 0..{done // len(heads) - 1}), scaled x{wl.num_kv_heads} heads per decode step")
    return us, sample, done


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64000)
    ap.add_argument("--warmup", type=int, default=640)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=8, help="independent layer caches rotated (L2 hygiene)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    ws, rank, local = dist_env()
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        return run_reference(args, ws, rank)

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import block_sparse_kv_summary_gb300 as P
    if rank == 0:
        P.build()
    barrier(ws)
    P.lib()

    work = QwenLayers(args.layers, device)
    cache = work.cache
    for _ in range(args.warmup):
        work.step()
    torch.cuda.synchronize(device)
    if cache.device_status() != 0:
        raise RuntimeError("device status error after warm-up: " + P.compkv_last_error())

    # ---- timed region: K decode steps, device time by CUDA events on the launch stream
    stream = torch.cuda.current_stream(device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize(device)
    n0 = cache.launch_count()
    ev0.record(stream)
    for _ in range(args.steps):
        work.step()
    ev1.record(stream)
    torch.cuda.synchronize(device)
    barrier(ws)
    clk = clocks.stop()
    launches = cache.launch_count() - n0
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, ws, device)
    if cache.device_status() != 0:
        raise RuntimeError("device status error in the timed region: " + P.compkv_last_error())

    # ---- device time per call, then per kernel of the chain (library events), separate passes
    kp = min(args.steps, 6400)
    fam_ms = {}
    for level, fams in ((1, ("decode",)), (2, ("k_score", "k_post"))):
        cache.profile(level)
        for fam in fams:
            cache.profile_read(fam)
        for _ in range(kp):
            work.step()
        torch.cuda.synchronize(device)
        fam_ms.update({fam: cache.profile_read(fam) for fam in fams})
        cache.profile(0)

    # ---- end to end through the public API with pinned host buffers
    ke = min(args.steps, 2000)
    R, S = work.R, work.wl.steps
    h_q = work.q.cpu().pin_memory()
    h_k = work.k_new.cpu().pin_memory()
    h_v = work.v_new.cpu().pin_memory()
    d_q, d_k, d_v = torch.empty_like(work.q[0, 0]), torch.empty_like(work.k_new[0, 0]), torch.empty_like(work.v_new[0, 0])
    h_out = torch.empty(work.out.shape, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize(device)
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(ke):
        layer, c = work.i % R, (work.i // R) % S
        if c == 0 and work.i >= R:
            cache.seq_len[layer].fill_(work.L0)
        d_q.copy_(h_q[layer, c], non_blocking=True)
        d_k.copy_(h_k[layer, c], non_blocking=True)
        d_v.copy_(h_v[layer, c], non_blocking=True)
        cache.decode(layer, d_q, d_k, d_v, out=work.out)
        h_out.copy_(work.out, non_blocking=True)
        stream.synchronize()
        work.i += 1
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, ws, device)
    if cache.device_status() != 0:
        raise RuntimeError("device status error in the e2e pass: " + P.compkv_last_error())

    if rank != 0:
        barrier(ws)
        return 0

    # ---- numbers
    by = work.bytes_per_step()
    us_step = ms_max * 1e3 / (args.steps * ws)        # whole-job time per decode step
    us_step_replica = ms_max * 1e3 / args.steps
    peak, peak_kind = measured_peaks()
    step_gbs = by["total"] / (us_step_replica * 1e-6) / 1e9
    kernels = {f: {"launches": n, "avg_us": (m * 1e3 / n if n else None)} for f, (m, n) in fam_ms.items()}
    kernels["decode"]["note"] = "one decode call: the two PDL-chained kernels"
    for f in ("k_score", "k_post"):
        kernels[f]["note"] = "timed alone (events between the kernels stop their early launch)"
    # the dominant HBM kernel: k_score streams the summaries (kbar, Dbar, vbar) of every block
    ks_us = kernels["k_score"]["avg_us"]
    ks_gbs = by["score_kernel"] / (ks_us * 1e-6) / 1e9
    traffic = ncu_traffic("decode_kernels.cu", "k_score")
    e2e_us = e2e_s * 1e6 / (ke * ws)
    cpu = None
    if not args.no_cpu_baseline:
        cpu_us, sample, _ = oracle_baseline()
        cpu = {"value": cpu_us, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample}
    line = {
        "metric": METRIC, "value": us_step, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us_step_replica / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 (bf16 K/V, fp32 summaries)",
        "data": "synthetic (seeded generator: per-block centres + LogUniform within-block noise, "
                "2 outlier channels x5, 3 needles; random queries)",
        "config": {"workload": "Qwen3-8B-shaped layer: 32 q / 8 KV heads, d 128, ctx 131072 (+64 decode steps), "
                               "budget 2048 tokens (K 128 blocks), r 4, block 16, batch 1",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": f"inputs larger than L2: {work.R} independent layer caches rotated, "
                         f"{work.R * by['total'] / 1e6:.0f} MB touched between visits of one layer",
                   "hbm_gbs_step": step_gbs,
                   "step_frac_of_peak": step_gbs / peak,
                   "bytes_per_step": by},
        "roofline": {"bound": "hbm",
                     "kernel": "k_score<128,4,decode> (two warps per 64-block item: append, kbar/Dbar/vbar "
                               "bulk-copy stream, zbar, sigma2, item LSE records, compensation partials)",
                     "achieved": ks_gbs, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": ks_gbs / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": by["score_kernel"], "avg_launch_us": ks_us},
        "kernels": kernels,
        "e2e": {"value": e2e_us, "unit": UNIT,
                "h2d_bytes_per_step": int(work.q[0, 0].numel() * 4 + 2 * work.k_new[0, 0].numel() * 2),
                "d2h_bytes_per_step": int(work.out.numel() * 4)},
        "gpu_launches": int(launches),
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    barrier(ws)
    return 0


def run_reference(args, ws, rank):
    """The oracle, as it stands, on the host cores: rank 0 only."""
    if rank != 0:
        return 0
    budget = 60.0
    us, sample, done = oracle_baseline(budget_s=budget)
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": ws,
        "steps": done, "warmup": 0, "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same generator as the GPU arm)",
        "config": {"workload": "Qwen3-8B-shaped layer: 32 q / 8 KV heads, d 128, ctx 131072 (+64 decode steps), "
                               "budget 2048 tokens (K 128 blocks), r 4, block 16, batch 1",
                   "requested_steps": args.steps,
                   "note": f"each timed step is one (head, step) oracle decode; capped at ~{budget:.0f} s of CPU work"},
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
