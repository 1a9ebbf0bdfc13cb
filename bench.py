#!/usr/bin/env python3
"""Benchmark of the CompKV decode step on one GB300 (replicas on N GPUs).

A step is one compkv_decode call: append one token, score every block from
its summary, select the sink, the two most recent blocks and the Top-K of
S_b, attend exactly to the selected blocks and add Mean compensation for the
rest.  Workloads (--workload), all bf16 K/V with fp32 summaries resident in HBM:

  qwen8b_128k  (default, the headline) Qwen3-8B-shaped layer: 32 q / 8 KV
               heads, d 128, 131072-token context, 2048-token budget, r 4,
               64 consecutive decode steps
  llama8b_32k  Llama-3.1-8B-shaped layer: 32 q / 8 KV heads, 32K context,
               512-token budget, r 4
  qwen32b_64k  Qwen3-32B-shaped layer: 64 q / 8 KV heads (G 8), 64K context,
               1024-token budget, r = d = 128
  batched      32 Llama-3.1-8B-shaped layers x 16 sequences of ragged length
               (U[8192, 131072]), 1024-token budget; one step = the 32 layers
  tiny         2 KV heads x G 4, d 64, 1024-token context, 128-token budget

R independent layer caches are rotated so that several times the L2 (129 MB)
is touched between two visits of the same data; after the workload's steps a
layer's lengths are rewound, which replays the same steps exactly (the append
recomputes the open block from its tokens).

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
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-step µs and achieved HBM GB/s (% of GB300 peak), 32K–128K ctx"
UNIT = "us/step"
FALLBACK_HBM_GBS = 6800.0
BLOCK = 16
L2_BYTES = 129e6

# name -> (synth workload, changes for the bench, rotated layer caches, description)
WORKLOADS = {
    "qwen8b_128k": ("qwen8b_128k", {}, 8,
                    "Qwen3-8B-shaped layer: 32 q / 8 KV heads, d 128, ctx 131072 (+64 decode steps), "
                    "budget 2048 tokens (K 128 blocks), r 4, block 16, batch 1"),
    "llama8b_32k": ("llama8b_32k", {"steps": 64}, 24,
                    "Llama-3.1-8B-shaped layer: 32 q / 8 KV heads, d 128, ctx 32768 (+64 decode steps), "
                    "budget 512 tokens (K 32 blocks), r 4, block 16, batch 1"),
    "qwen32b_64k": ("qwen32b_64k", {"steps": 64}, 8,
                    "Qwen3-32B-shaped layer: 64 q / 8 KV heads (G 8), d 128, ctx 65536 (+64 decode steps), "
                    "budget 1024 tokens (K 64 blocks), r 128, block 16, batch 1"),
    "batched": ("batched", {}, 1,
                "32 Llama-3.1-8B-shaped layers x 16 sequences (ragged U[8192, 131072]), 32 q / 8 KV heads, "
                "d 128, budget 1024 tokens (K 64 blocks), r 4, 16 decode steps; one step = 32 layer calls"),
    "tiny": ("tiny", {"steps": 64}, 1,
             "2 KV heads x G 4, d 64, ctx 1024 (+64 decode steps), budget 128 tokens (K 8), r 4, batch 1"),
}


# ----------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device):
    if ws == 1:
        return x
    import torch
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


def ncu_traffic(kernel_file: str, kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, or None if absent or taken on a different version of the kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(workload, {}).get(os.path.basename(kernel_file), {})
    src = os.path.join(ROOT, "block_sparse_kv_summary_gb300", "csrc", os.path.basename(kernel_file))
    if rec.get("source_sha") != source_sha(src):
        return None
    return rec.get("kernels", {}).get(kernel, {}).get("dram_bytes_per_launch")


def bench_workload(name, r=None, budget=None, dense=False, layers=None):
    """The synth workload behind a bench workload name, with optional overrides:
    r (variance groups), budget (tokens), or dense (budget covering the whole
    context: every block selected, i.e. exact attention over the cache)."""
    import synth
    base, changes, R, desc = WORKLOADS[name]
    changes = dict(changes)
    if r is not None:
        changes["r"] = int(r)
        desc += f"; r overridden to {r}"
    if dense:
        wl0 = synth.WORKLOADS[base]
        top = max(synth.sequence_lengths(wl0)) + changes.get("steps", wl0.steps)
        budget = ((top + BLOCK - 1) // BLOCK) * BLOCK
        desc += f"; dense: budget {budget} tokens covers the context (every block selected: exact attention)"
    elif budget is not None:
        desc += f"; budget overridden to {budget} tokens"
    if budget is not None:
        changes["budget_tokens"] = int(budget)
    wl = synth.small_variant(base, **changes) if changes else synth.WORKLOADS[base]
    if layers is not None:
        R = int(layers)
        desc += f"; {R} rotated layer cache(s)"
    return wl, R, desc


def step_bytes(wl):
    """Algorithmic bytes per decode call, averaged over the workload's steps:
    the summary rows of every block (of the units that select, N > K), the K/V
    of the selected blocks, q and out (and, per kernel: what the stream reads,
    what the post kernel reads)."""
    import synth
    d, r, H, G, K = wl.head_dim, wl.r, wl.num_kv_heads, wl.group_size, wl.K_blocks
    summ = sel_kv = stream = post = 0.0
    lens = synth.sequence_lengths(wl)
    for c in range(wl.steps):
        for L0 in lens:
            L = L0 + c + 1
            N = (L + BLOCK - 1) // BLOCK
            n_last = L - BLOCK * (N - 1)
            if N > K:  # (with every block selected the summaries are not read)
                summ += H * N * (2 * d + r + 1) * 4
                stream += H * N * (2 * d + r) * 4
            tok = min(N, K) * BLOCK - (BLOCK - n_last)
            sel_kv += H * tok * d * 2 * 2
            post += H * (tok * d * 2 * 2 + min(N, K) * d * 4)
    S = wl.steps
    qo = 2 * wl.batch * H * G * d * 4
    return {"summary": summ / S, "selected_kv": sel_kv / S, "q_out": qo,
            "total": (summ + sel_kv) / S + qo, "k_stream": stream / S, "k_post": post / S + qo}


# ----------------------------------------------------------------------------- device workload
class Layers:
    """R independent layer caches of a workload on one GPU, with the inputs of
    every step staged on the device and the call arguments prepared once."""

    def __init__(self, name, device, kv_memory="device", **overrides):
        import torch

        import synth
        from block_sparse_kv_summary_gb300.cache import CompKVCache
        wl, R, desc = bench_workload(name, **overrides)
        if kv_memory == "host":
            desc += "; K/V rows in page-locked host memory (read over the chip-to-chip link)"
        self.name, self.wl, self.desc, self.device = name, wl, desc, device
        self.R = wl.layers if wl.layers > 1 else R
        self.lens = synth.sequence_lengths(wl)
        self.caps = synth.capacity_tokens(wl)
        B, H, G, d, S = wl.batch, wl.num_kv_heads, wl.group_size, wl.head_dim, wl.steps
        self.cache = CompKVCache(num_layers=self.R, batch=B, num_kv_heads=H, group_size=G, head_dim=d, r=wl.r,
                                 budget_tokens=wl.budget_tokens, capacity_tokens=self.caps, device=device,
                                 kv_memory=kv_memory)
        self.kv_memory = kv_memory
        self.k_new = torch.empty((self.R, S, B, H, d), dtype=torch.bfloat16, device=device)
        self.v_new = torch.empty_like(self.k_new)
        self.q = torch.empty((self.R, S, B, H * G, d), dtype=torch.float32, device=device)
        for layer in range(self.R):
            src_layer = layer if wl.layers > 1 else 0
            for s in range(B):
                K, V = synth.sequence_tokens(wl, src_layer, s, self.caps[s], self.lens[s], device=device)
                L = self.lens[s]
                for h in range(H):
                    kv, vv = self.cache.token_view(layer, s, h)
                    kv[:L] = K[h, :L]
                    vv[:L] = V[h, :L]
                self.k_new[layer, :, s] = K[:, L:L + S].transpose(0, 1)
                self.v_new[layer, :, s] = V[:, L:L + S].transpose(0, 1)
                del K, V
            for c in range(S):
                self.q[layer, c] = torch.from_numpy(synth.step_queries(wl, src_layer, c)).to(device)
            self.cache.prefill(layer, self.lens)
        self.out = self.cache.new_out()
        self.sel = self.cache.new_sel()
        self.lens_dev = torch.tensor(self.lens, dtype=torch.int32, device=device)
        self.call = self.cache.prepared_decode()
        # per (layer, step): the addresses of that call's inputs
        self.args = [[(self.q[layer, c].data_ptr(), self.k_new[layer, c].data_ptr(), self.v_new[layer, c].data_ptr())
                      for c in range(S)] for layer in range(self.R)]
        self.out_ptr, self.sel_ptr = self.out.data_ptr(), self.sel.data_ptr()
        self.calls_per_step = self.R if wl.layers > 1 else 1
        self.i = 0
        torch.cuda.synchronize(device)

    def call_once(self):
        """The next decode call (layer rotation; lengths rewound after the workload's steps)."""
        layer = self.i % self.R
        c = (self.i // self.R) % self.wl.steps
        if c == 0 and self.i >= self.R:
            self.cache.seq_len[layer].copy_(self.lens_dev)   # replay the same steps
        q, k, v = self.args[layer][c]
        self.call(layer, q, k, v, self.out_ptr, self.sel_ptr)
        self.i += 1

    def step(self):
        for _ in range(self.calls_per_step):
            self.call_once()


def trace_spans(cache, work, device, calls=8):
    """Median over `calls` traced decode calls of each kernel's span inside the chain:
    the earliest CTA start to the latest CTA end of the stream and of the post kernel."""
    import torch

    from block_sparse_kv_summary_gb300 import compkv as C
    buf = torch.zeros(1 + 8 * 8192, dtype=torch.int64, device=device)
    C.compkv_trace(cache.ctx, buf.data_ptr(), buf.numel() * 8)
    st, po = [], []
    try:
        for _ in range(calls):
            buf.zero_()
            work.call_once()
            torch.cuda.synchronize(device)
            tr = buf.cpu().numpy()[1:].reshape(-1, 8).astype(np.int64)
            used = tr[:, 2] != 0
            kind = (tr[:, 0] >> 24) & 0xff
            s_rec, p_rec = tr[used & (kind == 0)], tr[used & (kind == 1)]
            if len(s_rec):
                st.append((s_rec[:, 5].max() - s_rec[:, 2].min()) / 1e3)
            if len(p_rec):
                po.append((p_rec[:, 6].max() - p_rec[:, 2].min()) / 1e3)
    finally:
        C.compkv_trace(cache.ctx, 0, 0)
    return {"k_stream": float(np.median(st)) if st else None, "k_post": float(np.median(po)) if po else None}


# ----------------------------------------------------------------------------- CPU oracle
def _oracle_worker(args):
    """One (sequence, KV head) of layer 0, run by the oracle for `steps` decode
    steps after a common start signal; returns seconds spent per step."""
    path_k, path_v, L0, r, K_blocks, qs, steps, barrier_obj = args
    import oracle as O
    Kh = np.load(path_k).astype(np.float64)
    Vh = np.load(path_v).astype(np.float64)
    st = O.HeadState(K=Kh, V=Vh, L=L0, r=r).summarise()
    barrier_obj.wait()
    t0 = time.perf_counter()
    for c in range(steps):
        st.append(Kh[L0 + c], Vh[L0 + c])
        O.decode_head(st, qs[c], K_blocks)
    return (time.perf_counter() - t0) / steps


def oracle_baseline(name, budget_s=8.0, threads=1, **overrides):
    """The fp64 oracle timed on the host on a bounded sample of the workload:
    decode steps of sequence 0 of layer 0.  threads=1: heads one after another
    in this process until `budget_s` of CPU time is spent, scaled to a full
    decode step; threads>1: one process per (sequence, head), all heads of the
    step side by side.  Returns (us per decode call, description, steps, cores)."""
    import multiprocessing as mp
    import tempfile

    import torch

    import oracle as O
    import synth
    wl, _, _ = bench_workload(name, **overrides)
    lens, caps = synth.sequence_lengths(wl), synth.capacity_tokens(wl)
    s = int(np.argmax(lens)) if wl.batch > 1 else 0
    L0, cap = lens[s], caps[s]
    K, V = synth.sequence_tokens(wl, 0, s, cap, L0, device="cpu")
    H = wl.num_kv_heads
    units_per_call = wl.batch * H
    if threads <= 1:
        done, t_total, heads_used = 0, 0.0, set()
        states = {}
        for c in range(wl.steps):
            for h in range(H):
                if h not in states:
                    Kh = K[h].float().numpy().astype(np.float64)
                    Vh = V[h].float().numpy().astype(np.float64)
                    states[h] = (O.HeadState(K=Kh.copy(), V=Vh.copy(), L=L0, r=wl.r).summarise(), Kh, Vh)
                st, Kh, Vh = states[h]
                q = synth.queries(wl, 0, s, h, c).astype(np.float64)
                t0 = time.perf_counter()
                st.append(Kh[L0 + c], Vh[L0 + c])
                O.decode_head(st, q, wl.K_blocks)
                t_total += time.perf_counter() - t0
                done += 1
                heads_used.add(h)
                if t_total > budget_s:
                    break
            if t_total > budget_s:
                break
        per_unit = t_total / done
        desc = (f"fp64 numpy oracle, 1 thread: {done} (head, step) decodes of sequence {s} of layer 0 "
                f"(L0 {L0}), scaled x{units_per_call} units per decode call")
        return per_unit * units_per_call * 1e6, desc, done / units_per_call, 1
    cores = len(os.sched_getaffinity(0))
    workers = min(cores, H)
    tmp = tempfile.mkdtemp(prefix="compkv_oracle_")
    jobs = []
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    bar = mgr.Barrier(workers)
    for h in range(workers):
        pk, pv = os.path.join(tmp, f"k{h}.npy"), os.path.join(tmp, f"v{h}.npy")
        np.save(pk, K[h].float().numpy())
        np.save(pv, V[h].float().numpy())
        jobs.append([pk, pv, L0, wl.r, wl.K_blocks, None, None, bar])
    # steps per head: about budget_s of wall time for the parallel section
    # (a head-step takes about 1.7 us per block on one core)
    est = 1.7e-6 * (L0 / BLOCK) + 1e-3
    steps = max(2, min(wl.steps, int(budget_s / est)))
    for h, j in enumerate(jobs):
        j[5] = [synth.queries(wl, 0, s, h, c).astype(np.float64) for c in range(steps)]
        j[6] = steps
    with ctx.Pool(workers) as pool:
        per_step = pool.map(_oracle_worker, [tuple(j) for j in jobs])
    mgr.shutdown()
    for f in os.listdir(tmp):
        os.remove(os.path.join(tmp, f))
    os.rmdir(tmp)
    # all heads of a step run side by side: a step takes the slowest head's time per
    # ceil(units / workers) rounds
    rounds = -(-units_per_call // workers)
    us = max(per_step) * rounds * 1e6
    desc = (f"fp64 numpy oracle, {workers} processes (one per KV head, spawn): {steps} decode steps of "
            f"sequence {s} of layer 0 (L0 {L0}) on {workers} heads at once; a decode call = "
            f"{units_per_call} units in {rounds} round(s)")
    return us, desc, steps * workers / units_per_call, workers


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (default: about 20k decode calls)")
    ap.add_argument("--warmup", type=int, default=0)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="qwen8b_128k")
    ap.add_argument("--r", type=int, default=None, help="override the variance groups r (r sweep)")
    ap.add_argument("--budget", type=int, default=None, help="override the budget in tokens (budget sweep)")
    ap.add_argument("--dense", action="store_true",
                    help="budget covering the whole context: every block selected (exact attention baseline)")
    ap.add_argument("--layers", type=int, default=None,
                    help="rotated layer caches (profiling runs: 1 keeps the device footprint small)")
    ap.add_argument("--kv-host", action="store_true",
                    help="K/V rows in page-locked host memory, read by the GPU over the chip-to-chip link")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    ws, rank, local = dist_env()
    overrides = {"r": args.r, "budget": args.budget, "dense": args.dense}
    layer_override = {"layers": args.layers} if args.layers else {}
    wl0, _, _ = bench_workload(args.workload, **overrides)
    calls_per_step = wl0.layers if wl0.layers > 1 else 1
    if args.steps <= 0:
        args.steps = max(20, 20000 // calls_per_step)
    if args.warmup <= 0:
        args.warmup = max(3, min(640, args.steps // 10))
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        return run_reference(args, ws, rank)

    # the CPU baseline first: its worker processes start before any GPU call
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        one_us, one_desc, _, _ = oracle_baseline(args.workload, budget_s=8.0, threads=1, **overrides)
        all_us, all_desc, _, all_cores = oracle_baseline(args.workload, budget_s=8.0, threads=8, **overrides)
        cpu = {"value": all_us, "unit": UNIT, "cores": all_cores, "kind": "oracle", "sample": all_desc,
               "one_core": {"value": one_us, "unit": UNIT, "cores": 1, "sample": one_desc},
               "host_cores": len(os.sched_getaffinity(0))}
        if calls_per_step > 1:
            for d in (cpu, cpu["one_core"]):
                d["value"] *= calls_per_step
                d["sample"] += f"; x{calls_per_step} layer calls per step"

    import torch
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

    work = Layers(args.workload, device, kv_memory="host" if args.kv_host else "device", **overrides,
                  **layer_override)
    cache = work.cache
    for _ in range(args.warmup):
        work.step()
    torch.cuda.synchronize(device)
    if cache.device_status() != 0:
        raise RuntimeError("device status error after warm-up: " + P.compkv_last_error())

    # ---- timed region: K steps, device time by CUDA events on the launch stream
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

    # ---- host issue rate: calls enqueued back to back right after a sync (no back-pressure)
    nh = min(200, args.steps * calls_per_step)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for _ in range(nh):
        work.call_once()
    host_us = (time.perf_counter() - t0) * 1e6 / nh
    torch.cuda.synchronize(device)

    # ---- device time per call, then per kernel (library events), separate passes
    kp = min(args.steps * calls_per_step, 4000)
    fam_ms = {}
    for level, fams in ((1, ("decode",)), (2, ("k_stream", "k_post"))):
        cache.profile(level)
        for fam in fams:
            cache.profile_read(fam)
        for _ in range(kp):
            work.call_once()
        torch.cuda.synchronize(device)
        fam_ms.update({fam: cache.profile_read(fam) for fam in fams})
        cache.profile(0)

    # ---- in-chain span of each kernel (first CTA start to last CTA end, %globaltimer), from
    # the device trace of a few calls; informational next to the event times above
    spans = trace_spans(cache, work, device)

    # ---- end to end through compkv_decode_host: pinned host inputs, output back, synchronised per call
    ke = min(args.steps * calls_per_step, 2000)
    R, S = work.R, work.wl.steps
    h_q = work.q.cpu().pin_memory()
    h_k = work.k_new.cpu().pin_memory()
    h_v = work.v_new.cpu().pin_memory()
    h_out = torch.empty(work.out.shape, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize(device)
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(ke):
        layer, c = work.i % R, (work.i // R) % S
        if c == 0 and work.i >= R:
            cache.seq_len[layer].copy_(work.lens_dev)
        cache.decode_host(layer, h_q[layer, c], h_k[layer, c], h_v[layer, c], h_out)
        work.i += 1
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, ws, device)
    if cache.device_status() != 0:
        raise RuntimeError("device status error in the e2e pass: " + P.compkv_last_error())

    if rank != 0:
        barrier(ws)
        return 0

    # ---- numbers
    by = step_bytes(work.wl)
    us_call = ms_max * 1e3 / (args.steps * calls_per_step)
    us_step_replica = ms_max * 1e3 / args.steps
    us_step = us_step_replica / ws           # whole-job time per step (replicas in parallel)
    peak, peak_kind = measured_peaks()
    step_gbs = by["total"] / (us_call * 1e-6) / 1e9
    kernels = {f: {"launches": n, "avg_us": (m * 1e3 / n if n else None)} for f, (m, n) in fam_ms.items()}
    kernels["decode"]["note"] = "one decode call: the two PDL-chained kernels"
    for f in ("k_stream", "k_post"):
        kernels[f]["span_in_chain_us"] = spans.get(f)
    for f in ("k_stream", "k_post"):
        kernels[f]["note"] = "timed alone (events between the kernels stop the second from launching early)"
    rooflines = {}
    for f, label, src in (("k_stream", "k_stream: append + summary stream (zbar, sigma2, logsumexp parts, "
                                       "compensation sums)", "stream_kernel.cu"),
                          ("k_post", "k_post: LSE, S_b, Top-K, exact attention, compensation, merge",
                           "post_kernel.cu")):
        us = kernels[f]["avg_us"]
        gbs = by[f] / (us * 1e-6) / 1e9
        rooflines[f] = {"bound": "hbm", "kernel": label, "achieved": gbs, "peak": peak, "peak_kind": peak_kind,
                        "unit": "GB/s", "frac": gbs / peak, "traffic": ncu_traffic(src, f, args.workload),
                        "algorithmic_bytes_per_launch": by[f], "avg_launch_us": us}
    dominant = max(rooflines, key=lambda f: rooflines[f]["avg_launch_us"])
    e2e_us = e2e_s * 1e6 / ke * calls_per_step / ws
    hbm_l2 = by["total"] * work.R / (calls_per_step if calls_per_step > 1 else 1)
    line = {
        "metric": METRIC, "value": us_step, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us_step_replica / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 (bf16 K/V, fp32 summaries)",
        "data": "synthetic (seeded generator: per-block centres + LogUniform within-block noise, "
                "2 outlier channels x5, 3 needles; random queries)",
        "config": {"workload": work.desc, "name": args.workload, "r": work.wl.r,
                   "budget_tokens": work.wl.budget_tokens, "dense": bool(args.dense),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": (f"inputs larger than L2: {work.R} independent layer caches rotated, "
                          f"{hbm_l2 / 1e6:.0f} MB touched between visits of one layer")
                   if hbm_l2 > 2 * L2_BYTES else "L2-resident (the workload is smaller than L2)",
                   "kv_memory": work.kv_memory,
                   "calls_per_step": calls_per_step, "us_per_call": us_call,
                   "hbm_gbs_step": step_gbs, "step_frac_of_peak": step_gbs / peak,
                   "bytes_per_call": by},
        "roofline": dict(rooflines[dominant], name=dominant),
        "rooflines": rooflines,
        "kernels": kernels,
        "host_issue_us_per_call": host_us,
        "e2e": {"value": e2e_us, "unit": UNIT, "api": "compkv_decode_host (pinned host buffers, synchronised)",
                "h2d_bytes_per_step": int((work.q[0, 0].numel() * 4 + 2 * work.k_new[0, 0].numel() * 2)
                                          * calls_per_step),
                "d2h_bytes_per_step": int(work.out.numel() * 4 * calls_per_step)},
        "gpu_launches": int(launches),
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    barrier(ws)
    return 0


def run_reference(args, ws, rank):
    """The oracle, as it stands, on the host cores (all of them): rank 0 only.
    Each timed step is one full decode call of the workload."""
    if rank != 0:
        return 0
    overrides = {"r": args.r, "budget": args.budget, "dense": args.dense}
    layer_override = {"layers": args.layers} if args.layers else {}
    wl, _, desc = bench_workload(args.workload, **overrides)
    t0 = time.perf_counter()
    us, sample, calls_done, cores = oracle_baseline(args.workload, budget_s=30.0, threads=8, **overrides)
    wall = time.perf_counter() - t0
    calls = wl.layers if wl.layers > 1 else 1
    us *= calls
    steps = max(1, int(round(calls_done / calls)))   # full decode steps the sample amounts to
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": ws,
        "steps": steps, "warmup": 0, "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same generator as the GPU arm)",
        "config": {"workload": desc, "name": args.workload, "requested_steps": args.steps,
                   "note": "each step is a full decode call of the workload, timed on a bounded sample",
                   "wall_s": wall},
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
