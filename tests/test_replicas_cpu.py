"""The N > 1 benchmark path on CPU: two gloo ranks (world size 2).

The decode step does not shard across GPUs here (replicas only: every rank
runs its own independent caches), so the only cross-rank steps are the host
ones: the barrier around the timed region, the maximum of the per-rank times,
and the reference arm that runs on rank 0 alone.
"""
import argparse
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    env = bench.dist_env()
    bench.barrier(ws)
    t_max = bench.max_over_ranks(10.0 + 5.0 * rank, ws, torch.device("cpu"))
    rc = None
    if rank != 0:
        # the reference arm: every rank but 0 returns at once, with no work
        rc = bench.run_reference(argparse.Namespace(steps=4, warmup=3), ws, rank)
    bench.barrier(ws)
    out.put((rank, env, t_max, rc))
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(2):
            rank, env, t_max, rc = out.get(timeout=120)
            got[rank] = (env, t_max, rc)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    assert got[0][0] == (2, 0, 0) and got[1][0] == (2, 1, 1)
    assert got[0][1] == got[1][1] == pytest.approx(15.0)
    assert got[1][2] == 0
