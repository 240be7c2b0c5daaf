"""CPU test of the multi-GPU bench path's host logic with two gloo ranks:
replicas draw distinct inputs, timing is the max over ranks, and the
whole-job value counts every rank's frames.  No data-path collective exists
to test: the ranks serve independent streams."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import argparse
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        args = argparse.Namespace(workload="c5_stress", streams=2)
        w = bench.workload(args, rank)
        ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        mx = bench.max_over_ranks(ms, world)
        val = bench.aggregate(bench.frames_per_step(w) * 100, mx, world)
        q.put((rank, w["seed"], mx, val))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    seeds = {r[1] for r in res}
    assert len(seeds) == world  # each replica serves its own streams
    assert all(r[2] == 15.0 for r in res)  # the slowest rank's time
    # 2 streams x 3 frames x 100 steps per rank, 2 ranks, 15 ms
    assert all(abs(r[3] - 2 * 3 * 100 * 2 / 0.015) < 1e-6 for r in res)
