"""Replica path of bench.py on CPU: two gloo ranks agree on the max-over-ranks time and the
whole-job sums that the JSON line reports (the path has no data-path collective)."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), STA_BENCH_BACKEND="gloo")
    import bench

    d = bench.Dist()
    try:
        d.barrier()
        t = d.max(1.0 + rank)          # slowest rank's time
        units = d.sum(10.0 * (rank + 1))  # units processed by all ranks
        q.put((rank, d.world, t, units))
    finally:
        d.close()


def test_two_gloo_ranks_reduce_like_the_bench():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, w, t, units in got:
        assert w == 2 and t == 2.0 and units == 30.0
