"""The bench's rank logic with two gloo processes on the CPU: each rank runs its
own streams (no data-path collective); the barrier and the max of the step time
are the only cross-rank steps, and the throughput counts every rank's rows."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.dist_barrier(w)
    ms_local = 2.0 + r          # rank 1 is the slower one
    value, ms_max = bench.aggregate(100, ms_local, w)
    q.put((r, value, ms_max))
    dist.destroy_process_group()


def test_two_ranks_weak_scaling():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, value, ms_max in out:
        assert ms_max == 3.0                          # the slowest rank's step
        assert value == pytest.approx(200 / 3e-3)     # both ranks' rows over that time


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(16, 0.5, 1) == (16 / 0.5e-3, 0.5)
