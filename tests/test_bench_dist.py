"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks (no GPU).

Under torchrun every rank scans its own full workload (rows are independent,
so there is no collective on the data path); the timed region is the slowest
rank's, and the reported value is all ranks' units over that time. These
tests run the same helpers bench.py uses, in two spawned processes.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    r, w = bench.dist_init("gloo")
    bench.barrier()
    seconds = 1.0 + r                     # rank 1 is the slow one
    slowest = bench.reduce_max(seconds)
    value = bench.aggregate(100.0, w, slowest)
    q.put((r, w, slowest, value))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_ranks_take_slowest_time_and_sum_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, world, slowest, value in got:
        assert world == 2
        assert slowest == pytest.approx(2.0)           # max over ranks
        assert value == pytest.approx(100.0 * 2 / 2.0)  # all ranks' units / slowest time


def test_single_process_defaults():
    import bench
    assert bench.dist_env()[1] >= 1
    assert bench.reduce_max(3.5) == 3.5
    assert bench.aggregate(10.0, 1, 2.0) == 5.0
