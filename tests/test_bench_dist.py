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


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched the way the multi-GPU run is: two
    ranks over torch.distributed.run; rank 0 times the oracle and prints the
    one JSON line, the other rank exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "vim_ti_224", "--cpu-seconds", "0.3"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
