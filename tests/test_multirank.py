"""The multi-rank host logic of bench.py on CPU: two `gloo` ranks (spawned
processes, rendezvous on 127.0.0.1).  The path runs replicas with no
data-path collective; what ranks share is the barrier around the timed
region, the max over ranks of the measured time, and the whole-job rate
(every replica's units over the slowest rank's time).  The reference arm
runs on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        ms = bench.max_over_ranks(1.5 * (rank + 1), world)      # rank 1 is the slow one
        rate = bench.job_rate(2048, world, ms)
        buf = io.StringIO()

        class Args:
            steps, warmup, gpus = 1, 0, world
        if rank != 0:
            with redirect_stdout(buf):
                bench.reference_arm(Args, rank)                  # non-zero ranks do no work
        bench.barrier(world)
        q.put((rank, ms, rate, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time_and_the_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    for rank, ms, rate, printed in got:
        assert ms == pytest.approx(3.0)                          # the max of 1.5 and 3.0
        assert rate == pytest.approx(2 * 2048 / 3.0e-3)          # both replicas' tokens
    assert got[1][3] == ""                                       # rank 1 printed nothing


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.job_rate(100, 1, 10.0) == pytest.approx(1e4)
