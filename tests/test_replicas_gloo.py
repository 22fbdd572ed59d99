"""The replica path of bench.py (one process per GPU, no collective on the data
path) run as two gloo ranks on the CPU: the job's time is the slowest rank's
(max over ranks), whole-job throughput counts every rank's tokens, and the
reference arm runs on rank 0 alone (other ranks return at once, printing
nothing)."""
import argparse
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        dist.barrier()
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        tput = bench.job_throughput(1000, world, ms)
        args = argparse.Namespace(warmup=1, steps=1, cpu_seconds=0.0)
        buf = io.StringIO()
        with redirect_stdout(buf):
            ret = bench.run_reference(args, rank, world) if rank != 0 else None
        results[rank] = (ms, tput, ret, buf.getvalue())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_throughput():
    import torch.multiprocessing as mp

    world, port = 2, _free_port()
    with mp.Manager() as man:
        results = man.dict()
        mp.spawn(_rank, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    for rank in range(world):
        ms, tput, ret, out = got[rank]
        assert ms == 5.0  # the slowest rank's time, on every rank
        assert tput == pytest.approx(1000 * world / 5e-3)
    # the reference arm does no work and prints nothing on rank 1
    assert got[1][2] is None and got[1][3] == ""


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.job_throughput(256, 1, 100.0) == pytest.approx(2560.0)
