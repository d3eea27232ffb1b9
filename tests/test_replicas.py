"""The N-GPU bookkeeping of bench.py, as two gloo ranks on the CPU.

Replicas: every rank runs the whole workload; the timed figure is the slowest rank's, and
the whole-job value counts every rank's patches.  Rank 0 alone runs and prints the
reference arm.  No GPU is involved.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [1.5, 2.25][rank]                 # rank 1 is the slow replica
        ms = bench.world_max(local_ms, world, "cpu")
        results[rank] = (ms, bench.replica_value(589824, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_value():
    world = 2
    results = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), results), nprocs=world, join=True)
    assert results[0] == results[1]
    ms, value = results[0]
    assert ms == 2.25
    assert value == pytest.approx(2 * 589824 / 2.25e-3)


def test_single_rank_needs_no_process_group():
    assert bench.world_max(3.5, 1, "cpu") == 3.5
    assert bench.replica_value(100, 1, 10.0) == pytest.approx(1e4)


def test_reference_arm_prints_on_rank_zero_only():
    class A:
        steps, warmup = 1, 0
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(A(), 1, 2) == 0
    assert buf.getvalue() == ""
