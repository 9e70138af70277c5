"""Host logic of bench.py's N-GPU replicas path, run as two gloo ranks on the
CPU: the job time is the maximum of the ranks' own times, the whole-job rate
counts every rank's units, and only rank 0 prints a line."""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        own = [120.0, 150.0][rank]
        ms = bench.job_time_ms(own, world, "cpu")
        rate = bench.job_rate(1000.0, world, ms)
        out.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_two_rank_job_time_is_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ms, rate in got:
        assert ms == 150.0                      # max over ranks, seen by every rank
        assert rate == pytest.approx(2 * 1000.0 / 0.150)   # both ranks' units / job time


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.job_time_ms(12.5, 1, "cpu") == 12.5
    assert bench.job_rate(10.0, 1, 1000.0) == pytest.approx(10.0)
