"""The N > 1 host path of bench.py on CPU: two gloo ranks (processes) with different timed-region durations.
The job's duration is the slowest rank's, and the throughput counts every rank's units (replicas, weak scaling)."""

from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    try:
        ms, value = bench.whole_job([12.0, 30.0][rank], 100 * 4, world, dist, "cpu")
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_whole_job_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, value in got:
        assert ms == 30.0, rank  # the slowest rank's duration
        assert value == pytest.approx(2 * 400 / 0.030)  # both ranks' 400 units over 30 ms


def test_whole_job_single_process():
    import bench

    ms, value = bench.whole_job(20.0, 50, 1)
    assert ms == 20.0 and value == pytest.approx(50 / 0.020)
