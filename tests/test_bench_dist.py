"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each timing its
own replica of the workload, agree on the slowest rank's time and report the
whole-job throughput from it."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.reduce_max(times[rank], dist)
        value = bench.job_throughput(1e9, 10, dist.get_world_size(), ms)
        results[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_job_throughput():
    world = 2
    times = [100.0, 125.0]
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_worker, args=(world, port, times, results), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(results)
    for rank in range(world):
        ms, value = res[rank]
        assert ms == 125.0
        # 2 ranks x 10 steps x 1 GB in the slowest rank's 125 ms
        assert abs(value - 160.0) < 1e-9


def test_single_process_identity():
    assert bench.reduce_max(3.5, None) == 3.5
    assert abs(bench.job_throughput(2e9, 5, 1, 1000.0) - 10.0) < 1e-12
