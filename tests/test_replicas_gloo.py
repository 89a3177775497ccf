"""Host logic of the multi-GPU bench (independent replicas): two gloo ranks
on CPU agree on the slowest rank's time and on the whole-job throughput."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from exact_io_aware_39_gb300.replicas import job_throughput, max_over_ranks


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = max_over_ranks(times[rank])
        out[rank] = (m, job_throughput(1e12, 10, world, m))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, times = 2, [120.0, 150.0]
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), times, out), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        m, v = out[r]
        assert m == 150.0
        assert v == pytest.approx(2 * 1e12 * 10 / 0.150 / 1e12)


def test_single_process_without_process_group():
    assert max_over_ranks(3.5) == 3.5
    assert job_throughput(2e12, 4, 1, 1000.0) == pytest.approx(8.0)
    with pytest.raises(ValueError):
        job_throughput(1.0, 1, 1, 0.0)
