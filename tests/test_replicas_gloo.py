"""The multi-GPU path of the benchmark runs independent replicas (the KDA core
has no exchange step): each rank times its own steps and the job is timed by
the slowest rank.  This checks that host logic with two gloo ranks on the CPU.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    # rank r measured (10 + r) ms for the timed steps and (20 - r) ms end to end
    got = bench.max_over_ranks([10.0 + rank, 20.0 - rank], dist, "cpu")
    results[rank] = (got, bench.whole_job_rate(world, 512, 100, got[0]))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank():
    world = 2
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world, start_method="spawn")
        res = dict(results)
    for rank in range(world):
        got, rate = res[rank]
        assert got == [11.0, 20.0]
        assert rate == pytest.approx(2 * 512 * 100 / 0.011)


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.whole_job_rate(1, 512, 10, 1000.0) == pytest.approx(5120.0)
