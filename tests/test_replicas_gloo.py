"""The multi-rank (replicas) host logic of bench.py on CPU: two gloo ranks, no GPU.

The indexer path shards by independent sequences with no data-path collective; the
only cross-rank steps are the barriers around the timed region and the maximum of the
timings over the ranks, from which the whole-job rate is computed.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r times (r + 1, 10 - r, 3): the job sees each timing's slowest rank
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank, 3.0], world, torch.device("cpu"))
        dist.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    with mp.get_context("spawn").Manager() as mgr:   # no fork of this (threaded) process
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1] == [2.0, 10.0, 3.0]


def test_single_rank_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks([1.5, 2.5], 1, torch.device("cpu")) == [1.5, 2.5]


def test_job_rate_is_weak_scaling_over_the_slowest_rank():
    # 1000 units per rank, 2 ms per step on the slowest of 4 ranks -> 2e6 units/s
    assert bench.job_rate(1000, 4, 2.0) == pytest.approx(2e6)
    assert bench.job_rate(1000, 1, 2.0) == pytest.approx(5e5)
