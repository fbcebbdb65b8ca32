"""Replica bookkeeping of bench.py across ranks, on CPU with two gloo processes: the job
time is the slowest rank's, the throughput counts every rank's tokens, and the
reference arm's other ranks leave without work."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.0 + rank, dist, "cpu")  # rank r took 1 + r ms
    out[rank] = (ms, bench.job_throughput(ms, world, 448))
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms, value = out[r]
        assert ms == 2.0
        assert value == pytest.approx(2 * 448 / 2e-3)


def test_single_process_is_its_own_max():
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_throughput(3.5, 1, 7) == pytest.approx(7 / 3.5e-3)


def test_reference_arm_other_ranks_exit_without_work():
    import argparse
    import bench
    a = argparse.Namespace(steps=1, warmup=0)
    assert bench.reference_arm(a, rank=1, world=2) == 0
