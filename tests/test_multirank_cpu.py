"""The multi-GPU bench path's host logic on two CPU ranks (gloo on 127.0.0.1): whole-job totals
take the slowest rank's time and the sum of the ranks' positions, and every rank gets its own
input seed."""
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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, pos = bench.job_totals(1.0 + rank, 10.0 * (rank + 1), dist, "cpu")
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.rank_seed(1000, rank))
        out[rank] = (ms, pos, tuple(seeds))
    finally:
        dist.destroy_process_group()


def test_two_rank_job_totals_and_seeds():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, pos, seeds = res[r]
        assert ms == pytest.approx(2.0)      # the slowest rank's time
        assert pos == pytest.approx(30.0)    # positions of both ranks
        assert len(set(seeds)) == world      # independent inputs per rank


def test_single_process_totals_are_local():
    assert bench.job_totals(3.5, 42, None) == (3.5, 42)
