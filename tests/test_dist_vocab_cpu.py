"""The vocabulary partition's exchange on two gloo ranks (CPU): chunk ranges, and the all-gather
of a workspace region by chunk columns, which leaves every rank with every rank's columns."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_verification_74_gb300.dist import chunk_ranges, gather_chunk_columns


def test_chunk_ranges_cover_the_vocabulary():
    for nc in (1, 5, 19, 38, 1024):
        for world in range(1, min(nc, 9) + 1):
            r = chunk_ranges(nc, world)
            assert r[0][0] == 0 and r[-1][1] == nc and all(a < b for a, b in r)
            assert all(r[k][1] == r[k + 1][0] for k in range(world - 1))
            sizes = [b - a for a, b in r]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        chunk_ranges(3, 4)


def _port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, nc, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ranges = chunk_ranges(nc, world)
        full = torch.from_numpy(np.random.default_rng(7).integers(0, 256, (6, nc, 16), dtype=np.uint8))
        region = torch.zeros_like(full)
        a, b = ranges[rank]
        region[:, a:b] = full[:, a:b]          # this rank's columns only
        gather_chunk_columns(region, ranges, rank)
        out[rank] = bool(torch.equal(region, full))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,nc", [(2, 19), (3, 38), (2, 2)])
def test_two_ranks_gather_every_column(world, nc):
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _port(), nc, out), nprocs=world, join=True)
    assert all(out[r] for r in range(world))
