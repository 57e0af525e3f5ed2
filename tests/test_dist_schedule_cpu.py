"""D-cut over a batch split across ranks (CPU, gloo on 127.0.0.1, world size 2).

Each rank holds its own requests (different counts, ragged draft lengths).  global_schedule
all-gathers the confidences, schedules the concatenated batch and keeps this rank's depths.  With
the oracle's dcut_schedule as the scheduling call (the library's kernel needs a GPU), both ranks
must see the single-process schedule of the concatenated batch: the same K and U(K), and their
slices of its keep_len."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle.schedule import dcut_schedule
from speculative_decoding_verification_74_gb300.dist import global_schedule

SIZES = (5, 3)
DMAX = 6
COST_A, COST_B = 1.0, 0.05


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_inputs(rank):
    rng = np.random.default_rng(100 + rank)
    B = SIZES[rank]
    alpha = rng.beta(6, 2, (B, DMAX)).astype(np.float32)
    dl = rng.integers(0, DMAX + 1, B).astype(np.int32)
    return alpha, dl


def _oracle_schedule(a, ca, cb, budget, dl):
    o = dcut_schedule(a.numpy(), dl.numpy(), ca, cb, budget)
    keep = torch.from_numpy(np.asarray(o["keep_len"], np.int32))
    return keep, None, o["K"], o["U_q48"]


def _worker(rank, world, port, budget, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        alpha, dl = _rank_inputs(rank)
        keep, offs, K, U = global_schedule(torch.from_numpy(alpha), COST_A, COST_B, budget,
                                           draft_len=torch.from_numpy(dl), schedule=_oracle_schedule)
        out[rank] = (keep.numpy().tolist(), offs.numpy().tolist(), int(K), int(U))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("budget", [0, 20])
def test_two_ranks_see_the_single_process_schedule(budget):
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), budget, out), nprocs=world, join=True)
        res = dict(out)
    alpha = np.concatenate([_rank_inputs(r)[0] for r in range(world)])
    dl = np.concatenate([_rank_inputs(r)[1] for r in range(world)])
    o = dcut_schedule(alpha, dl, COST_A, COST_B, budget)
    start = 0
    for r in range(world):
        keep, offs, K, U = res[r]
        assert K == o["K"] and U == o["U_q48"]
        assert keep == list(o["keep_len"][start: start + SIZES[r]])
        assert offs == [0] + np.cumsum(np.asarray(keep) + 1).tolist()
        start += SIZES[r]
    # the shared budget moves depth between ranks: the kept depths differ from scheduling each
    # rank's requests alone with half the budget
    if budget:
        split = [dcut_schedule(_rank_inputs(r)[0], _rank_inputs(r)[1], COST_A, COST_B, budget // 2)["keep_len"]
                 for r in range(world)]
        assert np.concatenate(split).tolist() != o["keep_len"].tolist()
