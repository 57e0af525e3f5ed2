"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times
(bench.GpuWorkload drives the C ABI exactly as the timed loop does).  The oracle checks every
request where it is quick (C2, C4, C5) and a seeded sample of requests for C3 (64 requests x 33
fp32 rows of 151936)."""
import numpy as np
import pytest
import torch

import bench
from oracle.schedule import dcut_schedule
from oracle.verify import verify_batch
from synth import workloads as W
from svtest import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _run(gw, j):
    gw.step(j)
    torch.cuda.synchronize()
    return [None if o is None else o.cpu().numpy() for o in gw.out]


def _oracle(b, keep, requests=None):
    if requests is None:
        return verify_batch(b.target, b.t_offsets, b.draft, b.d_offsets, b.tokens, keep, b.temperature, b.seed,
                            b.round, b.request_ids, b.dtype, b.Kmax), None
    # a subset of requests: the oracle takes the packed layout request by request
    sub = np.asarray(requests)
    res = verify_batch(b.target, b.t_offsets[sub], b.draft, None if b.d_offsets is None else b.d_offsets[sub],
                       None if b.tokens is None else b.tokens[sub], keep[sub], b.temperature[sub], b.seed,
                       b.round, b.request_ids[sub], b.dtype, b.Kmax)
    return res, sub


def _check(out, orc, keep, sub=None, batch=None):
    tok, alen, p, q = out[0], out[1], out[2], out[3]
    if sub is not None:
        tok, alen, p, q, keep = tok[sub], alen[sub], p[sub], q[sub], keep[sub]
    return compare(orc, tok, alen, p, q, keep, batch=batch)


def test_fullsize_c2_mtp_every_request():
    sets = bench.make_sets("c2", 2, 500)
    gw = bench.GpuWorkload("c2", sets, torch.device("cuda", 0))
    for j in range(2):
        b = sets[j]["batch"]
        out = _run(gw, j)
        orc, _ = _oracle(b, b.keep_len)
        _check(out, orc, b.keep_len, batch=b)


def test_fullsize_c3_dfly_sampled_requests():
    sets = bench.make_sets("c3", 1, 600)
    gw = bench.GpuWorkload("c3", sets, torch.device("cuda", 0))
    b = sets[0]["batch"]
    out = _run(gw, 0)
    req = np.sort(np.random.default_rng(3).choice(b.B, 16, replace=False))
    orc, sub = _oracle(b, b.keep_len, req)
    _check(out, orc, b.keep_len, sub)


def test_fullsize_c4_schedule_then_ragged_verify():
    sets = bench.make_sets("c4", 1, 700)
    gw = bench.GpuWorkload("c4", sets, torch.device("cuda", 0))
    s, b = sets[0]["sched"], sets[0]["batch"]
    out = _run(gw, 0)
    keep_gpu = gw.sched_out[0].cpu().numpy()
    o = dcut_schedule(s.alpha, None, s.cost_a, s.cost_b, s.budget)
    assert np.array_equal(keep_gpu, o["keep_len"])
    assert int(gw.sched_out[2].item()) == o["K"] and int(gw.sched_out[3].item()) == o["U_q48"]
    orc, _ = _oracle(b, o["keep_len"])
    _check(out, orc, o["keep_len"], batch=b)


def test_fullsize_c5_mixed_rounds():
    sets = bench.make_sets("c5", 2, 800)
    gw = bench.GpuWorkload("c5", sets, torch.device("cuda", 0))
    for j in range(2):
        b = sets[j]["batch"]
        out = _run(gw, j)
        orc, _ = _oracle(b, b.keep_len)
        _check(out, orc, b.keep_len, batch=b)


def test_fullsize_c1_greedy():
    sets = bench.make_sets("c1", 3, 900)
    gw = bench.GpuWorkload("c1", sets, torch.device("cuda", 0))
    for j in range(3):
        b = sets[j]["batch"]
        out = _run(gw, j)
        orc, _ = _oracle(b, b.keep_len)
        tok, alen = out[0], out[1]
        compare(orc, tok, alen)
