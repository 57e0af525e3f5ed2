"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times
(bench.GpuWorkload drives the C ABI exactly as the timed loop does).  The oracle checks every
request of every workload (C3's 64 requests x 33 fp32 rows of 151936 in host threads), and C5
over 100 rounds."""
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


def test_fullsize_c3_dfly_every_request():
    """All 64 C3 requests (33 fp32 rows of 151936 each); the oracle takes them in host threads,
    16 requests each."""
    from concurrent.futures import ThreadPoolExecutor
    sets = bench.make_sets("c3", 1, 600)
    gw = bench.GpuWorkload("c3", sets, torch.device("cuda", 0))
    b = sets[0]["batch"]
    out = _run(gw, 0)
    groups = [np.arange(g, min(b.B, g + 16)) for g in range(0, b.B, 16)]
    with ThreadPoolExecutor(max_workers=len(groups)) as ex:
        parts = [orc for orc, _ in ex.map(lambda req: _oracle(b, b.keep_len, req), groups)]
    orc = {k: np.concatenate([part[k] for part in parts]) for k in parts[0]}  # the groups in request order
    _check(out, orc, b.keep_len, batch=b)


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


def test_fullsize_c5_hundred_rounds():
    """C5 as stated: 100 rounds from one seed (the request roles fixed by the seed, rows and
    temperatures redrawn each round), every round at full size through one workspace, every
    request of every round against the oracle.  Rounds are drawn and run through the oracle in
    host threads (numpy releases the GIL in its generators and large array operations) a few
    rounds ahead of the GPU; no thread touches CUDA."""
    import os
    from collections import deque
    from concurrent.futures import ThreadPoolExecutor
    import speculative_decoding_verification_74_gb300 as sv
    from svtest import run_ragged, oracle

    rounds, seed = 100, 800

    def make(r):
        b = W.c5_mixed(seed=seed, rnd=r)
        return b, oracle(b)

    workers = max(1, min(16, os.cpu_count() or 1))
    ws = sv.workspace(sv.SV_OP_VERIFY, 64, 16, 151936, sv.SV_BF16)
    near = 0
    with ThreadPoolExecutor(max_workers=workers) as ex:
        pending = deque(ex.submit(make, r) for r in range(min(rounds, workers + 2)))
        nxt = len(pending)
        for r in range(rounds):
            b, orc = pending.popleft().result()
            if nxt < rounds:
                pending.append(ex.submit(make, nxt))
                nxt += 1
            tok, alen, p, q, fl = run_ragged(b, ws=ws)
            near += compare(orc, tok, alen, p, q, b.keep_len, batch=b)
            assert sv.sv_query_status(ws) == (sv.SV_OK, 0)
            del b, orc
    print(f"c5: {rounds} rounds, {near} requests excused in all")
