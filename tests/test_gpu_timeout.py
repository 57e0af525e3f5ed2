"""A bounded wait that runs out: the kernel gives up, reports SV_ERR_TIMEOUT, and leaves the
context usable.

No GPU fault is involved.  The library's test hook makes the next verification call's stream
kernel leave one CTA without copies and bounds every wait of the launch by 50 ms: that CTA's
consumer warps wait for a ring stage nothing fills, give up, record SV_DEV_TIMEOUT and finish
the launch on what they hold; no copy is in flight when the CTA exits.  The call after it runs
normally on the same workspace and is exact."""
import time

import pytest
import torch

import speculative_decoding_verification_74_gb300 as sv
from synth import workloads as W
from svtest import dev_rows, i32, f32, oracle, compare

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_reports_timeout_and_the_next_call_is_exact():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    b = W.small("c2", 3)                                   # 5 sampled requests (T = 1)
    args = (dev_rows(b.target, "bf16"), dev_rows(b.draft, "bf16"), i32(b.tokens), f32(b.temperature), b.Kmax)
    kw = dict(seed=b.seed, round_=b.round, request_ids=i32(b.request_ids))
    ws = sv.workspace(sv.SV_OP_VERIFY, b.B, b.Kmax, b.V, sv.SV_BF16)
    sv.sv_test_stall_next_verify(50)
    t0 = time.time()
    sv.verify_sample(*args, ws=ws, **kw)
    st, bits = sv.sv_query_status(ws)                       # synchronizes
    assert st == sv.SV_ERR_TIMEOUT and bits & sv.SV_DEV_TIMEOUT, (st, bits)
    assert time.time() - t0 < 30.0                          # the waits were bounded

    for _ in range(2):
        tok, alen, p, q, fl = sv.verify_sample(*args, ws=ws, **kw)
        torch.cuda.synchronize()
        compare(oracle(b), tok.cpu().numpy(), alen.cpu().numpy(), p.cpu().numpy(), q.cpu().numpy(), b.keep_len,
                batch=b)
        assert sv.sv_query_status(ws) == (sv.SV_OK, 0)
