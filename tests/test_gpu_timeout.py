"""A bounded wait that runs out: the kernel gives up, reports SV_ERR_TIMEOUT, and leaves the
context usable.

No GPU fault is involved.  The verification kernel runs a request's accept chain once every
stream unit of the request has counted itself in a per-request completion counter; the CTA
that takes the request's accept-chain unit waits (about 2 s at most) for the count to reach the
request's task total, and the draw units wait for the flag the accept chain sets.  Here the host
breaks the workspace contract (zero-filled before use): request 0's counter starts at 2^30, far
above its task total, so the count never matches, the accept chain never runs, and nothing sets
the flag.  Every other request completes; the waits for request 0 give up, the grid's other waits
see the timeout bit and give up too, and every CTA drains its copies and exits.  After zeroing the
workspace again, the next call is exact."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_74_gb300 as sv
from synth import workloads as W
from svtest import dev_rows, i32, f32, oracle, compare

pytestmark = pytest.mark.gpu

COUNTERS_OFFSET = 256  # the completion counters start right after the 256-byte status region


def test_a_wait_that_runs_out_reports_timeout_and_the_next_call_is_exact():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    b = W.small("c2", 3)                                   # 5 sampled requests (T = 1)
    args = (dev_rows(b.target, "bf16"), dev_rows(b.draft, "bf16"), i32(b.tokens), f32(b.temperature), b.Kmax)
    kw = dict(seed=b.seed, round_=b.round, request_ids=i32(b.request_ids))
    ws = sv.workspace(sv.SV_OP_VERIFY, b.B, b.Kmax, b.V, sv.SV_BF16)
    ws.view(torch.int32)[COUNTERS_OFFSET // 4] = 1 << 30    # request 0: a count its units never reach
    sv.verify_sample(*args, ws=ws, **kw)
    st, bits = sv.sv_query_status(ws)                       # synchronizes (about 2 s)
    assert st == sv.SV_ERR_TIMEOUT and bits & sv.SV_DEV_TIMEOUT, (st, bits)

    ws.zero_()                                              # counters may be mid-count after a timeout
    for _ in range(2):
        tok, alen, p, q, fl = sv.verify_sample(*args, ws=ws, **kw)
        torch.cuda.synchronize()
        compare(oracle(b), tok.cpu().numpy(), alen.cpu().numpy(), p.cpu().numpy(), q.cpu().numpy(), b.keep_len,
                batch=b)
        assert sv.sv_query_status(ws) == (sv.SV_OK, 0)
