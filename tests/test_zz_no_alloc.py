"""sv_verify_sample_noalloc: sampled verification for callers that cannot allocate device memory
(e.g. code running while its stream is captured into a CUDA graph, plugins whose device memory
belongs to a host framework's allocator, serving loops that forbid allocation on the hot path).

The entry point runs the same kernels on a scratch array built into the library, so its outputs
must equal sv_verify_sample's (with a caller workspace) on the same inputs, call after call.
This file is collected last so that a failure here leaves every other test already run."""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_verification_74_gb300 as sv
from synth import workloads as W
from svtest import dev_rows, i32, f32, P_TOL

pytestmark = pytest.mark.gpu


def _outputs(B, K):
    return (torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, K), -7.0, dtype=torch.float32, device="cuda"),
            torch.full((B, K), -7.0, dtype=torch.float32, device="cuda"),
            torch.zeros(B, dtype=torch.uint8, device="cuda"))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    for call, (name, seed) in enumerate([("c2", 11), ("c3", 12)]):
        b = W.small(name, seed)
        dt = sv.SV_BF16 if b.dtype == "bf16" else sv.SV_F32
        tgt, dr = dev_rows(b.target, b.dtype), dev_rows(b.draft, b.dtype)
        tok, temp, rid = i32(b.tokens), f32(b.temperature), i32(b.request_ids)
        ref = sv.verify_sample(tgt, dr, tok, temp, b.Kmax, seed=b.seed, round_=b.round, request_ids=rid)
        out = _outputs(b.B, b.Kmax)
        sv.sv_verify_sample_noalloc(tgt, b.V, dr, b.V, tok, temp, b.seed, b.round, rid, dt, b.B, b.Kmax, b.V, *out)
        torch.cuda.synchronize()
        ref = [x.cpu().numpy() for x in ref]
        got = [x.cpu().numpy() for x in out]
        assert np.array_equal(got[0], ref[0]), f"call {call}: tokens differ"
        assert np.array_equal(got[1], ref[1]), f"call {call}: accepted lengths differ"
        assert np.allclose(got[2], ref[2], atol=P_TOL, rtol=0, equal_nan=True)
        assert np.allclose(got[3], ref[3], atol=P_TOL, rtol=0, equal_nan=True)
        assert np.array_equal(got[4], ref[4])


def test_noalloc_rejects_sizes_beyond_its_scratch():
    L = sv.lib()
    fake = 1 << 20
    st = L.sv_verify_sample_noalloc(fake, 151936, fake, 151936, fake, fake, 0, 0, None, sv.SV_F32, 4096, 64,
                                    151936, fake, fake, None, None, None, None)
    assert st == sv.SV_ERR_WORKSPACE
    assert b"built-in scratch" in L.sv_last_error_string()
