"""Vocabulary-parallel verification on one GPU: the vocabulary's chunks are split into shards,
and each shard's steps (sv_verify_sample_phase) run on its own column slice of the rows, as a
rank of a tensor-parallel LM head would.  The shards share one workspace here, which stands in
for the two all-gathers.  Results must match sv_verify_sample (decisions exactly, p and q to
float32 rounding) and the oracle."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_74_gb300 as sv
from speculative_decoding_verification_74_gb300.dist import chunk_ranges
from synth import workloads as W
from svtest import dev_rows, i32, f32, oracle, compare

pytestmark = pytest.mark.gpu


def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _whole(b, target, draft, dt):
    return sv.verify_sample(target, draft, i32(b.tokens), f32(b.temperature), b.Kmax, seed=b.seed, round_=b.round,
                            request_ids=i32(b.request_ids))


def _sharded(b, target, draft, dt, n_shards):
    B, K, V = b.B, b.Kmax, b.V
    cl, nc = sv.sv_vocab_chunks(V, dt)
    ranges = chunk_ranges(nc, n_shards)
    ws = sv.workspace(sv.SV_OP_VERIFY, B, K, V, dt)
    dev = target.device
    out = (torch.full((B, K + 1), -1, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev),
           torch.empty((B, K), dtype=torch.float32, device=dev), torch.empty((B, K), dtype=torch.float32, device=dev),
           torch.zeros(B, dtype=torch.uint8, device=dev))
    # each shard's own columns, as separate arrays with their own row stride
    local = []
    for c0, c1 in ranges:
        v0, v1 = c0 * cl, min(V, c1 * cl)
        local.append((target[:, v0:v1].contiguous(), draft[:, v0:v1].contiguous()))
    tok, temp, rid = i32(b.tokens), f32(b.temperature), i32(b.request_ids)

    def run(phase, s):
        t, d = local[s]
        c0, c1 = ranges[s]
        sv.sv_verify_sample_phase(t, t.stride(0), d, d.stride(0), tok, temp, b.seed, b.round, rid, dt, B, K, V, c0, c1,
                                  phase, *out, ws)

    for s in range(n_shards):
        run(sv.SV_PHASE_STATS, s)
    run(sv.SV_PHASE_ACCEPT, 0)
    for s in range(n_shards):
        run(sv.SV_PHASE_WEIGHTS, s)
    for s in range(n_shards):
        run(sv.SV_PHASE_PICK, s)
    torch.cuda.synchronize()
    assert sv.sv_query_status(ws) == (sv.SV_OK, 0)
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n_shards", [2, 3, 8])
def test_shards_equal_the_whole_call(dtype, n_shards):
    _gpu()
    # every request drafts K = 7 positions, so the packed rows are sv_verify_sample's fixed-K layout
    b = W.make_batch("vp", ["chat"] * 12 + ["code"] * 12, [7] * 24, [1.0, 0.6, 0.0, 1.3] * 6, 65537, dtype,
                     seed=4, rnd=1, sigma={"chat": (3.0, 1.0), "code": (0.0, 0.3)})
    dt = sv.SV_BF16 if dtype == "bf16" else sv.SV_F32
    assert np.array_equal(b.t_offsets, np.arange(b.B + 1) * (b.Kmax + 1))
    assert np.array_equal(b.d_offsets, np.arange(b.B + 1) * b.Kmax)
    target, draft = dev_rows(b.target, dtype), dev_rows(b.draft, dtype)
    whole = [o.cpu().numpy() for o in _whole(b, target, draft, dt)]
    parts = [o.cpu().numpy() for o in _sharded(b, target, draft, dt, n_shards)]
    orc = oracle(b)
    # the same chunk arithmetic, but a chunk record merges the chunks one CTA streams in a row, so
    # shard boundaries group the sums differently: p and q agree to float32 rounding, and every
    # decision outside the oracle's near-boundary band agrees exactly
    assert np.allclose(whole[2], parts[2], rtol=2e-6, atol=0, equal_nan=True)
    assert np.allclose(whole[3], parts[3], rtol=2e-6, atol=0, equal_nan=True)
    far = orc["near_pos"] < 0
    assert np.array_equal(whole[0][far], parts[0][far]) and np.array_equal(whole[1][far], parts[1][far])
    assert np.array_equal(whole[4][far], parts[4][far])
    compare(orc, parts[0], parts[1], parts[2], parts[3], b.keep_len, batch=b)


def test_shard_arguments_are_checked():
    _gpu()
    b = W.small("c2", 1)
    dt = sv.SV_BF16
    cl, nc = sv.sv_vocab_chunks(b.V, dt)
    target, draft = dev_rows(b.target, "bf16"), dev_rows(b.draft, "bf16")
    out = sv.verify_sample(target, draft, i32(b.tokens), f32(b.temperature), b.Kmax)
    ws = sv.workspace(sv.SV_OP_VERIFY, b.B, b.Kmax, b.V, dt)
    for c0, c1, phase in ((0, nc + 1, sv.SV_PHASE_STATS), (1, 1, sv.SV_PHASE_STATS), (0, nc, 7)):
        with pytest.raises(sv.SVError):
            sv.sv_verify_sample_phase(target, b.V, draft, b.V, i32(b.tokens), f32(b.temperature), 0, 0, None, dt, b.B,
                                      b.Kmax, b.V, c0, c1, phase, *out, ws)
