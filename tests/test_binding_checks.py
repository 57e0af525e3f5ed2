"""The binding checks every array argument's dtype and extent on the host, before its pointer
reaches the kernels (CPU tensors: a call that passes every check stops at the device check)."""
import os

import numpy as np
import pytest
import torch

import speculative_decoding_verification_74_gb300 as sv

DEVICE_MSG = "libsv takes device tensors"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_verification_74_gb300 import build
    try:
        build.build()
    except RuntimeError as e:  # no nvcc on this machine
        if not os.path.exists(sv.LIB_PATH):
            pytest.skip(str(e))
    sv.lib()


def _raises(fn, match):
    with pytest.raises(ValueError, match=match):
        fn()


def _sample_args(B=4, K=3, V=64):
    return dict(target=torch.zeros(B * (K + 1), V, dtype=torch.bfloat16), draft=torch.zeros(B * K, V, dtype=torch.bfloat16),
                tokens=torch.zeros(B, K, dtype=torch.int32), temperature=torch.ones(B),
                out=(torch.empty(B, K + 1, dtype=torch.int32), torch.empty(B, dtype=torch.int32), torch.empty(B, K),
                     torch.empty(B, K), torch.empty(B, dtype=torch.uint8)))


def _sample(B=4, K=3, V=64, **over):
    a = _sample_args(B, K, V)
    a.update(over)
    sv.sv_verify_sample(a["target"], V, a["draft"], V, a["tokens"], a["temperature"], 1, 0, a.get("rid"),
                        sv.SV_BF16, B, K, V, *a["out"], None)


def test_sample_checks():
    _raises(lambda: _sample(), DEVICE_MSG)                                     # every check passes
    _raises(lambda: _sample(target=torch.zeros(15, 64, dtype=torch.bfloat16)), "target holds")
    _raises(lambda: _sample(target=torch.zeros(16, 64)), "target must be torch.bfloat16")
    _raises(lambda: _sample(draft=torch.zeros(11, 64, dtype=torch.bfloat16)), "draft holds")
    _raises(lambda: _sample(tokens=torch.zeros(4, 3, dtype=torch.int64)), "draft_tokens must be torch.int32")
    _raises(lambda: _sample(tokens=torch.zeros(4, 2, dtype=torch.int32)), "draft_tokens holds")
    _raises(lambda: _sample(temperature=torch.ones(3)), "temperature holds")
    _raises(lambda: _sample(temperature=torch.ones(4, dtype=torch.float64)), "temperature must be torch.float32")
    _raises(lambda: _sample(rid=torch.arange(4)), "request_ids must be torch.int32")
    out = list(_sample_args()["out"])
    out[4] = torch.empty(4, dtype=torch.int32)
    _raises(lambda: _sample(out=tuple(out)), "out_flags must be torch.uint8")
    out = list(_sample_args()["out"])
    out[2] = torch.empty(4, 2)
    _raises(lambda: _sample(out=tuple(out)), "out_p holds")


def test_views_are_checked_through_their_storage():
    """A row view is checked against what lies behind its data pointer: a view whose stride
    reaches past its own shape is fine while the storage covers the reads, not beyond."""
    big = torch.zeros(32, 64, dtype=torch.bfloat16)
    _raises(lambda: _sample(target=big[16:]), DEVICE_MSG)
    _raises(lambda: _sample(target=big[17:]), "target holds")


def test_ragged_checks():
    B, Km, V = 3, 4, 40
    tgt = torch.zeros(B * (Km + 1), V)
    offs = torch.arange(B + 1, dtype=torch.int32) * (Km + 1)
    toks = torch.zeros(B, Km, dtype=torch.int32)
    keep = torch.full((B,), 2, dtype=torch.int32)
    temp = torch.ones(B)
    out = (torch.empty(B, Km + 1, dtype=torch.int32), torch.empty(B, dtype=torch.int32), torch.empty(B, Km),
           torch.empty(B, Km), torch.empty(B, dtype=torch.uint8))

    def call(t_off=offs, tok=toks, tok_stride=Km, kl=keep, o=out, t_rows=B * (Km + 1)):
        sv.sv_verify_ragged(tgt, V, t_off, t_rows, None, V, None, 0, tok, tok_stride, kl, temp, 0, 0, None, sv.SV_F32,
                            B, Km, V, *o, None)
    _raises(call, DEVICE_MSG)
    _raises(lambda: call(t_off=offs[:B].clone()), "t_row_offsets holds")
    _raises(lambda: call(t_rows=B * (Km + 1) + 1), "target holds")       # more rows claimed than stored
    _raises(lambda: call(t_off=offs.long()), "t_row_offsets must be torch.int32")
    _raises(lambda: call(kl=keep[:2].clone()), "keep_len holds")
    _raises(lambda: call(tok_stride=Km + 1), "draft_tokens holds")       # the last request's tokens run past
    _raises(lambda: call(o=(torch.empty(B, Km, dtype=torch.int32),) + out[1:]), "out_tokens holds")


def test_schedule_checks():
    a = torch.rand(8, 5)
    so = (torch.empty(8, dtype=torch.int32), torch.empty(9, dtype=torch.int32), torch.empty(1, dtype=torch.int32),
          torch.empty(1, dtype=torch.int64))
    _raises(lambda: sv.sv_schedule_depth(a, 5, None, 8, 5, 1.0, 0.05, 0, None, 0, *so, None), DEVICE_MSG)
    _raises(lambda: sv.sv_schedule_depth(a.double(), 5, None, 8, 5, 1.0, 0.05, 0, None, 0, *so, None),
            "alpha must be torch.float32")
    _raises(lambda: sv.sv_schedule_depth(a[:7].clone(), 5, None, 8, 5, 1.0, 0.05, 0, None, 0, *so, None), "alpha holds")
    _raises(lambda: sv.sv_schedule_depth(a, 5, torch.full((7,), 5, dtype=torch.int32), 8, 5, 1.0, 0.05, 0, None, 0,
                                         *so, None), "draft_len holds")
    _raises(lambda: sv.sv_schedule_depth_table(a, 5, None, 8, 5, [10, 40], [1.0, 2.0], 0, None, 0,
                                               so[0], so[1], so[2], torch.empty(1, dtype=torch.int32), None),
            "out_utility_q48 must be torch.int64")
    _raises(lambda: sv.schedule_depth(torch.zeros(8, 0), 1.0, 0.02, 0), DEVICE_MSG)      # Dmax = 0 passes


def test_greedy_and_empty_batch():
    B, K, V = 2, 3, 50
    tgt = torch.zeros(B * (K + 1), V, dtype=torch.bfloat16)
    o = (torch.empty(B, K + 1, dtype=torch.int32), torch.empty(B, dtype=torch.int32))
    _raises(lambda: sv.sv_verify_greedy(tgt, V, None, 0, torch.zeros(B, K, dtype=torch.int32), sv.SV_BF16, B, K, V,
                                        *o, None), DEVICE_MSG)
    _raises(lambda: sv.sv_verify_greedy(tgt, V, tgt[: B * K - 1].clone(), V, None, sv.SV_BF16, B, K, V, *o, None),
            "draft holds")
    empty = torch.empty((0, 4), dtype=torch.int32)
    _raises(lambda: sv.sv_verify_greedy(None, 0, None, 0, None, sv.SV_BF16, 0, 3, 100, empty, empty, None),
            DEVICE_MSG)


def test_vocab_shard_checks():
    # a shard's arrays hold the columns of its chunks: a shard of the first two chunks of a bf16
    # row of V = 20000 holds 2 * chunk_len columns, and its rows are checked at that width
    B, K, V = 2, 3, 20000
    cl, nc = sv.sv_vocab_chunks(V, sv.SV_BF16)
    assert nc >= 3
    w = 2 * cl

    def phase(target_rows=B * (K + 1), width=w, stride=w, c_end=2):
        a = _sample_args(B, K, 1)
        sv.sv_verify_sample_phase(torch.zeros(target_rows, width, dtype=torch.bfloat16), stride,
                                  torch.zeros(B * K, width, dtype=torch.bfloat16), stride, a["tokens"],
                                  a["temperature"], 1, 0, None, sv.SV_BF16, B, K, V, 0, c_end, sv.SV_PHASE_STATS,
                                  *a["out"], None)

    _raises(lambda: phase(), DEVICE_MSG)                                        # every check passes
    _raises(lambda: phase(target_rows=B * (K + 1) - 1), "target holds")
    _raises(lambda: phase(width=w - 1), "target holds")                         # narrower than the shard
    _raises(lambda: phase(stride=V, c_end=3), "target holds")                   # a third chunk's columns

