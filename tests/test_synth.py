"""The seeded input generators follow their stated recipes (CPU only): bf16 rounding, the chat
and Zipf row recipes, the drafter's token choice, the D-cut confidences, the mixed round's roles
and temperatures, packing and determinism."""
import math

import numpy as np
import torch

from synth import workloads as W


def _rows32(b, which):
    x = b.target if which == "t" else b.draft
    return W.bf16_bits_to_f32(x) if b.dtype == "bf16" else x


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 7,
                        rng.standard_normal(2000).astype(np.float32) * 1e-30,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.0e38, 0.0, -0.0], np.float32)])
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(W.f32_to_bf16_bits(W.bf16_bits_to_f32(ours)), ours)     # widening is exact


def test_chat_recipe_and_sampled_tokens():
    b = W.c2_mtp(seed=3, B=6, K=3, V=20011)
    t, d = _rows32(b, "t"), _rows32(b, "d")
    assert t.shape == (6 * 4, 20011) and d.shape == (6 * 3, 20011)
    assert abs(t.std() - 3.0) < 0.03
    noise = np.concatenate([d[b.d_offsets[i]: b.d_offsets[i + 1]] - t[b.t_offsets[i]: b.t_offsets[i] + 3]
                            for i in range(b.B)])
    assert abs(noise.std() - 1.0) < 0.02
    assert b.tokens.shape == (6, 3) and np.all((b.tokens >= 0) & (b.tokens < b.V))
    assert np.all(b.temperature == 1.0) and np.array_equal(b.request_ids, np.arange(6))
    # x ~ softmax(d / T): sampled tokens sit high in their draft row, and are not all the argmax
    ranks = [int(np.sum(d[b.d_offsets[i] + k] > d[b.d_offsets[i] + k, b.tokens[i, k]]))
             for i in range(b.B) for k in range(3)]
    assert np.median(ranks) < 50 and any(r > 0 for r in ranks)


def test_zipf_recipe():
    b = W.c3_dfly(seed=1, B=3, K=2, V=5003)
    assert b.dtype == "f32" and np.all(b.temperature == np.float32(0.6))
    t, d = _rows32(b, "t"), _rows32(b, "d")
    A = 6.0 / math.log(2.0)
    for row in t:
        top = np.sort(row)[::-1]
        assert 5.3 < top[0] - top[1] < 6.7                      # top-1 / top-2 gap ~ 6 nats
        assert abs(top[0]) < 0.5 and abs(top[-1] + A * math.log(5003)) < 0.5
        # ranks are a permutation: the sorted row follows -A ln(rank) up to the N(0, 0.1) noise
        ideal = -A * np.log(np.arange(1, 5004))
        assert np.median(np.abs(top - ideal)) < 0.1
    noise = np.concatenate([d[b.d_offsets[i]: b.d_offsets[i + 1]] - t[b.t_offsets[i]: b.t_offsets[i] + 2]
                            for i in range(b.B)])
    assert abs(noise.std() - 0.3) < 0.01


def test_greedy_batch_takes_the_draft_argmax():
    b = W.c1_greedy(seed=2, B=3, K=3, V=4001)
    assert b.tokens is None and np.all(b.temperature == 0.0) and np.all(b.keep_len == 3)
    t, d = _rows32(b, "t"), _rows32(b, "d")
    assert abs(t.std() - 2.0) < 0.05
    b2 = W.make_batch("g", ["chat"] * 3, [3] * 3, [0.0] * 3, 4001, "bf16", 2, 0, {"chat": (2.0, 0.5)})
    d2 = _rows32(b2, "d")
    for i in range(3):
        for k in range(3):
            row = d2[b2.d_offsets[i] + k]
            assert b2.tokens[i, k] == int(np.argmax(row))           # T = 0: first argmax, not a sample


def test_dcut_confidences():
    s = W.c4_alpha(seed=4)
    assert s.alpha.shape == (64, 16) and s.alpha.dtype == np.float32
    code = np.array([k == "code" for k in s.kinds])
    assert code.sum() == 32
    assert np.all(s.alpha > 0) and np.all(s.alpha < 1)
    assert abs(s.alpha[code].mean() - 0.8) < 0.03 and abs(s.alpha[~code].mean() - 0.5) < 0.03
    assert (s.cost_a, s.cost_b, s.budget) == (1.0, 0.05, 384)


def test_mixed_round_roles_and_temperatures():
    r0 = W.c5_mixed(seed=5, rnd=0, B=12, V=3001)
    r1 = W.c5_mixed(seed=5, rnd=1, B=12, V=3001)
    kinds0 = [int(k) for k in r0.keep_len]
    assert kinds0 == [int(k) for k in r1.keep_len]                 # roles (and so K) fixed by the seed
    assert sorted(set(kinds0)) == [3, 16] and kinds0.count(16) == 6
    assert set(r0.temperature.tolist()) <= {float(np.float32(x)) for x in (0.0, 0.6, 1.0)}
    assert not np.array_equal(r0.target, r1.target)                # rows redrawn each round
    for b in (r0, r1):
        assert b.t_offsets[-1] == sum(k + 1 for k in b.keep_len) == b.target.shape[0]
        assert b.d_offsets[-1] == sum(b.keep_len) == b.draft.shape[0]


def test_determinism():
    a, b = W.c2_mtp(seed=9, B=2, K=3, V=1001), W.c2_mtp(seed=9, B=2, K=3, V=1001)
    c = W.c2_mtp(seed=10, B=2, K=3, V=1001)
    for f in ("target", "draft", "tokens", "t_offsets", "d_offsets"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    assert not np.array_equal(a.target, c.target)
    assert np.array_equal(W.c4_alpha(3).alpha, W.c4_alpha(3).alpha)
