"""Host logic of the startup cost-table profiler (CPU only, fake step and clock)."""
import math

import numpy as np
import pytest

from speculative_decoding_verification_74_gb300.cost_table import (profile_cost_table, tokens_for,
                                                                   MAX_COST_KNOTS)


def test_tokens_for_follows_eq_k_rho():
    # eq. K_rho with N = b (D + 1): the printed budgets (B=64, D=16 -> 272 at 0.25, 1088 at 1)
    assert tokens_for(64, 16, 0.25) == 272
    assert tokens_for(64, 16, 1.0) == 1088
    assert tokens_for(6, 7, 0.5) == 24
    assert tokens_for(4, 0, 0.25) == 4          # floor of one slot per request
    for b in (1, 5, 33):
        for D in (0, 3, 16):
            for r in (0.1, 0.25, 0.3, 0.75):
                assert tokens_for(b, D, r) == max(b, math.ceil(np.float64(np.float32(r)) * b * (D + 1)))


def _fake(latency):
    """A step that records its calls and a timer that returns latency(b, K) of the call it times."""
    calls = []

    def step(b, K):
        calls.append((b, K))

    def timer(fn):
        fn()
        b, K = calls[-1]
        return latency(b, K, len(calls))
    return step, timer, calls


def test_grid_warmup_reps_and_medians():
    step, timer, calls = _fake(lambda b, K, n: 1.0 + 0.01 * K + (5.0 if n % 5 == 0 else 0.0))
    Ks, cs = profile_cost_table(step, [16, 64], 16, reps=5, warmup=2, timer=timer)
    grid = sorted({tokens_for(b, 16, r) for b in (16, 64) for r in (0.25, 0.5, 0.75, 1.0)})
    assert Ks == grid
    assert len(calls) == 8 * (2 + 5)
    # one outlier in five per grid point at most: the median is the clean value
    assert np.allclose(cs, [1.0 + 0.01 * K for K in Ks])


def test_equal_token_counts_share_a_knot():
    # b=8 at rho=1 and b=16 at rho=0.5 both verify 8*9 = 72 tokens; their medians average
    step, timer, _ = _fake(lambda b, K, n: float(b))
    Ks, cs = profile_cost_table(step, [8, 16], 8, ratios=(0.5, 1.0), reps=3, warmup=0, timer=timer)
    assert Ks == [36, 72, 144]
    assert cs == [8.0, 12.0, 16.0]


def test_bad_grids_and_timings():
    step, timer, _ = _fake(lambda b, K, n: 1.0)
    for kw in (dict(batch_sizes=[]), dict(batch_sizes=[0]), dict(ratios=()), dict(ratios=(1.5,)),
               dict(reps=0), dict(warmup=-1), dict(depth=-1)):
        args = dict(batch_sizes=[4], depth=3, reps=1, warmup=0, timer=timer)
        args.update(kw)
        with pytest.raises(ValueError):
            profile_cost_table(step, **args)
    zero_step, zero_timer, _ = _fake(lambda b, K, n: 0.0)
    with pytest.raises(ValueError):
        profile_cost_table(zero_step, [4], 3, reps=1, warmup=0, timer=zero_timer)
    many = [17, 19, 23, 29, 31, 37, 41, 43, 47]
    assert len({tokens_for(b, 16, r) for b in many for r in (0.25, 0.5, 0.75, 1.0)}) > 32
    with pytest.raises(ValueError):
        profile_cost_table(step, many, 16, reps=1, warmup=0, timer=timer)
    assert MAX_COST_KNOTS == 32
