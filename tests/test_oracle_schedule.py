"""Pins for the D-cut scheduling oracle (CPU only): exhaustive allocation search,
exact rational objectives, the printed budgets of eq. K_rho and its figure, and the
structural claims of the D-cut section (fixed depth never beats the global ranking at
equal budget; ratio 1 keeps everything; only drafts are discarded)."""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle.schedule import dcut_schedule, candidate_budgets, k_rho, prefix_confidences
from synth import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _scores(alpha, Ds):
    # library route: numpy's float32 running product
    out = []
    for i, D in enumerate(Ds):
        s = np.cumprod(np.concatenate([[np.float32(1.0)], alpha[i, :D].astype(np.float32)]),
                       dtype=np.float32)
        out.append([int(np.rint(np.float64(v) * 2.0 ** 48)) for v in s])
    return out


def test_prefix_confidences_match_cumprod():
    a = np.random.default_rng(0).beta(8, 2, 30).astype(np.float32)
    s = prefix_confidences(a, 30)
    ref = np.cumprod(np.concatenate([[np.float32(1)], a]), dtype=np.float32)
    assert np.array_equal(s, ref)


def test_budgets_printed_values():
    with open(os.path.join(GOLDEN, "dcut_budgets.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        assert c["B"] * (c["D"] + 1) == c["N"]
        assert k_rho(c["B"], c["N"], c["rho"]) == c["K"]
    assert candidate_budgets(64, 1088, 384) == [272, 384]
    assert candidate_budgets(6, 48, 0) == [12, 24, 36, 48]


@pytest.mark.parametrize("trial", range(12))
def test_exhaustive_allocation_search(trial):
    """For every candidate K the oracle's U(K) equals the best prefix allocation over all
    (n_1..n_B) with sum(n_i + 1) = K, and its chosen K maximises the exact rational
    objective (ties -> smaller K)."""
    rng = np.random.default_rng(trial)
    B = int(rng.integers(1, 4))
    Dmax = int(rng.integers(0, 4))
    Ds = rng.integers(0, Dmax + 1, B)
    alpha = rng.random((B, Dmax)).astype(np.float32)
    if trial % 3 == 0:                      # force exact ties between requests
        alpha[:] = np.float32(0.5)
    a, b = [(1.0, 0.05), (0.0, 1.0), (2.0, 0.3)][trial % 3]
    budget = [0, B + 1, 2 * B][trial % 3]
    S = _scores(alpha, Ds)
    for objective in ("throughput", "net"):
        res = dcut_schedule(alpha, Ds, a, b, budget, objective=objective)
        best_by_K = {}
        for alloc in itertools.product(*[range(D + 1) for D in Ds]):
            K = sum(n + 1 for n in alloc)
            U = sum(sum(S[i][: alloc[i] + 1]) for i in range(B))
            best_by_K[K] = max(best_by_K.get(K, -1), U)
        for K, U, _ in res["table"]:
            assert best_by_K[K] == U
        # the chosen allocation is feasible and reaches the optimum at its K
        keep = res["keep_len"]
        assert all(0 <= keep[i] <= Ds[i] for i in range(B))
        assert sum(int(n) + 1 for n in keep) == res["K"]
        assert sum(sum(S[i][: keep[i] + 1]) for i in range(B)) == best_by_K[res["K"]]
        # exact rational objective
        fa = Fraction(float(np.float32(a)))
        fb = Fraction(float(np.float32(b)))
        def obj(K):
            u = Fraction(best_by_K[K], 2 ** 48)
            return u / (fa + fb * K) if objective == "throughput" else u - (fa + fb * K)
        cands = [K for K, _, _ in res["table"]]
        top = max(obj(K) for K in cands)
        assert res["K"] == min(K for K in cands if obj(K) == top)


def test_full_ratio_keeps_everything_and_floor_keeps_roots():
    sch = W.c4_alpha(seed=1, B=16, D=8)
    full = dcut_schedule(sch.alpha, None, 1.0, 0.0, 0, ratios=(1.0,))
    assert np.array_equal(full["keep_len"], np.full(16, 8))
    tiny = dcut_schedule(sch.alpha, None, 1.0, 0.05, 16, ratios=(0.01,))
    assert tiny["K"] == 16 and np.all(tiny["keep_len"] == 0)


def test_global_never_worse_than_fixed_depth():
    """At the same budget K = B (m+1), the global top-K keeps at least the expected
    progress of cutting every request at depth m (the D-cut section's comparison)."""
    for seed in range(10):
        sch = W.c4_alpha(seed=seed, B=12, D=8)
        S = _scores(sch.alpha, [8] * 12)
        for m in range(9):
            K = 12 * (m + 1)
            ratio = K / (12 * 9)
            res = dcut_schedule(sch.alpha, None, 1.0, 0.0, K, ratios=(ratio,))
            assert res["K"] == K
            fixed = sum(sum(S[i][: m + 1]) for i in range(12))
            assert res["U_q48"] >= fixed


def test_reallocation_favours_confident_requests():
    alpha = np.array([[0.95] * 6, [0.2] * 6], np.float32)
    res = dcut_schedule(alpha, None, 1.0, 0.0, 8, ratios=(0.5,))
    assert res["K"] == 7 and list(res["keep_len"]) == [5, 0]
    alpha2 = np.array([[0.5] * 3, [0.5] * 3], np.float32)      # exact tie -> lower request first
    res2 = dcut_schedule(alpha2, None, 1.0, 0.0, 3, ratios=(1.0,))
    assert list(res2["keep_len"]) == [1, 0]


def test_prefix_closed_and_only_discards():
    sch = W.c4_alpha(seed=5)
    res = dcut_schedule(sch.alpha, sch.draft_len, sch.cost_a, sch.cost_b, sch.budget)
    kept = {(i, k) for _, i, k in res["order"][: res["K"]]}
    for i in range(64):
        n = res["keep_len"][i]
        assert all((i, k) in kept for k in range(n + 1))
        assert 0 <= n <= 16
    assert res["K"] in (272, 384)


def test_invalid_alpha_rejected():
    with pytest.raises(ValueError):
        dcut_schedule(np.array([[0.5, 1.5]], np.float32), None, 1.0, 0.1, 0)
    with pytest.raises(ValueError):
        dcut_schedule(np.array([[np.nan, 0.5]], np.float32), None, 1.0, 0.1, 0)


def test_objective_ties_pick_the_smaller_budget():
    """alpha = 0 makes every extra slot worth nothing; with no per-token cost all candidates
    tie on either objective and the smallest K wins."""
    alpha = np.zeros((4, 5), np.float32)
    for objective in ("throughput", "net"):
        res = dcut_schedule(alpha, None, 1.0, 0.0, 0, objective=objective)
        assert len({o for _, _, o in res["table"]}) == 1
        assert res["K"] == min(K for K, _, _ in res["table"]) == 6
        assert np.all(res["keep_len"] == 0) or res["K"] > 4


# ---- profiled latency table c(K) (AngelSpec explainer, D-cut section, Figure 3 panel 2) ----

from oracle.schedule import table_cost, check_cost_table  # noqa: E402


def _exact_interp(K, Ks, cs):
    """Piecewise-linear interpolation in exact rationals, end values held outside."""
    if K <= Ks[0]:
        return Fraction(cs[0])
    if K >= Ks[-1]:
        return Fraction(cs[-1])
    for j in range(len(Ks) - 1):
        if Ks[j] <= K < Ks[j + 1]:
            return Fraction(cs[j]) + (Fraction(cs[j + 1]) - Fraction(cs[j])) * Fraction(K - Ks[j], Ks[j + 1] - Ks[j])
    raise AssertionError


def _random_table(rng, lo, hi):
    n = int(rng.integers(1, 9))
    Ks = sorted(set(int(v) for v in rng.integers(lo, hi + 1, n)))
    cs = [float(v) for v in rng.uniform(0.5, 40.0, len(Ks))]
    return Ks, cs


def test_table_cost_matches_library_interpolation():
    """numpy.interp is piecewise-linear interpolation holding the end values outside the
    knots; the table cost agrees with it to a few ulp of the largest latency everywhere,
    exactly at the knots, and with the exact rational interpolant to within the four
    roundings of its formula (each at most half an ulp of the largest latency)."""
    rng = np.random.default_rng(7)
    for _ in range(200):
        Ks, cs = _random_table(rng, 1, 400)
        for K in range(0, 420, 7):
            got = table_cost(K, Ks, cs)
            ref = float(np.interp(K, Ks, cs))
            ulp = Fraction(float(np.spacing(max(cs))))
            assert abs(Fraction(got) - Fraction(ref)) <= 8 * ulp
            assert abs(Fraction(got) - _exact_interp(K, Ks, cs)) <= 2 * ulp
        for k, c in zip(Ks, cs):
            assert table_cost(k, Ks, cs) == c


@pytest.mark.parametrize("trial", range(12))
def test_table_cost_exhaustive_allocation_search(trial):
    """With a latency table the chosen K maximises U(K) / c(K) (or U(K) - c(K)) computed in
    exact rationals from the exhaustive best allocation and the exact interpolant; near-ties
    within two roundings may go either way and are skipped."""
    rng = np.random.default_rng(100 + trial)
    B = int(rng.integers(1, 4))
    Dmax = int(rng.integers(0, 4))
    Ds = rng.integers(0, Dmax + 1, B)
    alpha = rng.random((B, Dmax)).astype(np.float32)
    N = int(sum(d + 1 for d in Ds))
    Ks, cs = _random_table(rng, 1, N + 2)
    if trial % 4 == 0:                      # knots exactly at every candidate
        cands = candidate_budgets(B, N, 0)
        Ks, cs = cands, [float(v) for v in rng.uniform(0.5, 5.0, len(cands))]
    S = _scores(alpha, Ds)
    best_by_K = {}
    for alloc in itertools.product(*[range(D + 1) for D in Ds]):
        K = sum(n + 1 for n in alloc)
        best_by_K[K] = max(best_by_K.get(K, -1), sum(sum(S[i][: alloc[i] + 1]) for i in range(B)))
    for objective in ("throughput", "net"):
        res = dcut_schedule(alpha, Ds, 0.0, 0.0, 0, objective=objective, cost_table=(Ks, cs))
        for K, U, _ in res["table"]:
            assert best_by_K[K] == U
        def obj(K):
            u = Fraction(best_by_K[K], 2 ** 48)
            c = _exact_interp(K, Ks, cs)
            return u / c if objective == "throughput" else u - c
        cands = [K for K, _, _ in res["table"]]
        vals = sorted((obj(K) for K in cands), reverse=True)
        if len(vals) > 1 and vals[0] != vals[1] and abs(vals[0] - vals[1]) < abs(vals[0]) * Fraction(1, 10 ** 12):
            continue
        top = vals[0]
        assert res["K"] == min(K for K in cands if obj(K) == top)


def test_table_cost_cliff_and_flat_tables():
    """A flat table leaves utility alone to decide (the largest candidate wins when every
    alpha > 0); a latency cliff past 300 tokens moves the C4 batch to the 272-token candidate;
    an affine table with dyadic values reproduces the linear cost model exactly."""
    sch = W.c4_alpha(seed=3)
    flat = dcut_schedule(sch.alpha, sch.draft_len, 0.0, 0.0, sch.budget, cost_table=([1], [2.0]))
    assert flat["K"] == max(K for K, _, _ in flat["table"]) == 384
    cliff = dcut_schedule(sch.alpha, sch.draft_len, 0.0, 0.0, sch.budget,
                          cost_table=([272, 300, 301], [10.0, 10.0, 1e6]))
    assert cliff["K"] == 272
    lin = dcut_schedule(sch.alpha, sch.draft_len, 1.0, 0.0625, sch.budget)
    aff = dcut_schedule(sch.alpha, sch.draft_len, 0.0, 0.0, sch.budget,
                        cost_table=([64, 1088], [1.0 + 0.0625 * 64, 1.0 + 0.0625 * 1088]))
    assert [t[:2] for t in aff["table"]] == [t[:2] for t in lin["table"]]
    assert aff["K"] == lin["K"] and np.array_equal(aff["keep_len"], lin["keep_len"])
    assert [t[2] for t in aff["table"]] == [t[2] for t in lin["table"]]


def test_cost_table_validation():
    for Ks, cs in [([], []), ([0, 5], [1.0, 2.0]), ([5, 5], [1.0, 2.0]), ([5, 3], [1.0, 2.0]),
                   ([5], [0.0]), ([5], [float("nan")]), ([5], [float("inf")]), ([1, 2], [1.0]),
                   (list(range(1, 34)), [1.0] * 33)]:
        with pytest.raises(ValueError):
            check_cost_table(Ks, cs)
    assert check_cost_table([1, 7], [0.5, 2]) == ([1, 7], [0.5, 2.0])
