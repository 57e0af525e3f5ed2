"""D-cut batch-shared verification-depth allocation, oracle.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

What is computed, and where it comes from (AngelSpec explainer, section
"D-cut: verification depth is a shared resource", its Figure 3 pipeline and
eq. K_rho; AngelSpec abstract: expected utility combined with a profiled
cost model):
  1. Per request i, the prefix-confidence scores s_{i,0} = 1 and
     s_{i,k} = s_{i,k-1} * alpha_{i,k} for k = 1..D_i.  Keeping n_i drafted
     positions is worth A_i(n_i) = sum_{k=0..n_i} s_{i,k} expected tokens.
  2. All positions of the whole batch are flattened and ranked by score;
     a global top-K is kept, whatever request a position belongs to.
  3. K is one of K_rho = max(B, ceil(rho * N)) for rho in {0.25, 0.5, 0.75,
     1.0}, N = sum_i (D_i + 1) (= B (D+1) when every request drafted D), and
     the rho picked is the one whose projected throughput U(K) / c(K) is
     largest, U(K) the kept scores' sum and c(K) the profiled round cost.

Readings where the pages are silent (each listed in the design notes):
  * s is computed in float32, left to right.
  * Slot k = 0 (the always-verified root / bonus position) has s = 1 and is
    always kept: the floor K >= B in eq. K_rho reserves one slot per request.
    Remaining slots are ranked by (s descending, request ascending, position
    ascending); with 0 <= alpha <= 1 this keeps a prefix of every request.
  * The profiled cost table is either the linear model c(K) = a + b*K
    (float64 from the float32 a, b) or a latency table: knots (K_j, c_j) with
    K_j strictly increasing verify-token counts and c_j > 0 the profiled
    latencies.  Batch size and keep ratio set the token count K = K_rho(b)
    together, so the table is read as latency against K: piecewise linear
    between knots, the end value held outside them (table_cost).  A budget cap
    clips every candidate to [B, min(budget, N)] (budget <= 0 means no cap);
    duplicate candidates collapse.
  * U(K) is summed exactly as integers round(s * 2^48).
  * objective "throughput" = (U / 2^48) / c(K) (the default, "projected
    throughput"); objective "net" = U / 2^48 - c(K) ("utility minus cost").
    Equal objectives pick the smaller K.
"""
from __future__ import annotations

import math

import numpy as np

Q48 = 2.0 ** 48
DEFAULT_RATIOS = (0.25, 0.5, 0.75, 1.0)


def prefix_confidences(alpha_row, D: int) -> np.ndarray:
    """s_0 = 1, s_k = s_{k-1} * alpha_k in float32 (alpha_row[k-1] is alpha_k)."""
    s = np.empty(D + 1, np.float32)
    s[0] = np.float32(1.0)
    for k in range(1, D + 1):
        s[k] = np.float32(s[k - 1] * np.float32(alpha_row[k - 1]))
    return s


def k_rho(B: int, N: int, rho: float) -> int:
    """eq. K_rho: max(B, ceil(rho * N)), rho taken as float32 then float64."""
    return max(B, int(math.ceil(float(np.float32(rho)) * float(N))))


def candidate_budgets(B: int, N: int, budget: int, ratios=DEFAULT_RATIOS) -> list[int]:
    cap = N if budget <= 0 else min(int(budget), N)
    out = []
    for rho in ratios:
        K = min(k_rho(B, N, rho), cap)
        K = max(K, B)
        if K not in out:
            out.append(K)
    return sorted(out)


def q48(s) -> int:
    return int(np.rint(np.float64(s) * Q48))


def check_cost_table(knots_K, knots_c) -> tuple[list[int], list[float]]:
    """Validate a latency table: 1..32 knots, K_j >= 1 strictly increasing, c_j finite > 0."""
    Ks = [int(k) for k in knots_K]
    cs = [float(c) for c in knots_c]
    if not 1 <= len(Ks) <= 32 or len(cs) != len(Ks):
        raise ValueError("a cost table has 1..32 knots")
    if Ks[0] < 1 or any(b <= a for a, b in zip(Ks, Ks[1:])):
        raise ValueError("cost-table token counts must be >= 1 and strictly increasing")
    if not all(math.isfinite(c) and c > 0.0 for c in cs):
        raise ValueError("cost-table latencies must be finite and positive")
    return Ks, cs


def table_cost(K: int, knots_K, knots_c) -> float:
    """Latency of verifying K tokens from the profiled table (float64).

    At or below the first knot: c_0; at or above the last: c_{n-1}.  Between
    knots j and j+1 (K_j <= K < K_{j+1}), in slope form: the segment's slope
    s_j = (c_{j+1} - c_j) / (K_{j+1} - K_j), then c_j + s_j * (K - K_j), each
    operation rounded once in that order."""
    n = len(knots_K)
    if K <= knots_K[0]:
        return float(knots_c[0])
    if K >= knots_K[n - 1]:
        return float(knots_c[n - 1])
    j = 0
    while knots_K[j + 1] <= K:
        j += 1
    slope = (float(knots_c[j + 1]) - float(knots_c[j])) / float(knots_K[j + 1] - knots_K[j])
    return float(knots_c[j]) + slope * float(K - knots_K[j])


def dcut_schedule(alpha, draft_len, cost_a: float, cost_b: float, budget: int,
                  ratios=DEFAULT_RATIOS, objective: str = "throughput", cost_table=None) -> dict:
    """Return keep_len [B] (n_i), the chosen K, U(K) as an exact Q48 integer and the
    per-candidate table.  cost_table = (knots_K, knots_c) replaces the linear cost
    a + b*K (cost_a, cost_b are then ignored)."""
    alpha = np.asarray(alpha, np.float32)
    B, Dmax = alpha.shape
    Ds = [Dmax] * B if draft_len is None else [int(v) for v in draft_len]
    if any(d < 0 or d > Dmax for d in Ds):
        raise ValueError("draft_len out of range")
    roots, rest = [], []
    for i in range(B):
        row = alpha[i, : Ds[i]]
        if np.any(~(row >= 0.0)) or np.any(row > 1.0):
            raise ValueError("alpha must lie in [0, 1]")
        s = prefix_confidences(row, Ds[i])
        roots.append((float(s[0]), i, 0))
        rest += [(float(s[k]), i, k) for k in range(1, Ds[i] + 1)]
    rest.sort(key=lambda e: (-e[0], e[1], e[2]))
    order = roots + rest
    N = len(order)
    if budget > 0 and budget < B:
        raise ValueError("budget below one slot per request")
    a = float(np.float32(cost_a))
    b = float(np.float32(cost_b))
    if cost_table is not None:
        knots_K, knots_c = check_cost_table(*cost_table)
    table = []
    best = None
    for K in candidate_budgets(B, N, budget, ratios):
        U = sum(q48(e[0]) for e in order[:K])
        cost = table_cost(K, knots_K, knots_c) if cost_table is not None else a + b * float(K)
        util = float(U) * (1.0 / Q48)
        obj = util / cost if objective == "throughput" else util - cost
        table.append((K, U, obj))
        if best is None or obj > best[2]:
            best = (K, U, obj)
    K, U, _ = best
    counts = [0] * B
    for _, i, _k in order[:K]:
        counts[i] += 1
    keep = np.asarray([c - 1 for c in counts], np.int32)
    return {"keep_len": keep, "K": K, "U_q48": U, "N": N, "table": table, "order": order}
