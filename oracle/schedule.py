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
  * The profiled cost table is the linear model c(K) = a + b*K (float64 from
    the float32 a, b); a budget cap clips every candidate to [B, min(budget, N)]
    (budget <= 0 means no cap); duplicate candidates collapse.
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


def dcut_schedule(alpha, draft_len, cost_a: float, cost_b: float, budget: int,
                  ratios=DEFAULT_RATIOS, objective: str = "throughput") -> dict:
    """Return keep_len [B] (n_i), the chosen K, U(K) as an exact Q48 integer and the
    per-candidate table."""
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
    table = []
    best = None
    for K in candidate_budgets(B, N, budget, ratios):
        U = sum(q48(e[0]) for e in order[:K])
        cost = a + b * float(K)
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
