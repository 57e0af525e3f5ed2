"""Startup profiling of the D-cut runtime latency table.

The D-cut pipeline (AngelSpec explainer, D-cut section, Figure 3 panel 2)
profiles a runtime cost table once, at startup, across batch sizes and keep
ratios.  Every step then uses it to pick the keep ratio whose projected
throughput is largest (panel 3, eq. K_rho).  For batch size b and depth D, a
keep ratio rho verifies K = max(b, ceil(rho * b * (D + 1))) tokens.  Batch size
and ratio therefore enter the verify cost together, through K, and the table
is kept as latency against K: sorted knots (K_j, c_j).  sv_schedule_depth_table
interpolates them linearly on the GPU.

The verify step being profiled belongs to the caller: the target model's
forward over the kept tokens, followed by the verification kernels.  This
module only times it on a (batch size x ratio) grid and reduces the grid to
knots.  It runs on the host once, outside the per-step path.
"""
from __future__ import annotations

import math
import statistics
from typing import Callable, Iterable

import torch

MAX_COST_KNOTS = 32  # SV_MAX_COST_KNOTS in include/sv.h
DEFAULT_RATIOS = (0.25, 0.5, 0.75, 1.0)


def tokens_for(b: int, depth: int, rho: float) -> int:
    """Verified tokens for batch size b, depth D and keep ratio rho: max(b, ceil(rho * b (D+1))),
    rho rounded to float32 first as the scheduler does."""
    rho32 = torch.tensor(rho, dtype=torch.float32).item()
    return max(b, int(math.ceil(rho32 * float(b * (depth + 1)))))


def cuda_event_timer(fn: Callable[[], None]) -> float:
    """Milliseconds of fn() on the current CUDA stream, by CUDA events."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    fn()
    end.record()
    end.synchronize()
    return float(start.elapsed_time(end))


def profile_cost_table(step: Callable[[int, int], None], batch_sizes: Iterable[int], depth: int,
                       ratios: Iterable[float] = DEFAULT_RATIOS, reps: int = 10, warmup: int = 3,
                       timer: Callable[[Callable[[], None]], float] | None = None
                       ) -> tuple[list[int], list[float]]:
    """Time step(b, K) on every (batch size, keep ratio) point and return the knots
    (token counts ascending, latencies).

    Each grid point runs `warmup` untimed calls, then `reps` timed calls; its latency is
    the median.  Grid points that verify the same K share one knot: the mean of their
    medians.  timer(fn) returns the duration of fn() (default: CUDA events on the
    current stream).  Raises ValueError on an empty grid, non-positive timings, or more
    than 32 distinct token counts."""
    if timer is None:
        timer = cuda_event_timer
    ratios = tuple(float(r) for r in ratios)
    batch_sizes = tuple(int(b) for b in batch_sizes)
    if not ratios or not batch_sizes or reps < 1 or warmup < 0 or depth < 0:
        raise ValueError("profiling needs batch sizes, ratios, depth >= 0, reps >= 1, warmup >= 0")
    if any(b < 1 for b in batch_sizes) or any(not 0.0 < r <= 1.0 for r in ratios):
        raise ValueError("batch sizes must be >= 1 and ratios in (0, 1]")
    by_K: dict[int, list[float]] = {}
    for b in batch_sizes:
        for rho in ratios:
            K = tokens_for(b, depth, rho)
            for _ in range(warmup):
                step(b, K)
            times = [float(timer(lambda: step(b, K))) for _ in range(reps)]
            med = statistics.median(times)
            if not (med > 0.0 and math.isfinite(med)):
                raise ValueError(f"non-positive or non-finite latency {med} at b={b}, K={K}")
            by_K.setdefault(K, []).append(med)
    if len(by_K) > MAX_COST_KNOTS:
        raise ValueError(f"{len(by_K)} distinct token counts; the table holds at most {MAX_COST_KNOTS}")
    Ks = sorted(by_K)
    return Ks, [sum(by_K[K]) / len(by_K[K]) for K in Ks]
