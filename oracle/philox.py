"""Philox4x32-10 counter-based generator (oracle side).

Written from the definition in Salmon, Moraes, Dror, Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3" (SC'11): a 4x32-bit counter and a 2x32-bit key;
each of the 10 rounds multiplies counter words 0 and 2 by two fixed odd
constants, splits the 64-bit products into high and low halves, and permutes
and xors them with the other counter words and the round key; the key is
advanced by two Weyl constants (the golden ratio and sqrt(3)-1 in 32-bit fixed
point) between rounds.

The pages name no generator.  Uniforms for the accept test and the resampling
draw are keyed (seed; position, request, purpose, round) so that every draw
is independent of launch order.  u = (word0 >> 8) * 2^-24 lies in [0, 1) and
is exact in float32 and float64.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).
Pinned by tests/test_oracle_philox.py against Triton's interpreter and by
uniformity tests.
"""
from __future__ import annotations

import numpy as np

_MASK = np.uint64(0xFFFFFFFF)
_MUL0 = np.uint64(0xD2511F53)
_MUL1 = np.uint64(0xCD9E8D57)
_WEYL0 = np.uint64(0x9E3779B9)
_WEYL1 = np.uint64(0xBB67AE85)

PURPOSE_ACCEPT = 0
PURPOSE_RESAMPLE = 1
PURPOSE_DRAFT = 2


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Return the four 32-bit output words for counter (c0..c3) and key (k0, k1).

    Arguments broadcast like numpy arrays; results are uint64 arrays holding
    32-bit values.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _MASK for c in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & _MASK
    k1 = np.asarray(k1, dtype=np.uint64) & _MASK
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + _WEYL0) & _MASK
            k1 = (k1 + _WEYL1) & _MASK
        prod0 = _MUL0 * c0          # < 2^64, exact in uint64
        prod1 = _MUL1 * c2
        hi0, lo0 = prod0 >> np.uint64(32), prod0 & _MASK
        hi1, lo1 = prod1 >> np.uint64(32), prod1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0), lo1, (hi0 ^ c3 ^ k1), lo0
    return c0, c1, c2, c3


def uniform(seed: int, position, request, purpose, rnd):
    """u in [0, 1): 24 high bits of output word 0, as float64 (exact in float32 too)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    w0, _, _, _ = philox4x32_10(position, request, purpose, rnd, seed & 0xFFFFFFFF, seed >> 32)
    return (w0 >> np.uint64(8)).astype(np.float64) * (2.0 ** -24)
