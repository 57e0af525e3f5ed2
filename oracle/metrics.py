"""Round-level acceptance metrics, oracle side.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Mean accepted length (MAL) counts, per verification round, the accepted
drafted tokens plus the one target token emitted after them; mean acceptance
is the accepted fraction of the drafted positions.  With D drafted positions
per round, MAL = 1 + D * mean acceptance (AngelSpec release article, "The
MTP path"; AngelSpec explainer, "MTP: fix position 2 and 3").  The expected
accepted length for fixed per-position acceptance rates beta_k is the sum of
prefix products sum_{m=1..D} prod_{k<m} beta_k (eq. L_e2e's product form).
"""
from __future__ import annotations

import numpy as np


def mean_accepted_length(accept_lens) -> float:
    return float(np.mean(np.asarray(accept_lens, np.float64) + 1.0))


def mean_acceptance(accept_lens, draft_lens) -> float:
    a = np.asarray(accept_lens, np.float64)
    d = np.asarray(draft_lens, np.float64)
    return float(np.sum(a) / np.sum(d))


def expected_accept_len(betas) -> float:
    """sum over m = 1..D of prod_{k < m} beta_k (a rejection voids every later position)."""
    total, run = 0.0, 1.0
    for b in betas:
        run *= float(b)
        total += run
    return total
