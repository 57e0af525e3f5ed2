"""Pins for the oracle's Philox4x32-10 and its uniforms (CPU only)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
from scipy import stats

from oracle.philox import philox4x32_10, uniform

_TRITON_SCRIPT = r"""
import json, os, sys
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl

@triton.jit
def _k(out_ptr, seed, c0p, c1p, c2p, c3p, N: tl.constexpr):
    i = tl.arange(0, N)
    a, b, c, d = tl.philox(seed, tl.load(c0p + i), tl.load(c1p + i), tl.load(c2p + i), tl.load(c3p + i))
    tl.store(out_ptr + i * 4 + 0, a)
    tl.store(out_ptr + i * 4 + 1, b)
    tl.store(out_ptr + i * 4 + 2, c)
    tl.store(out_ptr + i * 4 + 3, d)

cases = json.loads(sys.stdin.read())
res = []
for seed, ctrs in cases:
    n = len(ctrs)
    cols = [torch.tensor([c[j] for c in ctrs], dtype=torch.int64).to(torch.uint32) for j in range(4)]
    out = torch.zeros(n * 4, dtype=torch.uint32)
    _k[(1,)](out, seed, *cols, N=n)
    res.append([[int(v) for v in row] for row in out.to(torch.int64).view(n, 4).tolist()])
print(json.dumps(res))
"""


def _triton_philox(cases):
    pytest.importorskip("triton")
    try:
        r = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(cases),
                           capture_output=True, text=True, timeout=600,
                           env={**os.environ, "TRITON_INTERPRET": "1", "CUDA_VISIBLE_DEVICES": ""})
    except subprocess.TimeoutExpired:
        pytest.skip("triton interpreter timed out")
    if r.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + r.stderr.strip().splitlines()[-1][:200])
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_philox_matches_triton_library():
    """Philox4x32-10 words equal Triton's independent implementation (its CPU interpreter)."""
    rng = np.random.default_rng(123)
    seeds = [0, 1, 0xDEADBEEF, 0x123456789ABCDEF, (1 << 64) - 1 - (1 << 63)]
    cases = []
    for s in seeds:
        ctrs = rng.integers(0, 1 << 32, size=(8, 4), dtype=np.uint64).tolist()
        ctrs[0] = [0, 0, 0, 0]
        ctrs[1] = [0xFFFFFFFF] * 4
        cases.append([int(s), [[int(v) for v in c] for c in ctrs]])
    ref = _triton_philox(cases)
    for (s, ctrs), words in zip(cases, ref):
        c = np.asarray(ctrs, np.uint64)
        got = philox4x32_10(c[:, 0], c[:, 1], c[:, 2], c[:, 3], s & 0xFFFFFFFF, s >> 32)
        got = np.stack([np.asarray(g, np.uint64) for g in got], axis=1)
        assert got.tolist() == words, f"seed {s:#x}"


def test_uniform_is_exact_float32_and_in_range():
    u = uniform(7, np.arange(10000), 3, 1, 5)
    assert np.all(u >= 0.0) and np.all(u < 1.0)
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    assert np.all(np.mod(u * 2 ** 24, 1.0) == 0.0)


def test_uniform_chi_square_and_bits():
    u = uniform(2024, np.arange(1 << 16), np.arange(1 << 16) % 97, 0, 11)
    counts = np.histogram(u, bins=64, range=(0.0, 1.0))[0]
    assert stats.chisquare(counts).pvalue > 1e-4
    bits = (u * 2 ** 24).astype(np.int64)
    for b in range(24):
        frac = np.mean((bits >> b) & 1)
        assert abs(frac - 0.5) < 5 * 0.5 / np.sqrt(len(bits))


def test_streams_differ_by_every_key_field():
    base = uniform(9, np.arange(64), 2, 0, 3)
    for other in (uniform(10, np.arange(64), 2, 0, 3), uniform(9, np.arange(64), 3, 0, 3),
                  uniform(9, np.arange(64), 2, 1, 3), uniform(9, np.arange(64), 2, 0, 4),
                  uniform(9, np.arange(1, 65), 2, 0, 3)):
        assert np.mean(base == other) < 0.1
