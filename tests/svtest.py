"""Shared helpers for the GPU parity tests: move a synthetic batch to the device, run the
library through its C ABI, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import speculative_decoding_verification_74_gb300 as sv
from oracle.verify import verify_batch, NEAR_PICK
from synth import workloads as W

P_TOL = 1e-5   # absolute tolerance on reported probabilities (the stated contract)


def dev_rows(rows: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(rows).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(rows, dtype=np.float32)).to(device)


def i32(a, device="cuda"):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def f32(a, device="cuda"):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def run_ragged(b, ws=None, keep_len=None, want_pq=True):
    """Run sv_verify_ragged on a synth VerifyBatch; returns numpy outputs."""
    kl = b.keep_len if keep_len is None else keep_len
    out = sv.verify_ragged(dev_rows(b.target, b.dtype), i32(b.t_offsets),
                           dev_rows(b.draft, b.dtype) if b.draft is not None else None,
                           i32(b.d_offsets) if b.draft is not None else None,
                           i32(b.tokens), i32(kl), f32(b.temperature), b.Kmax, seed=b.seed, round_=b.round,
                           request_ids=i32(b.request_ids), ws=ws, want_pq=want_pq)
    torch.cuda.synchronize()
    return tuple(None if o is None else o.cpu().numpy() for o in out)


def oracle(b, keep_len=None):
    kl = b.keep_len if keep_len is None else keep_len
    return verify_batch(b.target, b.t_offsets, b.draft, b.d_offsets, b.tokens, kl, b.temperature, b.seed,
                        b.round, b.request_ids, b.dtype, b.Kmax)


NEAR_TOL = 1e-6  # the oracle's near-boundary band: |u - p/q| < 1e-6, or u' Z within 1e-6 Z of a bin edge


def near_cap(n_requests: int) -> int:
    """Most requests a comparison without its batch may excuse at a near-boundary decision: one
    per 32 requests compared, at least one."""
    return max(1, n_requests // 32)


def _decode(rows, dtype):
    return (W.bf16_bits_to_f32(rows) if dtype == "bf16" else np.asarray(rows, np.float32)).astype(np.float64)


def expected_excused(b, orc, idx, keep_len) -> float:
    """Expected number of requests the oracle's near-boundary band excuses, computed without the
    oracle's band code: a draw uniform u' lands within NEAR_TOL * Z of an edge of the bin it picks
    with probability sum_v min(r_v / Z, 2 NEAR_TOL) (r = the weights drawn from, here from scipy's
    softmax of the row the oracle drew from), and each accept test is near with probability at
    most 2 NEAR_TOL.  Wide flat rows (chat rows over 151936 entries at T = 1) put several percent
    of their draws in the band; peaked rows almost none."""
    from scipy.special import softmax
    lam = 0.0
    for i in idx:
        T = float(np.float32(b.temperature[i]))
        a = int(orc["accept_len"][i])
        if not T > 0.0 or a < 0:
            continue
        n = int(keep_len[i])
        P = softmax(_decode(b.target[b.t_offsets[i] + a], b.dtype) / T)
        r = P
        if a < n:
            r = np.maximum(0.0, P - softmax(_decode(b.draft[b.d_offsets[i] + a], b.dtype) / T))
            if not r.sum() > 0.0:
                r = P
        lam += float(np.minimum(r / r.sum(), 2 * NEAR_TOL).sum()) + 2 * NEAR_TOL * (a + 1)
    return lam


def compare(orc, tok, alen, p=None, q=None, keep_len=None, temps=None, requests=None, max_near=None, batch=None):
    """Tokens and accepted lengths bit-exact up to the first near-boundary decision the oracle
    reports (|u - p/q| < 1e-6, or an inverse-CDF pick within 1e-6 Z of a bin edge); p, q within
    P_TOL.  The number of requests that stop at such a decision is bounded: with the batch given,
    by lam + 4 sqrt(lam) + 2 with lam = expected_excused (a Poisson tail of about 1e-4); without
    it, by near_cap; `max_near` overrides both.  Returns that number, which is also printed."""
    B = len(alen)
    near = 0
    idx = list(range(B) if requests is None else requests)
    for i in idx:
        npos = int(orc["near_pos"][i])
        if npos < 0:
            assert alen[i] == orc["accept_len"][i], (i, alen[i], orc["accept_len"][i])
            assert np.array_equal(tok[i], orc["tokens"][i]), (i, tok[i], orc["tokens"][i])
        else:
            near += 1
            assert np.array_equal(tok[i, :npos], orc["tokens"][i, :npos]), i
            if orc["near_kind"][i] == NEAR_PICK:
                assert alen[i] == orc["accept_len"][i], i
        if p is not None and keep_len is not None:
            n = int(keep_len[i])
            if n:
                assert np.allclose(p[i, :n], orc["p"][i, :n], atol=P_TOL, rtol=0), (i, p[i, :n], orc["p"][i, :n])
                assert np.allclose(q[i, :n], orc["q"][i, :n], atol=P_TOL, rtol=0), (i, q[i, :n], orc["q"][i, :n])
            assert np.all(np.isnan(p[i, n:])) and np.all(np.isnan(q[i, n:]))
    if max_near is not None:
        cap = max_near
    elif batch is not None:
        lam = expected_excused(batch, orc, idx, batch.keep_len if keep_len is None else keep_len)
        cap = int(lam + 4.0 * np.sqrt(lam) + 2.0)
    else:
        cap = near_cap(len(idx))
    print(f"parity: {len(idx)} requests compared, {near} excused at a near-boundary decision (cap {cap})")
    assert near <= cap, (near, cap)
    return near


# ------------------------------------------------------------------ trees

def run_tree(b, ws=None):
    """Run sv_verify_tree on a synth TreeBatch; returns numpy (path, tokens, accept_len, flags)."""
    out = sv.verify_tree(dev_rows(b.target, b.dtype), dev_rows(b.draft, b.dtype), i32(b.node_offsets), i32(b.parent),
                         i32(b.tokens), f32(b.temperature), b.Nmax, seed=b.seed, round_=b.round,
                         request_ids=i32(b.request_ids), ws=ws)
    torch.cuda.synchronize()
    return tuple(o.cpu().numpy() for o in out)


def oracle_tree(b):
    from oracle.tree import verify_tree_batch
    return verify_tree_batch(b.target, b.draft, b.node_offsets, b.parent, b.tokens, b.temperature, b.seed, b.round,
                             b.request_ids, b.dtype)


def expected_excused_tree(b, orc, i) -> float:
    """Expected near-boundary excusals of tree request i, without the oracle's band code: the draw's
    weights rebuilt with scipy's softmax at the node where the oracle's walk stopped (p, or the
    residual after every child there was rejected: p' = norm(max(0, p' - q)) per child), then
    sum_v min(r_v / Z, 2 NEAR_TOL), plus 2 NEAR_TOL per accept test."""
    from scipy.special import softmax
    T = float(np.float32(b.temperature[i]))
    if not T > 0.0:
        return 0.0
    o, N = int(b.node_offsets[i]), b.nodes(i)
    par = b.parent[o:o + N]
    path = orc[i]["path"]
    node = path[-1] if path else 0
    P = softmax(_decode(b.target[o + node], b.dtype) / T)
    r = P
    kids = [c for c in range(1, N) if par[c] == node]
    if kids:
        Q = softmax(_decode(b.draft[o + node], b.dtype) / T)
        pr = P
        for _ in kids:
            res = np.maximum(0.0, pr - Q)
            if res.sum() > 0.0:
                r, pr = res, res / res.sum()
    return float(np.minimum(r / r.sum(), 2 * NEAR_TOL).sum()) + 2 * NEAR_TOL * N


def compare_tree(orc, path, tok, alen, b, requests=None, max_near=None):
    """Paths, emitted tokens and accepted lengths bit-exact up to the first near-boundary decision
    the oracle reports: an accept test of child c within 1e-6 of its threshold (the path must agree
    up to c's parent), or a pick within 1e-6 Z of a bin edge (the path must agree; the drawn token
    is free).  Excused requests are bounded by lam + 4 sqrt(lam) + 2 with lam the sum of
    expected_excused_tree, unless max_near is given.  Returns the number excused."""
    idx = list(range(b.B) if requests is None else requests)
    near = 0
    lam = 0.0
    for i in idx:
        r = orc[i]
        L = len(r["path"])
        lam += expected_excused_tree(b, orc, i)
        if r["near"] is None:
            assert alen[i] == L, (i, alen[i], L)
            assert list(path[i, :L]) == r["path"], (i, path[i, :L], r["path"])
            assert list(tok[i, :L + 1]) == r["tokens"], (i, tok[i, :L + 1], r["tokens"])
            assert np.all(path[i, L:] == -1) and np.all(tok[i, L + 1:] == -1), i
            continue
        near += 1
        kind, where = r["near"]
        if kind == NEAR_PICK:
            assert alen[i] == L and list(path[i, :L]) == r["path"], (i, path[i, :L], r["path"])
            assert list(tok[i, :L]) == r["tokens"][:L], i
        else:  # an accept test of child `where`: everything decided before it agrees
            pc = int(b.parent[b.node_offsets[i] + where])  # the walk reached pc before testing `where`
            pre = [] if pc == 0 else r["path"][: r["path"].index(pc) + 1]
            k = len(pre)
            assert list(path[i, :k]) == pre, (i, path[i, :k], pre)
    cap = max_near if max_near is not None else int(lam + 4.0 * np.sqrt(lam) + 2.0)
    print(f"tree parity: {len(idx)} requests compared, {near} excused at a near-boundary decision (cap {cap})")
    assert near <= cap, (near, cap)
    return near
