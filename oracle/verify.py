"""Lossless draft verification, fp64 oracle.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

What is computed, and where it comes from:
  * One verification pass checks every drafted token of a request against the
    target, by rejection sampling, and emits only what the target would have
    sampled (AngelSpec release article, "Why one universal drafter
    underperforms"; AngelSpec explainer, introduction and "D-cut": pruning
    never changes the target distribution).
  * One rejection voids every later drafted position, so the accepted length
    is the number of leading accepts: a product over the prefix, not a sum
    (AngelSpec explainer, "MTP: fix position 2 and 3", eq. L_e2e).
  * The pages do not spell out the accept rule, the residual or the bonus
    draw.  This oracle takes the textbook speculative-sampling reading:
      p_k = softmax(t_k / T), q_k = softmax(d_k / T)
      accept position k  <=>  u_k * q_k(x_k) < p_k(x_k)   (u < min(1, p/q))
      a = first rejected position (n if none)
      y ~ norm(max(0, p_a - q_a)) if a < n, else y ~ p_n (bonus row)
    drawn by inverse CDF: y = first v with cumsum(r)[v] > u' * sum(r), the
    cumulative sum taken sequentially in vocabulary order.
  * T == 0 is greedy: accept x_k iff x_k is the first argmax of t_k; the
    emitted token after the accepted prefix is the first argmax of t_a
    (AngelSpec release article, "The MTP path": T = 0 acceptance).

Readings where the pages are silent (each listed in the design notes):
  * q_k(x_k) == 0: the product form accepts iff p_k(x_k) > 0; flag bit 0.
  * sum(r) == 0 at a rejection: draw from p_a instead; flag bit 1.
  * Greedy rows report p_k = 1 if x_k is the target argmax else 0, q_k = 1.
  * Near-boundary decisions (|u - p/q| < 1e-6 for an accept test,
    |cumsum - u' Z| < 1e-6 Z next to the picked index) are reported in
    `near`, so a comparison can stop exact checking from that position on.
"""
from __future__ import annotations

import numpy as np

from .philox import uniform, PURPOSE_ACCEPT, PURPOSE_RESAMPLE

NEAR_ACCEPT = 1
NEAR_PICK = 2
NEAR_TOL = 1e-6

FLAG_Q_ZERO = 1
FLAG_Z_ZERO = 2


def decode_rows(rows: np.ndarray, dtype: str) -> np.ndarray:
    """bf16 bits (uint16) or float32 rows -> float64, exactly."""
    rows = np.asarray(rows)
    if dtype == "bf16":
        return (rows.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return rows.astype(np.float32).astype(np.float64)


def softmax_T(x: np.ndarray, T: float) -> np.ndarray:
    """softmax(x / T) in float64, shifted by the row max for range."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp((x - np.max(x)) / T)
    return e / np.sum(e)


def request_uniforms(seed: int, request_id: int, rnd: int, n: int):
    """u_k for the accept test at positions 0..n-1 and u'_j for a draw at position j = 0..n."""
    u_acc = uniform(seed, np.arange(n), request_id, PURPOSE_ACCEPT, rnd) if n else np.zeros(0)
    u_res = uniform(seed, np.arange(n + 1), request_id, PURPOSE_RESAMPLE, rnd)
    return np.atleast_1d(u_acc), np.atleast_1d(u_res)


def verify_request(t: np.ndarray, d: np.ndarray | None, tokens, T: float, u_acc, u_res) -> dict:
    """Verify one request.

    t       [n+1, V] float64 target logits (row n is the bonus row)
    d       [n, V] float64 draft logits, or None (greedy with tokens given)
    tokens  [n] drafted tokens, or None (greedy: x_k = first argmax of d_k)
    T       temperature, 0 = greedy
    u_acc   [n] uniforms for the accept tests; u_res [n+1] uniforms for the draw at position a
    """
    n = t.shape[0] - 1
    V = t.shape[1]
    out = {"flags": 0, "near": None}
    if T == 0.0:
        g = [int(np.argmax(t[k])) for k in range(n + 1)]
        x = [int(v) for v in tokens[:n]] if tokens is not None else [int(np.argmax(d[k])) for k in range(n)]
        a = n
        for k in range(n):
            if x[k] != g[k]:
                a = k
                break
        out.update(tokens=x[:a] + [g[a]], accept_len=a,
                   p=[1.0 if x[k] == g[k] else 0.0 for k in range(n)], q=[1.0] * n)
        return out

    x = [int(v) for v in tokens[:n]]
    P = [softmax_T(t[k], T) for k in range(n + 1)]
    Q = [softmax_T(d[k], T) for k in range(n)]
    p = [float(P[k][x[k]]) for k in range(n)]
    q = [float(Q[k][x[k]]) for k in range(n)]

    # accept tests, left to right; the first rejection ends the accepted prefix
    a = n
    for k in range(n):
        if q[k] == 0.0:
            out["flags"] |= FLAG_Q_ZERO
        elif out["near"] is None and abs(u_acc[k] - p[k] / q[k]) < NEAR_TOL:
            out["near"] = (NEAR_ACCEPT, k)
        if not (u_acc[k] * q[k] < p[k]):
            a = k
            break

    # residual at the first rejection, or the bonus row when everything was accepted
    r = np.maximum(0.0, P[a] - Q[a]) if a < n else P[n]
    c = np.cumsum(r)
    Z = c[-1]
    if not Z > 0.0:
        out["flags"] |= FLAG_Z_ZERO
        r = P[a]
        c = np.cumsum(r)
        Z = c[-1]
    thr = u_res[a] * Z
    y = int(np.searchsorted(c, thr, side="right"))   # first v with c[v] > thr
    if y >= V:                                        # cannot happen for u' < 1; keep it defined
        y = int(np.nonzero(r > 0)[0][-1])
    if out["near"] is None:
        if abs(c[y] - thr) < NEAR_TOL * Z or (y > 0 and abs(c[y - 1] - thr) < NEAR_TOL * Z):
            out["near"] = (NEAR_PICK, a)
    out.update(tokens=x[:a] + [y], accept_len=a, p=p, q=q)
    return out


def verify_batch(target, t_offsets, draft, d_offsets, tokens, keep_len, temperature, seed, rnd,
                 request_ids, dtype, Kmax) -> dict:
    """Verify a packed ragged batch (the library's layout), request by request.

    Returns tokens [B, Kmax+1] (-1 padded), accept_len [B], p/q [B, Kmax] (NaN beyond n_i),
    flags [B], near_kind [B] (0 none, 1 accept test, 2 pick) and near_pos [B] (-1 none).
    """
    B = len(keep_len)
    toks = np.full((B, Kmax + 1), -1, np.int32)
    alen = np.zeros(B, np.int32)
    P = np.full((B, max(Kmax, 1)), np.nan)
    Qo = np.full((B, max(Kmax, 1)), np.nan)
    flags = np.zeros(B, np.uint8)
    near_kind = np.zeros(B, np.int32)
    near_pos = np.full(B, -1, np.int32)
    for i in range(B):
        n = int(keep_len[i])
        T = float(np.float32(temperature[i]))
        t = decode_rows(target[t_offsets[i]: t_offsets[i] + n + 1], dtype)
        need_d = (T > 0.0) or tokens is None
        d = decode_rows(draft[d_offsets[i]: d_offsets[i] + n], dtype) if need_d else None
        tk = None if tokens is None else np.asarray(tokens[i])
        rid = int(request_ids[i]) if request_ids is not None else i
        u_acc, u_res = request_uniforms(seed, rid, rnd, n)
        res = verify_request(t, d, tk, T, u_acc, u_res)
        a = res["accept_len"]
        toks[i, : a + 1] = res["tokens"]
        alen[i] = a
        P[i, :n] = res["p"]
        Qo[i, :n] = res["q"]
        flags[i] = res["flags"]
        if res["near"] is not None:
            near_kind[i], near_pos[i] = res["near"]
    return {"tokens": toks, "accept_len": alen, "p": P[:, :Kmax], "q": Qo[:, :Kmax], "flags": flags,
            "near_kind": near_kind, "near_pos": near_pos}
