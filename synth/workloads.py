"""Seeded synthetic inputs for the verification and depth-scheduling path.

This module is the only code shared by the CUDA path's tests/bench and the
CPU oracle.  It draws random logits, draft tokens, temperatures and draft
confidences; it holds none of the verification or scheduling arithmetic
(no softmax, no accept test, no residual, no ranking).  The drafter's own
token choice is simulated here (it is an input to verification): sampled
requests draw x ~ softmax(d / T) by the Gumbel-max trick, greedy requests take
the first argmax of the draft row.

Recipes (sigma is a standard deviation):
  chat rows  : target ~ N(0, sigma_t), draft = target + N(0, sigma_n)
  code rows  : target_v = -A * ln(rank_v) + N(0, 0.1), rank a seeded random
               permutation of 1..V (affine family (a*v + c) mod V), with
               A = 6 / ln 2 so the top-1 / top-2 gap is about 6 nats;
               draft = target + N(0, sigma_n)
  bf16 rows are rounded to nearest-even from float32 and stored as uint16 bits.

Every array is a pure function of (config name, seed, round).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BF16 = "bf16"
F32 = "f32"

ZIPF_A = 6.0 / math.log(2.0)


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng([int(k) & 0xFFFFFFFF for k in key])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return uint16 bits.  In 32-bit integer
    arithmetic: bits + 0x7FFF + lsb cannot wrap for a non-NaN float (the largest, -inf, is
    0xFF800000), and NaNs are set apart."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + (np.uint32(0x7FFF) + lsb)) >> np.uint32(16)
    # keep NaN a NaN (never produced by the recipes, but be safe)
    nan = np.isnan(x)
    out = r.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32 (used only to build draft rows)."""
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _encode(x32: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x32) if dtype == BF16 else np.ascontiguousarray(x32, dtype=np.float32)


def _decode32(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(x) if dtype == BF16 else x


def chat_rows(rng: np.random.Generator, n: int, V: int, sigma: float) -> np.ndarray:
    return rng.standard_normal((n, V), dtype=np.float32) * np.float32(sigma)


def code_rows(rng: np.random.Generator, n: int, V: int) -> np.ndarray:
    """Zipf-peaked rows: -A*ln(rank) + N(0, 0.1) over a random permutation of ranks."""
    logtab = (-ZIPF_A * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    out = np.empty((n, V), dtype=np.float32)
    v = np.arange(V, dtype=np.int64)
    for r in range(n):
        while True:
            a = int(rng.integers(1, V)) if V > 1 else 1
            if math.gcd(a, V) == 1:
                break
        c = int(rng.integers(0, V))
        out[r] = logtab[(a * v + c) % V]
    out += rng.standard_normal((n, V), dtype=np.float32) * np.float32(0.1)
    return out


def gumbel_max_tokens(rng: np.random.Generator, d32: np.ndarray, T: float) -> np.ndarray:
    """Drafter sampling x ~ softmax(d / T) by the Gumbel-max trick (float64)."""
    g = -np.log(-np.log(rng.random(d32.shape)))
    return np.argmax(d32.astype(np.float64) / T + g, axis=-1).astype(np.int32)


def argmax_tokens(d32: np.ndarray) -> np.ndarray:
    return np.argmax(d32, axis=-1).astype(np.int32)


@dataclass
class VerifyBatch:
    """One verification round in the packed (ragged) layout the library takes.

    target      [sum_i (n_i + 1) or more, V] rows (uint16 bf16 bits or float32)
    t_offsets   [B + 1] int32, request i's target rows start at t_offsets[i]
    draft       [rows, V] or None; request i's draft row k is draft[d_offsets[i] + k]
    d_offsets   [B + 1] int32 or None
    tokens      [B, Kmax] int32 drafted tokens (-1 padding) or None (greedy from draft argmax)
    keep_len    [B] int32, positions to verify per request (n_i <= Kmax)
    temperature [B] float32 (0 = greedy)
    """
    name: str
    dtype: str
    B: int
    Kmax: int
    V: int
    target: np.ndarray
    t_offsets: np.ndarray
    draft: np.ndarray | None
    d_offsets: np.ndarray | None
    tokens: np.ndarray | None
    keep_len: np.ndarray
    temperature: np.ndarray
    seed: int
    round: int
    request_ids: np.ndarray
    meta: dict = field(default_factory=dict)

    def positions(self) -> int:
        return int(self.keep_len.sum())


def _pack(req_rows: list[np.ndarray], V: int, dtype: str) -> tuple[np.ndarray, np.ndarray]:
    offs = np.zeros(len(req_rows) + 1, dtype=np.int32)
    for i, r in enumerate(req_rows):
        offs[i + 1] = offs[i] + r.shape[0]
    store = np.uint16 if dtype == BF16 else np.float32
    out = np.empty((int(offs[-1]), V), dtype=store)
    for i, r in enumerate(req_rows):
        out[offs[i]:offs[i + 1]] = r
    return out, offs


def _request(rng, kind: str, K: int, V: int, sigma_t: float, sigma_n: float, T: float,
             dtype: str, draft_tokens_from: str):
    """Rows and drafted tokens for one request: (target[K+1], draft[K], tokens[K])."""
    t32 = chat_rows(rng, K + 1, V, sigma_t) if kind == "chat" else code_rows(rng, K + 1, V)
    t_enc = _encode(t32, dtype)
    t32 = _decode32(t_enc, dtype)
    d32 = t32[:K] + rng.standard_normal((K, V), dtype=np.float32) * np.float32(sigma_n)
    d_enc = _encode(d32, dtype)
    d32 = _decode32(d_enc, dtype)
    if K == 0:
        tok = np.zeros(0, np.int32)
    elif draft_tokens_from == "argmax" or T == 0.0:
        tok = argmax_tokens(d32)
    else:
        tok = gumbel_max_tokens(rng, d32, T)
    return t_enc, d_enc, tok


def make_batch(name: str, kinds: list[str], Ks: list[int], temps: list[float], V: int, dtype: str,
               seed: int, rnd: int, sigma: dict, *, tokens_given: bool = True,
               Kmax: int | None = None, keep_len: np.ndarray | None = None) -> VerifyBatch:
    B = len(kinds)
    Kmax = max(Ks) if Kmax is None else Kmax
    rng = _rng(seed, rnd, _name_key(name))
    ts, ds, toks = [], [], np.full((B, max(Kmax, 1)), -1, np.int32)
    for i in range(B):
        st, sn = sigma[kinds[i]]
        t_enc, d_enc, tok = _request(rng, kinds[i], Ks[i], V, st, sn, temps[i], dtype,
                                     "argmax" if not tokens_given else "sample")
        ts.append(t_enc)
        ds.append(d_enc)
        toks[i, :Ks[i]] = tok
    target, t_off = _pack(ts, V, dtype)
    draft, d_off = _pack(ds, V, dtype)
    kl = np.asarray(Ks, np.int32) if keep_len is None else np.asarray(keep_len, np.int32)
    return VerifyBatch(name=name, dtype=dtype, B=B, Kmax=Kmax, V=V, target=target, t_offsets=t_off,
                       draft=draft, d_offsets=d_off, tokens=toks[:, :Kmax] if tokens_given else None,
                       keep_len=kl, temperature=np.asarray(temps, np.float32), seed=seed, round=rnd,
                       request_ids=np.arange(B, dtype=np.int32))


def _name_key(name: str) -> int:
    h = 2166136261
    for ch in name.encode():
        h = ((h ^ ch) * 16777619) & 0xFFFFFFFF
    return h


# --------------------------------------------------------------------------------------------
# The five workloads (sizes can be shrunk for fast tests; defaults are the full sizes)
# --------------------------------------------------------------------------------------------

def c1_greedy(seed: int = 0, B: int = 4, K: int = 3, V: int = 32000) -> VerifyBatch:
    """Greedy T=0: target ~ N(0,2), draft = target + N(0,0.5), draft tokens = draft argmax (fused)."""
    return make_batch("c1", ["chat"] * B, [K] * B, [0.0] * B, V, BF16, seed, 0,
                      {"chat": (2.0, 0.5)}, tokens_given=False)


def c2_mtp(seed: int = 0, B: int = 16, K: int = 3, V: int = 151936, rnd: int = 0) -> VerifyBatch:
    """MTP-style T=1: target ~ N(0,3), draft = target + N(0,1), x ~ q."""
    return make_batch("c2", ["chat"] * B, [K] * B, [1.0] * B, V, BF16, seed, rnd,
                      {"chat": (3.0, 1.0)})


def c3_dfly(seed: int = 0, B: int = 64, K: int = 16, V: int = 151936, rnd: int = 0) -> VerifyBatch:
    """DFly-style T=0.6, fp32, Zipf-peaked target, draft = target + N(0,0.3), x ~ q."""
    return make_batch("c3", ["code"] * B, [K] * B, [0.6] * B, V, F32, seed, rnd,
                      {"code": (0.0, 0.3)})


@dataclass
class ScheduleInput:
    alpha: np.ndarray          # [B, Dmax] float32 in (0, 1)
    draft_len: np.ndarray      # [B] int32
    kinds: list[str]
    cost_a: float
    cost_b: float
    budget: int


def c4_alpha(seed: int = 0, B: int = 64, D: int = 16) -> ScheduleInput:
    """Draft confidences: half the requests Beta(8,2) (code-like), half Beta(3,3) (chat-like)."""
    rng = _rng(seed, 0, _name_key("c4-alpha"))
    code = np.zeros(B, bool)
    code[rng.permutation(B)[: B // 2]] = True
    a = np.where(code[:, None], rng.beta(8.0, 2.0, (B, D)), rng.beta(3.0, 3.0, (B, D)))
    a = np.clip(a.astype(np.float32), np.float32(1e-7), np.nextafter(np.float32(1), np.float32(0)))
    return ScheduleInput(alpha=a, draft_len=np.full(B, D, np.int32),
                         kinds=["code" if c else "chat" for c in code], cost_a=1.0, cost_b=0.05,
                         budget=384)


def c4_verify(sched: ScheduleInput, keep_len: np.ndarray, seed: int = 0, V: int = 151936,
              rnd: int = 0, full_rows: bool = True) -> VerifyBatch:
    """Ragged T=1 verify over the kept prefixes.  Every request carries all D draft positions
    (rows are laid out [B, D+1] / [B, D]); only the first keep_len[i] are verified."""
    B, D = sched.alpha.shape
    b = make_batch("c4", sched.kinds, [D] * B, [1.0] * B, V, BF16, seed, rnd,
                   {"chat": (3.0, 1.0), "code": (0.0, 0.3)}, Kmax=D, keep_len=keep_len)
    return b


def c5_mixed(seed: int = 0, rnd: int = 0, B: int = 64, V: int = 151936, Kc: int = 3, Kx: int = 16
             ) -> VerifyBatch:
    """Mixed round: half chat (K=3, N(0,3), noise 1.0), half code (K=16, Zipf, noise 0.3);
    temperature per request uniform in {0, 0.6, 1.0}; the roles are fixed by the seed, the
    rows and temperatures are redrawn each round."""
    role_rng = _rng(seed, 0, _name_key("c5-roles"))
    code = np.zeros(B, bool)
    code[role_rng.permutation(B)[: B // 2]] = True
    t_rng = _rng(seed, rnd, _name_key("c5-temps"))
    temps = [float(x) for x in np.asarray([0.0, 0.6, 1.0], np.float32)[t_rng.integers(0, 3, B)]]
    kinds = ["code" if c else "chat" for c in code]
    Ks = [Kx if c else Kc for c in code]
    return make_batch("c5", kinds, Ks, temps, V, BF16, seed, rnd,
                      {"chat": (3.0, 1.0), "code": (0.0, 0.3)})


def small(name: str, seed: int = 0) -> VerifyBatch:
    """Reduced versions that the oracle finishes in seconds (several vocab tiles, ragged tail)."""
    if name == "c1":
        return c1_greedy(seed, B=4, K=3, V=32000)
    if name == "c2":
        return c2_mtp(seed, B=5, K=3, V=20011)
    if name == "c3":
        return c3_dfly(seed, B=4, K=16, V=9001)
    if name == "c5":
        return c5_mixed(seed, 0, B=8, V=12007, Kc=3, Kx=16)
    raise KeyError(name)
