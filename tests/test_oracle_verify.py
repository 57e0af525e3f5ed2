"""Pins for the verification oracle (CPU only).

Everything here checks the oracle against something other than itself:
library routines (scipy softmax, torch bf16 decoding), the target
distribution that lossless verification must reproduce (exact integration of
the oracle's own decisions over its uniforms), brute force over every draft
tuple, and the closed-form expected accepted length.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax as sp_softmax

from oracle.verify import (decode_rows, softmax_T, verify_request, verify_batch, request_uniforms,
                           NEAR_ACCEPT, NEAR_PICK)
from oracle.metrics import mean_accepted_length, mean_acceptance, expected_accept_len
from synth import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ library special cases

def test_softmax_matches_scipy():
    rng = np.random.default_rng(0)
    for T in (0.3, 0.6, 1.0, 2.5):
        x = rng.normal(0, 4, 5000)
        assert np.max(np.abs(softmax_T(x, T) - sp_softmax(x / T))) < 1e-14


def test_decode_matches_torch_bf16():
    bits = np.random.default_rng(1).integers(0, 1 << 16, 4096).astype(np.uint16)
    finite = np.isfinite(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy())
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = decode_rows(bits, "bf16")
    assert np.array_equal(got[finite], ref[finite])


def test_generator_bf16_rounding_matches_torch():
    x = np.random.default_rng(2).normal(0, 3, 100000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.f32_to_bf16_bits(x), ref)


# ------------------------------------------------------------------ greedy brute force

def _first_max(row):
    return int(np.flatnonzero(row == row.max()).min())


@pytest.mark.parametrize("V,K", [(3, 1), (4, 3), (5, 2)])
def test_greedy_brute_force_all_draft_tuples(V, K):
    rng = np.random.default_rng(V * 10 + K)
    t = rng.integers(-2, 3, size=(K + 1, V)).astype(np.float64)   # integer logits: many ties
    chain = [_first_max(t[j]) for j in range(K + 1)]
    for x in itertools.product(range(V), repeat=K):
        res = verify_request(t, None, list(x), 0.0, np.zeros(K), np.zeros(K + 1))
        a = res["accept_len"]
        # the emitted tokens are exactly the target's greedy chain, cut at the first mismatch
        assert res["tokens"] == chain[: a + 1]
        assert list(x[:a]) == chain[:a]
        assert a == K or x[a] != chain[a]


def test_greedy_from_draft_argmax():
    rng = np.random.default_rng(5)
    t = rng.normal(size=(4, 50))
    d = t[:3] + rng.normal(scale=0.01, size=(3, 50))
    d[1] = -d[1]                      # position 1's draft argmax differs from the target's
    res = verify_request(t, d, None, 0.0, np.zeros(3), np.zeros(4))
    assert res["accept_len"] == 1
    assert res["tokens"] == [_first_max(t[0]), _first_max(t[1])]


# ------------------------------------------------------------------ losslessness, exactly

def _bisect(pred, iters=48):
    """Smallest u in [0,1) where pred(u) becomes True (pred monotone False->True)."""
    lo, hi = 0.0, 1.0
    if pred(0.0):
        return 0.0
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if pred(mid):
            hi = mid
        else:
            lo = mid
    return hi


def _emission_law(t, d, T, x):
    """Exact law of the oracle's output for draft tuple x: {emitted tuple: probability},
    integrating the oracle's decisions over its uniforms (each decision is a threshold
    in its own uniform)."""
    K = len(x)
    V = t.shape[1]
    law = {}
    prefix_prob = 1.0
    for a in range(K + 1):
        # probability that positions < a accept and position a rejects (or all accept at a=K)
        if a < K:
            def rejects(u, a=a):
                ua = np.zeros(K)
                ua[a] = u
                return verify_request(t, d, list(x), T, ua, np.zeros(K + 1))["accept_len"] == a
            theta = _bisect(rejects)                  # accept iff u < theta
            p_stop = prefix_prob * (1.0 - theta)
            u_force = 0.5 * (1.0 + theta) if theta < 1.0 else None
        else:
            p_stop = prefix_prob
            u_force = None
        if p_stop > 0.0:
            ua = np.zeros(K)
            if a < K:
                ua[a] = u_force
            # inverse-CDF draw: boundaries of y(u') for each vocabulary entry
            def pick(u):
                ur = np.zeros(K + 1)
                ur[a] = u
                r = verify_request(t, d, list(x), T, ua, ur)
                assert r["accept_len"] == a
                return r["tokens"][-1]
            prev = 0.0
            for v in range(V):
                b = 1.0 if v == V - 1 else _bisect(lambda u, v=v: pick(u) > v)
                if b > prev:
                    key = tuple(x[:a]) + (v,)
                    law[key] = law.get(key, 0.0) + p_stop * (b - prev)
                prev = b
        if a < K:
            prefix_prob *= theta
    return law


@pytest.mark.parametrize("V,K,T", [(2, 3, 1.0), (3, 2, 0.7), (3, 3, 1.6), (4, 2, 1.0)])
def test_lossless_exact_enumeration(V, K, T):
    """Completing the oracle's emission with target draws gives exactly prod_j p_j."""
    rng = np.random.default_rng(100 + V * 7 + K)
    t = rng.normal(0, 1.5, size=(K + 1, V))
    d = rng.normal(0, 1.5, size=(K, V))
    p = [sp_softmax(t[j] / T) for j in range(K + 1)]
    q = [sp_softmax(d[j] / T) for j in range(K)]
    emitted = {}
    for x in itertools.product(range(V), repeat=K):
        wx = float(np.prod([q[j][x[j]] for j in range(K)]))
        for seq, pr in _emission_law(t, d, T, x).items():
            emitted[seq] = emitted.get(seq, 0.0) + wx * pr
    assert abs(sum(emitted.values()) - 1.0) < 1e-9
    for full in itertools.product(range(V), repeat=K + 1):
        target = float(np.prod([p[j][full[j]] for j in range(K + 1)]))
        got = 0.0
        for L in range(1, K + 2):
            pre = tuple(full[:L])
            if pre in emitted:
                got += emitted[pre] * float(np.prod([p[j][full[j]] for j in range(L, K + 1)]))
        assert abs(got - target) < 1e-9, (full, got, target)


@pytest.mark.parametrize("V,K,T", [(3, 3, 1.0), (4, 2, 0.5)])
def test_expected_accept_len_closed_form(V, K, T):
    """E[a] = sum_m prod_{k<m} beta_k with beta_k = sum_v min(p_k, q_k) = 1 - TV(p_k, q_k)."""
    rng = np.random.default_rng(7 + V + K)
    t = rng.normal(0, 1.0, size=(K + 1, V))
    d = rng.normal(0, 1.0, size=(K, V))
    q = [sp_softmax(d[j] / T) for j in range(K)]
    p = [sp_softmax(t[j] / T) for j in range(K + 1)]
    ea = 0.0
    for x in itertools.product(range(V), repeat=K):
        wx = float(np.prod([q[j][x[j]] for j in range(K)]))
        for seq, pr in _emission_law(t, d, T, x).items():
            ea += wx * pr * (len(seq) - 1)
    betas = [float(np.sum(np.minimum(p[k], q[k]))) for k in range(K)]
    assert abs(ea - expected_accept_len(betas)) < 1e-9


def test_philox_driven_monte_carlo_acceptance():
    """Through the Philox uniforms and Gumbel-max drafts, the mean accepted length and the
    first emitted token's law match the closed forms."""
    V, K, T, n = 12, 3, 0.8, 3000
    rng = np.random.default_rng(11)
    t = rng.normal(0, 1.2, size=(K + 1, V))
    d = t[:K] + rng.normal(0, 0.8, size=(K, V))
    p0 = sp_softmax(t[0] / T)
    betas = [float(np.sum(np.minimum(sp_softmax(t[k] / T), sp_softmax(d[k] / T)))) for k in range(K)]
    lens, first = [], np.zeros(V)
    for s in range(n):
        x = W.gumbel_max_tokens(np.random.default_rng([s, 99]), d.astype(np.float32), T)
        u_acc, u_res = request_uniforms(s, 0, 0, K)
        r = verify_request(t, d, x, T, u_acc, u_res)
        lens.append(r["accept_len"])
        first[r["tokens"][0]] += 1
    lens = np.asarray(lens, float)
    mu = expected_accept_len(betas)
    assert abs(lens.mean() - mu) < 4.5 * lens.std() / np.sqrt(n)
    from scipy.stats import chisquare
    assert chisquare(first, p0 * n).pvalue > 1e-4


# ------------------------------------------------------------------ reading-specific cases

def test_zero_draft_probability_accepts_iff_target_positive():
    t = np.array([[0.0, 1.0, 2.0], [0.0, 0.0, 0.0]])
    d = np.array([[0.0, -np.inf, 5.0]])
    r = verify_request(t, d, [1], 1.0, np.array([0.999]), np.array([0.5, 0.5]))
    assert r["accept_len"] == 1 and r["flags"] & 1
    t2 = np.array([[0.0, -np.inf, 2.0], [0.0, 0.0, 0.0]])
    r2 = verify_request(t2, d, [1], 1.0, np.array([0.0]), np.array([0.5, 0.5]))
    assert r2["accept_len"] == 0


def test_identical_rows_accept_everything():
    rng = np.random.default_rng(3)
    t = rng.normal(size=(5, 40))
    u_acc, u_res = request_uniforms(5, 1, 0, 4)
    r = verify_request(t, t[:4].copy(), [3, 1, 4, 1], 1.3, u_acc, u_res)
    assert r["accept_len"] == 4 and r["p"] == r["q"]


def test_zero_kept_positions_is_a_plain_target_draw():
    rng = np.random.default_rng(4)
    t = rng.normal(size=(1, 30))
    counts = np.zeros(30)
    for s in range(4000):
        _, u_res = request_uniforms(s, 0, 0, 0)
        r = verify_request(t, np.zeros((0, 30)), [], 1.0, np.zeros(0), u_res)
        assert r["accept_len"] == 0
        counts[r["tokens"][0]] += 1
    from scipy.stats import chisquare
    assert chisquare(counts, sp_softmax(t[0]) * 4000).pvalue > 1e-4


def test_near_boundary_flag():
    t = np.log(np.array([[0.3, 0.7], [0.5, 0.5]]))
    d = np.log(np.array([[0.6, 0.4]]))
    # p/q at token 0 = 0.5 exactly; u = 0.5 + 1e-9 sits on the boundary
    r = verify_request(t, d, [0], 1.0, np.array([0.5 + 1e-9]), np.array([0.1, 0.1]))
    assert r["near"] == (NEAR_ACCEPT, 0)


# Near-boundary inverse-CDF picks.  The rows below have cumulative draw weights known in closed
# form, so u' can be placed a chosen distance from one bin edge.  A pick is flagged when
# u' * Z lies within 1e-6 * Z of either edge of the picked bin (the same band, relative to
# the accept test's 1e-6, that the design notes state for the draw).

def _pick_case(t, d, x, u_acc, u_res):
    return verify_request(np.log(np.asarray(t, float)), np.log(np.asarray(d, float)), x, 1.0,
                          np.asarray(u_acc, float), np.asarray(u_res, float))


@pytest.mark.parametrize("delta,flagged", [(1e-8, True), (5e-7, True), (5e-6, False), (2e-5, False)])
@pytest.mark.parametrize("side", [+1, -1])
def test_near_pick_band_bonus_draw(delta, flagged, side):
    """Bonus draw (every drafted token accepted), Z = 1: bonus row p = (.1, .2, .3, .4) has the
    inner edge c[1] = 0.3.  u' = 0.3 + delta picks entry 2 with the edge below it (c[y-1]);
    u' = 0.3 - delta picks entry 1 with the edge above it (c[y])."""
    t = [[0.4, 0.3, 0.2, 0.1], [0.1, 0.2, 0.3, 0.4]]
    r = _pick_case(t, [t[0]], [0], [0.5], [0.0, 0.3 + side * delta])
    assert r["accept_len"] == 1
    assert r["tokens"] == [0, 2 if side > 0 else 1]
    assert r["near"] == ((NEAR_PICK, 1) if flagged else None)


@pytest.mark.parametrize("dist,flagged", [(1e-8, True), (1e-7, True), (5e-7, False), (5e-6, False)])
@pytest.mark.parametrize("side", [+1, -1])
def test_near_pick_band_residual_draw(dist, flagged, side):
    """Residual draw after a rejection, Z = 0.2: max(0, p - q) = (0, .1, .1, 0) has the inner
    edge c[1] = 0.1.  The band is 1e-6 * Z = 2e-7 wide here, so an absolute distance of
    5e-7 (inside 1e-6, outside 1e-6 * Z) must not be flagged: the band scales with Z."""
    p = [0.1, 0.3, 0.2, 0.4]
    q = [0.3, 0.2, 0.1, 0.4]
    Z = 0.2
    r = _pick_case([p, [0.25] * 4], [q], [0], [0.9], [(0.1 + side * dist) / Z, 0.0])
    assert r["accept_len"] == 0                       # 0.9 * 0.3 >= 0.1: position 0 rejects
    assert r["tokens"] == [2 if side > 0 else 1]
    assert r["near"] == ((NEAR_PICK, 0) if flagged else None)


def test_near_pick_band_first_and_last_entries():
    """Edges at the ends of the vocabulary: the first entry has no edge below it (c[-1] is not
    consulted), and a threshold just under the total mass picks the last entry."""
    t = [[0.4, 0.3, 0.2, 0.1], [0.1, 0.2, 0.3, 0.4]]
    r = _pick_case(t, [t[0]], [0], [0.5], [0.0, 5e-9])        # u' Z close to c[-1] = 0 only
    assert r["tokens"] == [0, 0] and r["near"] is None
    r = _pick_case(t, [t[0]], [0], [0.5], [0.0, 1.0 - 5e-9])  # u' Z close to c[V-1] = Z
    assert r["tokens"] == [0, 3] and r["near"] == (NEAR_PICK, 1)
    r = _pick_case(t, [t[0]], [0], [0.5], [0.0, 0.1 - 5e-9])  # just below c[0]
    assert r["tokens"] == [0, 0] and r["near"] == (NEAR_PICK, 1)


def test_near_accept_takes_precedence_and_only_the_first_is_reported():
    """The first near-boundary decision of a request is the one reported: a near accept test at
    position 0 hides a near pick later in the same request."""
    t = [[0.3, 0.7], [0.5, 0.5]]
    d = [[0.6, 0.4]]
    # residual (0, 0.3): u' = 1e-9 puts u' Z next to the edge c[0] = 0 of the picked entry 1
    r = _pick_case(t, d, [0], [0.9], [1e-9, 0.0])
    assert r["accept_len"] == 0 and r["tokens"] == [1] and r["near"] == (NEAR_PICK, 0)
    r = _pick_case(t, d, [0], [0.5 + 1e-9], [1e-9, 0.0])   # p/q = 0.5: the accept test is near too
    assert r["accept_len"] == 0 and r["near"] == (NEAR_ACCEPT, 0)


def test_near_pick_rate_matches_the_band_width():
    """On flat rows (V = 20000, sigma = 1, T = 1) nearly every entry weighs more than 2e-6, so the
    band's measure, sum_v min(r_v / Z, 2e-6), grows in proportion to its width (about 4% of the
    draws here).  Over 3000 uniform pairs the oracle's flag count must match that measure,
    computed from scipy's softmax (rejections draw from max(0, p - q), acceptances from the bonus
    row): a band twice as wide, or half as wide, fails."""
    rng = np.random.default_rng(17)
    V = 20000
    t = rng.normal(0, 1, size=(2, V))
    d = t[:1] + rng.normal(0, 0.7, size=(1, V))
    x = int(np.argmax(d[0] + rng.gumbel(size=V)))
    P0, Q0, P1 = sp_softmax(t[0]), sp_softmax(d[0]), sp_softmax(t[1])
    alpha = min(1.0, P0[x] / Q0[x])
    r = np.maximum(0.0, P0 - Q0)
    band = lambda w: float(np.minimum(w / w.sum(), 2e-6).sum())
    n = 3000
    lam = n * ((1.0 - alpha) * band(r) + alpha * band(P1))
    u = rng.random((n, 2))
    hits = sum(verify_request(t, d, [x], 1.0, u[j, :1], np.array([u[j, 1], u[j, 1]]))["near"] is not None
               for j in range(n))
    assert lam > 60                                   # enough expected flags to tell widths apart
    assert abs(hits - lam) < 4.5 * np.sqrt(lam), (hits, lam)


def test_batch_matches_per_request_and_padding():
    b = W.small("c5", seed=3)
    res = verify_batch(b.target, b.t_offsets, b.draft, b.d_offsets, b.tokens, b.keep_len,
                       b.temperature, b.seed, b.round, b.request_ids, b.dtype, b.Kmax)
    for i in range(b.B):
        n = int(b.keep_len[i])
        a = res["accept_len"][i]
        assert 0 <= a <= n
        assert np.all(res["tokens"][i, a + 1:] == -1)
        assert np.all(res["tokens"][i, : a + 1] >= 0)
        assert np.all(np.isnan(res["p"][i, n:]))
        if b.temperature[i] == 0:
            g = _first_max(decode_rows(b.target[b.t_offsets[i] + a], b.dtype))
            assert res["tokens"][i, a] == g


# ------------------------------------------------------------------ printed numbers

def test_mal_identity_printed_values():
    with open(os.path.join(GOLDEN, "mal_identity.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        D = c["D"]
        n = 1000
        total = int(round(c["mean_acceptance"] * D * n))
        lens = np.zeros(n, int)
        for j in range(total):          # spread `total` accepted positions over n rounds
            lens[j % n] += 1
        assert lens.max() <= D
        assert abs(mean_acceptance(lens, [D] * n) - c["mean_acceptance"]) < 1e-12
        assert round(mean_accepted_length(lens), 2) == pytest.approx(c["MAL_printed"])


def test_draw_never_emits_a_zero_probability_token():
    """u' = 0 with masked (-inf) leading tokens: the inverse-CDF draw must skip zero mass,
    both for the bonus row and for a residual whose leading entries are zero."""
    t = np.array([[-np.inf, -np.inf, 0.0, 1.0], [-np.inf, -np.inf, 0.5, 0.0]])
    d = np.array([[5.0, 5.0, -3.0, 1.0]])
    for u_acc in (np.array([0.0]), np.array([0.9999])):     # accept (bonus) / reject (residual)
        r = verify_request(t, d, [3], 1.0, u_acc, np.array([0.0, 0.0]))
        y = r["tokens"][-1]
        assert y >= 2, r
