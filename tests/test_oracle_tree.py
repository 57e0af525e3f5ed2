"""Pins for the multi-candidate (tree) verification oracle (CPU only).

  * A chain (one child per node) is the chain oracle, decision for decision.
  * Losslessness, exactly: the children of every node are drafted independently from the node's
    draft distribution; integrating the oracle's own decisions over its uniforms (each decision is
    a threshold in its uniform, found by bisection) and over every drafted tree, the first L
    emitted tokens, completed by target draws, follow the target's law to 1e-9.
  * Greedy: brute force over every drafted tree on integer logits with ties.
  * The walk's closed form of the repeated residual (what the library's walk sums in each pass)
    equals the oracle's rule applied j times, in exact rational arithmetic.
"""
import itertools

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

from oracle.tree import verify_tree, children_of
from oracle.verify import verify_request, request_uniforms

# ------------------------------------------------------------------ the chain is a special case


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0, 1.6])
def test_a_chain_is_the_chain_oracle(T):
    for seed in range(40):
        rng = np.random.default_rng(seed)
        V, K = 30, int(rng.integers(0, 6))
        t = rng.normal(0, 2, size=(K + 1, V))
        d = t[:K] + rng.normal(0, 1, size=(K, V))
        tok = [int(x) for x in (np.argmax(d, axis=1) if T == 0 else rng.integers(0, V, K))]
        if T > 0:                                   # make some positions accept: draft the argmax of q
            for k in range(0, K, 2):
                tok[k] = int(np.argmax(d[k]))
        u_acc, u_res = request_uniforms(seed, 2, 1, K)
        a = verify_request(t, d if T > 0 else None, tok, T, u_acc, u_res)
        b = verify_tree([-1] + list(range(K)), [0] + tok, t, list(d) + [None], T, u_acc, u_res)
        assert b["tokens"] == a["tokens"] and b["accept_len"] == a["accept_len"]
        if T > 0:
            assert b["flags"] == a["flags"]
            # the chain oracle names positions; the tree oracle names nodes (child c = position c - 1)
            if a["near"] is None:
                assert b["near"] is None
            else:
                kind, pos = a["near"]
                assert b["near"] == (kind, pos + 1 if kind == 1 else pos)


# ------------------------------------------------------------------ losslessness, exactly

def _bisect(pred, iters=52):
    """Smallest u in [0, 1) where pred becomes True (pred monotone False -> True); 1 if never."""
    lo, hi = 0.0, 1.0
    if pred(0.0):
        return 0.0
    if not pred(np.nextafter(1.0, 0.0)):
        return 1.0
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if pred(mid):
            hi = mid
        else:
            lo = mid
    return hi


class _Tables:
    """Target and draft logits of the next token after any token path (fixed random tables)."""

    def __init__(self, V, seed):
        self.V, self.rng, self.t, self.d = V, np.random.default_rng(seed), {}, {}

    def target(self, path):
        if path not in self.t:
            self.t[path] = self.rng.normal(0, 1.2, self.V)
        return self.t[path]

    def draft(self, path):
        if path not in self.d:
            self.d[path] = self.target(path) + self.rng.normal(0, 1.0, self.V)
        return self.d[path]


def _emission_law(parent, token, tab, T, L):
    """Exact law of the first L tokens: the oracle's emission, then target draws."""
    N = len(parent)
    ch = children_of(parent)
    paths = [()] * N
    for c in range(1, N):
        paths[c] = paths[parent[c]] + (token[c],)
    t = [tab.target(paths[n]) for n in range(N)]
    d = [tab.draft(paths[n]) for n in range(N)]
    V = tab.V
    law = {}

    def run(u_acc, u_res):
        return verify_tree(parent, token, t, d, T, u_acc, u_res)

    def complete(seq, prob):
        if len(seq) >= L:
            key = tuple(seq[:L])
            law[key] = law.get(key, 0.0) + prob
            return
        p = sp_softmax(tab.target(tuple(seq)) / T)
        for v in range(V):
            if p[v] > 0:
                complete(seq + [v], prob * p[v])

    def draw_law(node, u_acc, prob):
        prev = 0.0
        for v in range(V):
            def above(u, v=v):
                ur = np.zeros(N)
                ur[node] = u
                return run(u_acc, ur)["tokens"][-1] > v
            b = 1.0 if v == V - 1 else _bisect(above)
            if b > prev:
                ur = np.zeros(N)
                ur[node] = 0.5 * (prev + b)
                res = run(u_acc, ur)
                assert res["tokens"][-1] == v
                complete(list(res["tokens"]), prob * (b - prev))
            prev = b

    def walk(node, u_acc, prob):
        if not ch[node]:
            draw_law(node, u_acc, prob)
            return
        remaining = prob
        u_acc = u_acc.copy()
        for c in ch[node]:
            def rejects(u, c=c):
                ua = u_acc.copy()
                ua[c - 1] = u
                return c not in run(ua, np.zeros(N))["path"]
            theta = _bisect(rejects)                  # child c is accepted iff its uniform < theta
            if theta > 0.0:
                ua = u_acc.copy()
                ua[c - 1] = 0.5 * theta
                walk(c, ua, remaining * theta)
            remaining *= 1.0 - theta
            if remaining == 0.0:
                return
            u_acc[c - 1] = 0.5 * (1.0 + theta)        # force the rejection, go on to the next child
        draw_law(node, u_acc, remaining)

    walk(0, np.zeros(max(N - 1, 1)), 1.0)
    return law


def _target_law(tab, T, L):
    law = {}

    def rec(seq, prob):
        if len(seq) == L:
            law[tuple(seq)] = prob
            return
        p = sp_softmax(tab.target(tuple(seq)) / T)
        for v in range(tab.V):
            rec(seq + [v], prob * p[v])
    rec([], 1.0)
    return law


SHAPES = {
    "two candidates": [-1, 0, 0],
    "three candidates": [-1, 0, 0, 0],
    "two chains of two": [-1, 0, 0, 1, 2],
}


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("V,T", [(2, 1.0), (3, 0.7)])
def test_lossless_exact_enumeration_over_drafted_trees(shape, V, T):
    parent = SHAPES[shape]
    N = len(parent)
    depth = [0] * N
    for c in range(1, N):
        depth[c] = depth[parent[c]] + 1
    L = max(depth) + 1
    tab = _Tables(V, seed=31 * V + N)
    total = {}
    # every drafted tree: each node's children drafted independently from its draft distribution
    for toks in itertools.product(range(V), repeat=N - 1):
        token = [0] + list(toks)
        w = 1.0
        path = [()] * N
        for c in range(1, N):
            path[c] = path[parent[c]] + (token[c],)
            w *= sp_softmax(tab.draft(path[parent[c]]) / T)[token[c]]
        for k, v in _emission_law(parent, token, tab, T, L).items():
            total[k] = total.get(k, 0.0) + w * v
    want = _target_law(tab, T, L)
    assert set(total) <= set(want)
    for k, v in want.items():
        assert abs(total.get(k, 0.0) - v) < 1e-9, (k, total.get(k, 0.0), v)


# ------------------------------------------------------------------ greedy

def test_greedy_brute_force_over_drafted_trees():
    rng = np.random.default_rng(4)
    V = 3
    parent = [-1, 0, 0, 1, 2, 2]
    N = len(parent)
    t = rng.integers(-2, 3, size=(N, V)).astype(np.float64)   # integer logits: many ties
    first_max = [int(np.flatnonzero(r == r.max()).min()) for r in t]
    ch = children_of(parent)
    for toks in itertools.product(range(V), repeat=N - 1):
        token = [0] + list(toks)
        res = verify_tree(parent, token, t, [None] * N, 0.0, np.zeros(N), np.zeros(N))
        # walk by hand: the first child holding the target argmax, else emit the argmax
        node, want = 0, []
        while True:
            nxt = next((c for c in ch[node] if token[c] == first_max[node]), None)
            if nxt is None:
                want.append(first_max[node])
                break
            want.append(token[nxt])
            node = nxt
        assert res["tokens"] == want
        assert res["accept_len"] == len(want) - 1


# ------------------------------------------------------ the repeated residual in closed form


def _iterated_residual(p, q, j):
    """The oracle's rule after j rejections at one node: p' <- norm(max(0, p' - q)), j times."""
    r = list(p)
    for _ in range(j):
        w = [max(0, a - b) for a, b in zip(r, q)]
        z = sum(w)
        if z == 0:
            return None
        r = [x / z for x in w]
    return r


@pytest.mark.parametrize("seed", range(6))
def test_repeated_residual_closed_form(seed):
    """After j rejections p' = max(0, p - a_j q) / N_j with a_0 = 0, N_0 = 1, a_{j+1} = a_j + N_j
    and N_{j+1} = sum_v max(0, p_v - a_{j+1} q_v): one pass over the node's rows per rejection.
    Checked exactly (fractions) on random rational distributions, for every j up to the first
    zero-mass residual."""
    from fractions import Fraction as F
    rng = np.random.default_rng(seed)
    V = int(rng.integers(3, 9))
    pw, qw = rng.integers(0, 20, V) + 1, rng.integers(0, 20, V)
    qw[rng.integers(1, V)] += 1
    if seed % 2 == 0:
        qw[0] = 0  # an entry q misses keeps the residual's mass above zero at every j
    p = [F(int(x), int(pw.sum())) for x in pw]
    q = [F(int(x), int(qw.sum())) for x in qw]
    a, N = F(0), F(1)
    checked = 0
    for j in range(8):
        it = _iterated_residual(p, q, j)
        if it is None:
            break
        closed = [max(F(0), pv - a * qv) / N for pv, qv in zip(p, q)]
        assert closed == it, (seed, j)
        checked += 1
        a_next = a + N
        N_next = sum(max(F(0), pv - a_next * qv) for pv, qv in zip(p, q))
        if N_next == 0:
            break
        a, N = a_next, N_next
    assert checked >= (8 if seed % 2 == 0 else 2)

