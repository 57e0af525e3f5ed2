"""Seeded token trees for multi-candidate verification (inputs only; no verification arithmetic).

A tree request has N nodes in breadth-first order (every parent precedes its children); node 0 is
the root, the verified context.  Shapes come from per-level branching factors: level-l nodes get
branch[l] children each, and the levels stop when the node budget is spent.  Per node the recipe
draws the target's next-token logits t[n] (chat rows, N(0, sigma_t)) and the drafter's logits
d[n] = t[n] + N(0, sigma_n); the children of node n are drafted independently from softmax(d[n] / T)
(Gumbel-max, with replacement) for a sampled request, or are the top-m entries of d[n] for a
greedy one.  Rows of every node are packed in node order: request i's node c is row
node_offsets[i] + c of both the target and the draft array (leaf draft rows are filler).

Every array is a pure function of (name, seed, round).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .workloads import (BF16, F32, _rng, _encode, _decode32, _name_key, chat_rows, gumbel_max_tokens)


@dataclass
class TreeBatch:
    """One tree-verification round in the packed layout the library takes.

    target, draft  [sum_i N_i, V] rows (uint16 bf16 bits or float32), node c of request i at row
                   node_offsets[i] + c
    node_offsets   [B + 1] int32
    parent         [sum_i N_i] int32 (root entries -1)
    tokens         [sum_i N_i] int32 drafted token of each node (root entries -1)
    temperature    [B] float32 (0 = greedy)
    """
    name: str
    dtype: str
    B: int
    Nmax: int
    V: int
    target: np.ndarray
    draft: np.ndarray
    node_offsets: np.ndarray
    parent: np.ndarray
    tokens: np.ndarray
    temperature: np.ndarray
    seed: int
    round: int
    request_ids: np.ndarray
    meta: dict = field(default_factory=dict)

    def nodes(self, i: int) -> int:
        return int(self.node_offsets[i + 1] - self.node_offsets[i])

    @property
    def keep_len(self) -> np.ndarray:
        """Drafted candidates per request (every node but the root)."""
        return (np.diff(self.node_offsets) - 1).astype(np.int32)


def tree_shape(branch: list[int], max_nodes: int) -> np.ndarray:
    """Parent array of a breadth-first tree: level-l nodes get branch[l] children each, until
    max_nodes nodes exist."""
    parent = [-1]
    level = [0]
    for b in branch:
        nxt = []
        for node in level:
            for _ in range(b):
                if len(parent) >= max_nodes:
                    break
                parent.append(node)
                nxt.append(len(parent) - 1)
        level = nxt
        if not level or len(parent) >= max_nodes:
            break
    return np.asarray(parent, np.int32)


def _top_m(d32_row: np.ndarray, m: int) -> np.ndarray:
    order = np.argsort(-d32_row, kind="stable")
    return order[:m].astype(np.int32)


def make_tree_batch(name: str, shapes: list[tuple[list[int], int]], temps: list[float], V: int, dtype: str,
                    seed: int, rnd: int = 0, sigma_t: float = 2.0, sigma_n: float = 1.0,
                    Nmax: int | None = None) -> TreeBatch:
    """shapes[i] = (branching factors per level, node budget) of request i."""
    B = len(shapes)
    rng = _rng(seed, rnd, _name_key(name))
    parents = [tree_shape(br, mx) for br, mx in shapes]
    offs = np.zeros(B + 1, np.int32)
    for i, par in enumerate(parents):
        offs[i + 1] = offs[i] + len(par)
    total = int(offs[-1])
    store = np.uint16 if dtype == BF16 else np.float32
    target = np.empty((total, V), store)
    draft = np.empty((total, V), store)
    parent = np.full(total, -1, np.int32)
    tokens = np.full(total, -1, np.int32)
    for i, par in enumerate(parents):
        N = len(par)
        t_enc = _encode(chat_rows(rng, N, V, sigma_t), dtype)
        t32 = _decode32(t_enc, dtype)
        d_enc = _encode(t32 + rng.standard_normal((N, V), dtype=np.float32) * np.float32(sigma_n), dtype)
        d32 = _decode32(d_enc, dtype)
        tok = np.full(N, -1, np.int32)
        for node in range(N):
            kids = np.nonzero(par == node)[0]
            if len(kids) == 0:
                continue
            if temps[i] > 0.0:
                tok[kids] = gumbel_max_tokens(rng, np.repeat(d32[node:node + 1], len(kids), axis=0), temps[i])
            else:
                tok[kids] = _top_m(d32[node], len(kids))
        a, b = offs[i], offs[i + 1]
        target[a:b], draft[a:b], parent[a:b], tokens[a:b] = t_enc, d_enc, par, tok
    nm = max(len(p) for p in parents) if Nmax is None else Nmax
    return TreeBatch(name=name, dtype=dtype, B=B, Nmax=nm, V=V, target=target, draft=draft, node_offsets=offs,
                     parent=parent, tokens=tokens, temperature=np.asarray(temps, np.float32), seed=seed,
                     round=rnd, request_ids=np.arange(B, dtype=np.int32))


# A DFly-style block of 8 verified as a tree: three candidates at the first position, two at the
# second, then chains; mixed with wider and deeper shapes.
TREE_SHAPES = [([3, 2, 1, 1, 1], 16), ([2, 2, 2, 1], 16), ([4, 1, 1, 1, 1, 1], 16), ([1] * 15, 16),
               ([2] * 4, 16), ([3, 3, 1], 16), ([1, 4, 1, 1], 16), ([5, 1, 1], 16)]


def t1_tree(seed: int = 0, B: int = 64, V: int = 151936, rnd: int = 0, dtype: str = BF16) -> TreeBatch:
    """Tree verification at T = 1: B requests of 16 nodes in eight shapes, chat rows."""
    shapes = [TREE_SHAPES[i % len(TREE_SHAPES)] for i in range(B)]
    return make_tree_batch("t1", shapes, [1.0] * B, V, dtype, seed, rnd)
