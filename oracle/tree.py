"""Multi-candidate (tree) verification, fp64 oracle.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The AngelSpec pages verify one drafted chain per request: the DFly block is one causal chain,
q(X_{t+1:t+B}) = prod_i q_i(x_{t+i} | x_{<=t}, x_{t+1:t+i-1}) (AngelSpec explainer, "DFly"), and
verification stays lossless (explainer, "D-cut").  Verifying several candidates per position
(a token tree) is not on the pages; this oracle takes the published rule of multi-step
speculative sampling (Miao et al., "SpecInfer: Accelerating Large Language Model Serving with
Tree-based Speculative Inference and Verification", ASPLOS 2024, section 4.2):

  At a node with target distribution p and children x_1..x_m drafted independently from the
  node's draft distribution q (with replacement), in order:
      p' = p
      for j = 1..m:
          accept x_j  <=>  u_j * q(x_j) < p'(x_j)        (u_j < min(1, p'(x_j) / q(x_j)))
          on a rejection: p' = norm(max(0, p' - q))
      an accepted child is emitted and verification continues at that child;
      if every child is rejected, y ~ p' is emitted and verification stops.
  At a node without children, y ~ p (the bonus draw) is emitted and verification stops.
  T == 0 (greedy): the first child equal to the target argmax is accepted; otherwise the
  target argmax is emitted and verification stops.

The draw is the same inverse CDF in vocabulary order as the chain oracle (first v whose
cumulative weight exceeds u' * Z).  A chain (every node with one child) reduces to the chain
oracle exactly: node k + 1 is drafted position k, its accept uniform is the chain's u_k, and the
draw at node a uses the chain's u'_a.

Tree layout (one request): nodes 0..N-1 in an order where every parent precedes its children;
parent[0] = -1 (the root: the verified context); token[c] is the drafted token of node c >= 1;
t[n] are the target logits of the next token after node n's path; d[n] the draft logits its
children were drafted from (rows of leaves are unused).  Children are tried in increasing node
order.  Uniforms: the accept test of child c uses u_acc[c - 1]; the draw at node n uses u_res[n].

Readings where the rule leaves a case open (same as the chain oracle): q(x) == 0 accepts iff
p'(x) > 0 (flag bit 0); a residual of zero mass draws from the current p' instead (flag bit 1).
"""
from __future__ import annotations

import numpy as np

from .verify import (softmax_T, decode_rows, request_uniforms, FLAG_Q_ZERO, FLAG_Z_ZERO, NEAR_ACCEPT, NEAR_PICK,
                     NEAR_TOL)


def children_of(parent) -> list[list[int]]:
    ch = [[] for _ in range(len(parent))]
    for c in range(1, len(parent)):
        ch[int(parent[c])].append(c)
    return ch


def _draw(r, u):
    """First v whose cumulative weight (index order) exceeds u * sum(r); the near-boundary test of
    the chain oracle on that pick."""
    c = np.cumsum(r)
    Z = c[-1]
    thr = u * Z
    y = int(np.searchsorted(c, thr, side="right"))
    if y >= len(r):
        y = int(np.nonzero(r > 0)[0][-1])
    near = abs(c[y] - thr) < NEAR_TOL * Z or (y > 0 and abs(c[y - 1] - thr) < NEAR_TOL * Z)
    return y, near


def verify_tree(parent, token, t, d, T, u_acc, u_res) -> dict:
    """Verify one request's drafted tree.  Returns the accepted node path (root excluded), the
    emitted tokens (accepted tokens, then the drawn or argmax token), accept_len, flags, and the
    first near-boundary decision ((NEAR_ACCEPT, child node) or (NEAR_PICK, node)) or None."""
    ch = children_of(parent)
    node, path, flags, near = 0, [], 0, None

    def out(y):
        return {"path": path, "tokens": [int(token[c]) for c in path] + [int(y)], "accept_len": len(path),
                "flags": flags, "near": near}

    while True:
        kids = ch[node]
        if T == 0.0:
            g = int(np.argmax(t[node]))
            nxt = next((c for c in kids if int(token[c]) == g), None)
            if nxt is None:
                return out(g)
            path.append(nxt)
            node = nxt
            continue
        P = softmax_T(t[node], T)
        if not kids:
            y, nr = _draw(P, u_res[node])
            if near is None and nr:
                near = (NEAR_PICK, node)
            return out(y)
        Q = softmax_T(d[node], T)
        Pr = P      # p' of the next test (normalised)
        r = P       # the weights a draw at this node would use
        accepted = None
        for c in kids:
            x = int(token[c])
            if Q[x] == 0.0:
                flags |= FLAG_Q_ZERO
            elif near is None and abs(u_acc[c - 1] - Pr[x] / Q[x]) < NEAR_TOL:
                near = (NEAR_ACCEPT, c)
            if u_acc[c - 1] * Q[x] < Pr[x]:
                accepted = c
                break
            res = np.maximum(0.0, Pr - Q)
            Z = res.sum()
            if Z > 0.0:
                r, Pr = res, res / Z
            else:
                flags |= FLAG_Z_ZERO
                r = Pr
        if accepted is None:
            y, nr = _draw(r, u_res[node])
            if near is None and nr:
                near = (NEAR_PICK, node)
            return out(y)
        path.append(accepted)
        node = accepted


def verify_tree_batch(target, draft, node_offsets, parent, tokens, temperature, seed, rnd, request_ids, dtype):
    """Verify a packed batch of trees (the library's layout: node c of request i is row
    node_offsets[i] + c of target and draft, and entry node_offsets[i] + c of parent and tokens),
    request by request.  Uniforms: the accept test of child c uses position c - 1, the draw at node
    n position n, as in the chain (request_uniforms with n = N - 1).  Returns one verify_tree
    result per request."""
    out = []
    for i in range(len(node_offsets) - 1):
        a, b = int(node_offsets[i]), int(node_offsets[i + 1])
        N = b - a
        T = float(np.float32(temperature[i]))
        t = list(decode_rows(target[a:b], dtype))
        d = list(decode_rows(draft[a:b], dtype)) if T > 0.0 else [None] * N
        rid = int(request_ids[i]) if request_ids is not None else i
        u_acc, u_res = request_uniforms(seed, rid, rnd, N - 1)
        out.append(verify_tree(np.asarray(parent[a:b]), np.asarray(tokens[a:b]), t, d, T, u_acc, u_res))
    return out
