"""Token-tree verification on the GPU (sv_verify_tree) against the fp64 tree oracle
(multi-step speculative sampling), request by request: accepted paths, emitted tokens and
accepted lengths bit-exact outside the near-boundary band."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_74_gb300 as sv
from synth.trees import make_tree_batch, TREE_SHAPES, t1_tree
from svtest import run_tree, oracle_tree, compare_tree, dev_rows, i32, f32

pytestmark = pytest.mark.gpu


def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_mixed_shapes_and_temperatures(dtype):
    _gpu()
    temps = [1.0, 0.7, 0.0, 1.5, 0.5, 1.0, 0.0, 1.2] * 3
    shapes = [TREE_SHAPES[i % len(TREE_SHAPES)] for i in range(len(temps))]
    b = make_tree_batch("mixed", shapes, temps, 20011, dtype, seed=5)  # several vocabulary chunks, ragged tail
    path, tok, alen, fl = run_tree(b)
    compare_tree(oracle_tree(b), path, tok, alen, b)
    assert np.all(fl & sv.SV_FLAG_INVALID == 0)


def test_wide_nodes_many_rejections():
    """Eight candidates per node and a far drafter: most children are rejected, so each node runs
    several residual passes (a_j accumulates) before its draw."""
    _gpu()
    shapes = [([8, 2], 20), ([6, 3, 1], 24), ([8], 9), ([5, 5], 31)] * 4
    b = make_tree_batch("wide", shapes, [1.0, 0.8, 1.3, 1.0] * 4, 9001, "bf16", seed=11, sigma_n=3.0)
    path, tok, alen, fl = run_tree(b)
    compare_tree(oracle_tree(b), path, tok, alen, b)


def test_greedy_trees_and_root_only():
    _gpu()
    shapes = [([3, 2, 1], 12), ([1] * 7, 8), ([], 1), ([4, 4], 21)] * 2
    temps = [0.0] * 4 + [1.0, 1.0, 1.0, 0.0]
    b = make_tree_batch("greedy", shapes, temps, 7777, "f32", seed=2, sigma_n=0.3)
    path, tok, alen, fl = run_tree(b)
    compare_tree(oracle_tree(b), path, tok, alen, b)
    assert alen[2] == 0 and path[2, 0] == -1 and tok[2, 1] == -1      # a root alone emits one token


def test_many_rounds_reuse_one_workspace():
    _gpu()
    shapes = [TREE_SHAPES[i % len(TREE_SHAPES)] for i in range(8)]
    ws = sv.workspace(sv.SV_OP_TREE, 8, 16, 4099, sv.SV_BF16)
    for rnd in range(4):
        b = make_tree_batch("rounds", shapes, [1.0] * 8, 4099, "bf16", seed=9, rnd=rnd)
        path, tok, alen, fl = run_tree(b, ws=ws)
        compare_tree(oracle_tree(b), path, tok, alen, b)
        assert sv.sv_query_status(ws) == (sv.SV_OK, 0)


def test_invalid_trees_are_flagged():
    _gpu()
    shapes = [TREE_SHAPES[0]] * 4
    b = make_tree_batch("bad", shapes, [1.0] * 4, 3001, "bf16", seed=1)
    o = b.node_offsets
    b.parent[o[1] + 5] = 9            # request 1: a parent after its child
    b.tokens[o[2] + 3] = b.V          # request 2: a token outside [0, V)
    ws = sv.workspace(sv.SV_OP_TREE, b.B, b.Nmax, b.V, sv.SV_BF16)
    path, tok, alen, fl = run_tree(b, ws=ws)
    st, bits = sv.sv_query_status(ws)
    assert st == sv.SV_ERR_DEVICE_INPUT and bits & sv.SV_DEV_BAD_PARENT and bits & sv.SV_DEV_BAD_TOKEN
    for i in (1, 2):
        assert alen[i] == -1 and fl[i] & sv.SV_FLAG_INVALID and np.all(path[i] == -1) and np.all(tok[i] == -1)
    orc = oracle_tree(b)
    compare_tree(orc, path, tok, alen, b, requests=[0, 3])


def test_fullsize_tree_workload_sample():
    """The tree workload at full size (64 requests of 16 nodes, V = 151936 bf16, T = 1): every
    request's path against the oracle."""
    _gpu()
    b = t1_tree(seed=0)
    path, tok, alen, fl = run_tree(b)
    compare_tree(oracle_tree(b), path, tok, alen, b)
