"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded
inputs.  Bit-exact tokens, accepted lengths and schedules (up to decisions the oracle marks as
within 1e-6 of a boundary), probabilities within 1e-5."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_74_gb300 as sv
from oracle.schedule import dcut_schedule
from oracle.verify import verify_batch, decode_rows
from synth import workloads as W
from svtest import dev_rows, i32, f32, run_ragged, oracle, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    sv.lib()


def _status(ws):
    st, bits = sv.sv_query_status(ws)
    return bits


# ------------------------------------------------------------------------ greedy (T = 0)

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_c1_greedy_fused_draft_argmax(seed):
    b = W.c1_greedy(seed)                        # B=4, K=3, V=32000 bf16, x_k = argmax(draft_k)
    K = b.Kmax
    ws = sv.workspace(sv.SV_OP_VERIFY, b.B, K, b.V, sv.SV_BF16)
    tok, alen = sv.verify_greedy(dev_rows(b.target, "bf16"), K, draft=dev_rows(b.draft, "bf16"), ws=ws)
    orc = oracle(b)
    compare(orc, tok.cpu().numpy(), alen.cpu().numpy())
    assert _status(ws) == 0


def test_greedy_given_tokens_every_rejection_point():
    b = W.c1_greedy(7, B=64, K=5, V=4099)         # ragged vocabulary tail (4099 = 512*8 + 3)
    t = decode_rows(b.target, "bf16").reshape(b.B, b.Kmax + 1, b.V)
    g = np.argmax(t, axis=-1).astype(np.int32)
    tokens = g[:, : b.Kmax].copy()
    rng = np.random.default_rng(0)
    for i in range(b.B):                          # request i rejects at position i % (K+1) (K = none)
        k = i % (b.Kmax + 1)
        if k < b.Kmax:
            tokens[i, k] = (tokens[i, k] + 1 + rng.integers(0, b.V - 1)) % b.V
    b.tokens = tokens
    tok, alen = sv.verify_greedy(dev_rows(b.target, "bf16"), b.Kmax, draft_tokens=i32(tokens))
    orc = oracle(b)
    compare(orc, tok.cpu().numpy(), alen.cpu().numpy())
    assert sorted(set(alen.cpu().numpy().tolist())) == list(range(b.Kmax + 1))


def test_greedy_ties_break_to_lowest_index():
    B, K, V = 8, 2, 1000
    rng = np.random.default_rng(3)
    x = rng.integers(-3, 3, size=(B * (K + 1), V)).astype(np.float32)    # many exact ties
    x[:, 900:] = 3.0                                                      # a tied maximum block late
    x[::2, 17] = 3.0                                                      # earlier tie in half the rows
    tgt = torch.from_numpy(x).cuda()
    tokens = np.full((B, K), 17, np.int32)
    tok, alen = sv.verify_greedy(tgt, K, draft_tokens=i32(tokens))
    b = W.VerifyBatch("ties", "f32", B, K, V, x, np.arange(B + 1, dtype=np.int32) * (K + 1), None, None, tokens,
                      np.full(B, K, np.int32), np.zeros(B, np.float32), 0, 0, np.arange(B, dtype=np.int32))
    compare(oracle(b), tok.cpu().numpy(), alen.cpu().numpy(), batch=b)


# ------------------------------------------------------------------------ sampled verification

@pytest.mark.parametrize("name,seed", [("c2", 0), ("c2", 1), ("c3", 0), ("c3", 5)])
def test_sample_small(name, seed):
    b = W.small(name, seed)
    ws = sv.workspace(sv.SV_OP_VERIFY, b.B, b.Kmax, b.V, sv.SV_BF16 if b.dtype == "bf16" else sv.SV_F32)
    tok, alen, p, q, fl = sv.verify_sample(dev_rows(b.target, b.dtype), dev_rows(b.draft, b.dtype), i32(b.tokens),
                                           f32(b.temperature), b.Kmax, seed=b.seed, round_=b.round,
                                           request_ids=i32(b.request_ids), ws=ws)
    torch.cuda.synchronize()
    compare(oracle(b), tok.cpu().numpy(), alen.cpu().numpy(), p.cpu().numpy(), q.cpu().numpy(), b.keep_len, batch=b)
    assert _status(ws) == 0


@pytest.mark.parametrize("make", [lambda: W.c3_dfly(21, B=3, K=16, V=70001),     # 33 rows x 18 chunks
                                  lambda: W.c2_mtp(22, B=4, K=12, V=90001)])      # 25 rows x 11 chunks
def test_sample_long_requests_separate_draw_weights(make):
    """Long requests (33 rows x 18 chunks, 25 rows x 11 chunks): each request's stream spans many
    units, and its draw spans many chunks with a ragged last chunk."""
    b = make()
    tok, alen, p, q, fl = sv.verify_sample(dev_rows(b.target, b.dtype), dev_rows(b.draft, b.dtype), i32(b.tokens),
                                           f32(b.temperature), b.Kmax, seed=b.seed, round_=b.round,
                                           request_ids=i32(b.request_ids))
    torch.cuda.synchronize()
    compare(oracle(b), tok.cpu().numpy(), alen.cpu().numpy(), p.cpu().numpy(), q.cpu().numpy(), b.keep_len, batch=b)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_ragged_mixed_small(seed):
    b = W.small("c5", seed)                      # mixed K in {3,16}, T in {0, 0.6, 1}, packed rows
    out = run_ragged(b)
    compare(oracle(b), out[0], out[1], out[2], out[3], b.keep_len, batch=b)


def test_many_rounds_and_workspace_reuse():
    ws = None
    for rnd in range(6):
        b = W.c5_mixed(seed=11, rnd=rnd, B=8, V=5003)
        if ws is None:
            ws = sv.workspace(sv.SV_OP_VERIFY, b.B, b.Kmax, b.V, sv.SV_BF16)
        out = run_ragged(b, ws=ws)
        compare(oracle(b), out[0], out[1], out[2], out[3], b.keep_len, batch=b)
    assert _status(ws) == 0


def test_one_workspace_across_call_shapes():
    """Calls of different sizes, dtypes and entry points share one workspace: its completion
    counters return to zero after every call, wherever the layout puts the other regions."""
    cases = [W.small("c3", 2), W.c3_dfly(21, B=3, K=16, V=70001), W.small("c5", 9), W.c1_greedy(4),
             W.small("c2", 6)]
    need = max(sv.sv_workspace_size(sv.SV_OP_VERIFY, b.B, b.Kmax, b.V,
                                    sv.SV_BF16 if b.dtype == "bf16" else sv.SV_F32) for b in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        for b in cases:
            if b.name.startswith("c5"):
                out = run_ragged(b, ws=ws)
                compare(oracle(b), out[0], out[1], out[2], out[3], b.keep_len, batch=b)
            elif not np.any(b.temperature > 0):
                tok, alen = sv.verify_greedy(dev_rows(b.target, b.dtype), b.Kmax, draft=dev_rows(b.draft, b.dtype),
                                             ws=ws)
                compare(oracle(b), tok.cpu().numpy(), alen.cpu().numpy(), batch=b)
            else:
                tok, alen, p, q, fl = sv.verify_sample(dev_rows(b.target, b.dtype), dev_rows(b.draft, b.dtype),
                                                       i32(b.tokens), f32(b.temperature), b.Kmax, seed=b.seed,
                                                       round_=b.round, request_ids=i32(b.request_ids), ws=ws)
                compare(oracle(b), tok.cpu().numpy(), alen.cpu().numpy(), p.cpu().numpy(), q.cpu().numpy(),
                        b.keep_len, batch=b)
    assert _status(ws) == 0


# ------------------------------------------------------------------------ D-cut scheduling

@pytest.mark.parametrize("seed", range(6))
def test_schedule_bit_exact(seed):
    s = W.c4_alpha(seed)
    alpha = f32(s.alpha)
    for objective, ratios, budget in ((sv.SV_OBJ_THROUGHPUT, None, 384), (sv.SV_OBJ_NET, None, 384),
                                      (sv.SV_OBJ_THROUGHPUT, (0.1, 0.3, 0.6, 0.9, 1.0), 0),
                                      (sv.SV_OBJ_NET, (0.2, 0.4), 700)):
        keep, offs, K, U = sv.schedule_depth(alpha, s.cost_a, s.cost_b, budget, ratios=ratios, objective=objective)
        torch.cuda.synchronize()
        o = dcut_schedule(s.alpha, None, s.cost_a, s.cost_b, budget,
                          ratios=ratios if ratios else (0.25, 0.5, 0.75, 1.0),
                          objective="net" if objective == sv.SV_OBJ_NET else "throughput")
        assert int(K.item()) == o["K"]
        assert int(U.item()) == o["U_q48"]
        assert np.array_equal(keep.cpu().numpy(), o["keep_len"])
        assert np.array_equal(offs.cpu().numpy(), np.concatenate([[0], np.cumsum(o["keep_len"] + 1)]))


def test_schedule_ragged_draft_len_and_ties():
    rng = np.random.default_rng(9)
    B, D = 37, 20
    alpha = rng.choice(np.array([0.0, 0.25, 0.5, 0.5, 0.75, 1.0], np.float32), size=(B, D))
    dl = rng.integers(0, D + 1, B).astype(np.int32)
    for budget in (0, B, 2 * B, 300):
        keep, offs, K, U = sv.schedule_depth(f32(alpha), 0.5, 0.01, budget, draft_len=i32(dl))
        o = dcut_schedule(alpha, dl, 0.5, 0.01, budget)
        assert int(K.item()) == o["K"] and int(U.item()) == o["U_q48"]
        assert np.array_equal(keep.cpu().numpy(), o["keep_len"])


def test_schedule_large_batch_limits():
    rng = np.random.default_rng(1)
    B, D = 1024, 16                               # 16384 slots: the largest sort
    alpha = rng.beta(5, 2, (B, D)).astype(np.float32)
    keep, offs, K, U = sv.schedule_depth(f32(alpha), 1.0, 0.05, 0)
    o = dcut_schedule(alpha, None, 1.0, 0.05, 0)
    assert int(K.item()) == o["K"] and int(U.item()) == o["U_q48"]
    assert np.array_equal(keep.cpu().numpy(), o["keep_len"])


def test_schedule_many_requests_per_thread_and_no_drafts():
    rng = np.random.default_rng(4)
    B, D = 3000, 5                                # 15000 slots, several requests per thread
    alpha = rng.beta(4, 2, (B, D)).astype(np.float32)
    dl = rng.integers(0, D + 1, B).astype(np.int32)
    for budget, draft_len in ((0, None), (4000, dl)):
        keep, offs, K, U = sv.schedule_depth(f32(alpha), 1.0, 0.02, budget, draft_len=None if draft_len is None
                                             else i32(draft_len))
        o = dcut_schedule(alpha, draft_len, 1.0, 0.02, budget)
        assert int(K.item()) == o["K"] and int(U.item()) == o["U_q48"]
        assert np.array_equal(keep.cpu().numpy(), o["keep_len"])
        assert np.array_equal(offs.cpu().numpy(), np.concatenate([[0], np.cumsum(o["keep_len"] + 1)]))
    a0 = torch.zeros((8, 0), dtype=torch.float32, device="cuda")   # Dmax = 0: roots only
    keep, offs, K, U = sv.schedule_depth(a0, 1.0, 0.02, 0)
    assert int(K.item()) == 8 and int(U.item()) == 8 << 48
    assert keep.cpu().numpy().tolist() == [0] * 8


@pytest.mark.parametrize("B,D", [(1, 7), (2, 5), (3, 4), (5, 16), (33, 7), (37, 20), (128, 16), (683, 3), (512, 16)])
def test_schedule_run_merge_shapes(B, D):
    """Batch shapes around the ranking's cases: one run, odd run counts (a run without a partner
    at some merge level), the largest merged size (128 x 16 = 2048 slots), the first size ranked
    by the bitonic sort (683 x 3 = 2049 slots) and a larger one; confidences with many ties."""
    rng = np.random.default_rng(B * 100 + D)
    ties = rng.choice(np.array([0.0, 0.5, 0.5, 0.9, 1.0], np.float32), size=(B, D))
    alpha = np.where(rng.random((B, D)) < 0.5, ties, rng.beta(6, 2, (B, D)).astype(np.float32)).astype(np.float32)
    dl = rng.integers(0, D + 1, B).astype(np.int32)
    for draft_len, budget in ((None, 0), (dl, max(B, (B * D) // 3))):
        keep, offs, K, U = sv.schedule_depth(f32(alpha), 0.8, 0.03, budget,
                                             draft_len=None if draft_len is None else i32(draft_len))
        o = dcut_schedule(alpha, draft_len, 0.8, 0.03, budget)
        assert int(K.item()) == o["K"] and int(U.item()) == o["U_q48"]
        assert np.array_equal(keep.cpu().numpy(), o["keep_len"])
        assert np.array_equal(offs.cpu().numpy(), np.concatenate([[0], np.cumsum(o["keep_len"] + 1)]))


def test_schedule_invalid_confidences_and_lengths():
    alpha = np.full((6, 4), 0.5, np.float32)
    for bad_alpha, dl, bit in ((1.5, None, 1 << 5), (np.nan, None, 1 << 5), (None, [1, 2, 5, 0, 4, 4], 1 << 6)):
        a = alpha.copy()
        if bad_alpha is not None:
            a[3, 1] = bad_alpha
        ws = sv.workspace(sv.SV_OP_SCHEDULE, 6, 4, 1, sv.SV_F32)
        keep, offs, K, U = sv.schedule_depth(f32(a), 1.0, 0.02, 0, draft_len=None if dl is None
                                             else i32(np.array(dl, np.int32)), ws=ws)
        torch.cuda.synchronize()
        assert int(K.item()) == -1 and int(U.item()) == -1
        assert keep.cpu().numpy().tolist() == [0] * 6
        assert offs.cpu().numpy().tolist() == list(range(7))
        assert _status(ws) & bit


def test_schedule_then_ragged_verify_on_device():
    """D-cut picks the kept prefixes on the device; the ragged verify consumes them without a
    host round trip (Figure 3 panels 3-4 of the D-cut section)."""
    s = W.c4_alpha(seed=2, B=16, D=16)
    keep_d, offs_d, K_d, U_d = sv.schedule_depth(f32(s.alpha), s.cost_a, s.cost_b, 96)
    o = dcut_schedule(s.alpha, None, s.cost_a, s.cost_b, 96)
    b = W.c4_verify(s, o["keep_len"], seed=2, V=7001)
    out = sv.verify_ragged(dev_rows(b.target, "bf16"), i32(b.t_offsets), dev_rows(b.draft, "bf16"), i32(b.d_offsets),
                           i32(b.tokens), keep_d, f32(b.temperature), b.Kmax, seed=b.seed, round_=b.round)
    torch.cuda.synchronize()
    out = [x.cpu().numpy() for x in out]
    compare(oracle(b), out[0], out[1], out[2], out[3], b.keep_len, batch=b)


# ------------------------------------------------------------------------ D-cut with a latency table

def _random_table(rng, lo, hi, n):
    Ks = sorted(set(int(v) for v in rng.integers(lo, hi + 1, n)))
    return Ks, [float(v) for v in rng.uniform(0.2, 50.0, len(Ks))]


def _check_table(alpha, draft_len, budget, table, ratios=None, objective=sv.SV_OBJ_THROUGHPUT):
    keep, offs, K, U = sv.schedule_depth(f32(alpha), 0.0, 0.0, budget, ratios=ratios, objective=objective,
                                         draft_len=None if draft_len is None else i32(draft_len),
                                         cost_table=table)
    torch.cuda.synchronize()
    o = dcut_schedule(alpha, draft_len, 0.0, 0.0, budget, ratios=ratios if ratios else (0.25, 0.5, 0.75, 1.0),
                      objective="net" if objective == sv.SV_OBJ_NET else "throughput", cost_table=table)
    assert int(K.item()) == o["K"] and int(U.item()) == o["U_q48"]
    assert np.array_equal(keep.cpu().numpy(), o["keep_len"])
    assert np.array_equal(offs.cpu().numpy(), np.concatenate([[0], np.cumsum(o["keep_len"] + 1)]))
    return o


@pytest.mark.parametrize("seed", range(6))
def test_schedule_table_bit_exact(seed):
    """Random latency tables on the D-cut batch (64 x 16): 1 to 32 knots inside, around and
    outside the candidate range, knots exactly at the candidates, both objectives."""
    s = W.c4_alpha(seed)
    rng = np.random.default_rng(500 + seed)
    N = 64 * 17
    tables = [_random_table(rng, 64, N, n) for n in (1, 2, 5, 32)]
    tables.append(_random_table(rng, 1, 63, 4))              # every candidate above the last knot
    tables.append(_random_table(rng, N + 1, 4 * N, 4))       # every candidate below the first knot
    cands = [272, 384]
    tables.append((cands, [3.0, 4.0]))                       # knots at the candidates
    tables.append(([272, 300, 301], [10.0, 10.0, 1e6]))      # a latency cliff past 300 tokens
    for table in tables:
        for objective in (sv.SV_OBJ_THROUGHPUT, sv.SV_OBJ_NET):
            for ratios, budget in ((None, 384), ((0.1, 0.3, 0.6, 0.9, 1.0), 0)):
                _check_table(s.alpha, None, budget, table, ratios, objective)
    o = _check_table(s.alpha, None, 384, ([272, 300, 301], [10.0, 10.0, 1e6]))
    assert o["K"] == 272


def test_schedule_table_ragged_shapes():
    for B, D in ((1, 7), (37, 20), (128, 16), (683, 3)):
        rng = np.random.default_rng(B + D)
        alpha = rng.beta(6, 2, (B, D)).astype(np.float32)
        dl = rng.integers(0, D + 1, B).astype(np.int32)
        N = int(np.sum(dl + 1))
        for draft_len, budget in ((None, 0), (dl, max(B, N // 2))):
            _check_table(alpha, draft_len, budget, _random_table(rng, 1, B * (D + 1), 9))


def test_schedule_table_profiled_from_ragged_verify():
    """Figure 3 panel 2 of the D-cut section: profile the latency table once, on a (batch size
    x keep ratio) grid, by timing a verify step; then every step schedules with it.  The
    profiled step here is the ragged verification itself (no target model), and the parity
    check holds for whatever the timings come out as."""
    from speculative_decoding_verification_74_gb300.cost_table import profile_cost_table
    D, Bmax, V = 16, 64, 32000
    s = W.c4_alpha(seed=11, B=Bmax, D=D)
    b = W.c4_verify(s, np.full(Bmax, D, np.int32), seed=11, V=V)
    target, draft = dev_rows(b.target, "bf16"), dev_rows(b.draft, "bf16")
    t_off, d_off, toks, temp = i32(b.t_offsets), i32(b.d_offsets), i32(b.tokens), f32(b.temperature)
    ws = sv.workspace(sv.SV_OP_VERIFY, Bmax, D, V, sv.SV_BF16)

    def step(nb, K):
        extra = K - nb                            # drafted positions spread evenly over nb requests
        keep = np.array([min(D, extra // nb + (1 if i < extra % nb else 0)) for i in range(nb)], np.int32)
        sv.verify_ragged(target, t_off[: nb + 1], draft, d_off[: nb + 1], toks[:nb], i32(keep), temp[:nb], D,
                         seed=b.seed, round_=b.round, ws=ws)

    Ks, cs = profile_cost_table(step, [16, 32, 64], D, reps=5, warmup=2)
    assert Ks == sorted(set(Ks)) and all(c > 0 for c in cs) and len(Ks) <= 12
    assert _status(ws) == 0
    for budget in (0, 384):
        _check_table(s.alpha, None, budget, (Ks, cs))


# ------------------------------------------------------------------------ edge cases

def test_zero_drafted_positions_and_zero_keep():
    b = W.c5_mixed(seed=4, rnd=0, B=8, V=3001)
    kl = b.keep_len.copy()
    kl[::2] = 0
    out = run_ragged(b, keep_len=kl)
    compare(oracle(b, keep_len=kl), out[0], out[1], out[2], out[3], kl, batch=b)
    b0 = W.make_batch("k0", ["chat"] * 5, [0] * 5, [1.0, 0.0, 0.6, 1.0, 1.0], 777, "bf16", 3, 0,
                      {"chat": (3.0, 1.0)})
    out = run_ragged(b0)
    compare(oracle(b0), out[0], out[1], out[2], out[3], b0.keep_len, batch=b0)
    assert np.all(out[1] == 0)


@pytest.mark.parametrize("V", [1, 5, 8, 17, 4097, 16385])
def test_vocab_sizes_and_tails(V):
    for dt in ("bf16", "f32"):
        b = W.make_batch("v", ["chat"] * 6, [3, 1, 0, 2, 3, 3], [1.0, 0.0, 0.6, 1.0, 0.0, 2.0], V, dt, V, 0,
                         {"chat": (3.0, 1.0)})
        out = run_ragged(b)
        compare(oracle(b), out[0], out[1], out[2], out[3], b.keep_len, batch=b)


def test_masked_logits():
    b = W.make_batch("mask", ["chat"] * 6, [3] * 6, [1.0, 0.6, 1.0, 0.0, 1.0, 1.0], 2048, "f32", 5, 0,
                     {"chat": (2.0, 1.0)})
    rng = np.random.default_rng(5)
    mask = rng.random(b.target.shape) < 0.5
    b.target[mask] = -np.inf
    dm = rng.random(b.draft.shape) < 0.5
    b.draft[dm] = -np.inf
    # drafted tokens must have q > 0: keep the drafted token's draft logit finite
    for i in range(b.B):
        for k in range(b.keep_len[i]):
            r = b.d_offsets[i] + k
            if not np.isfinite(b.draft[r, b.tokens[i, k]]):
                b.draft[r, b.tokens[i, k]] = 0.0
    out = run_ragged(b)
    orc = oracle(b)
    compare(orc, out[0], out[1], out[2], out[3], b.keep_len)
    for i in range(b.B):                          # never emits a token the target masks
        for j in range(out[1][i] + 1):
            assert np.isfinite(b.target[b.t_offsets[i] + j, out[0][i, j]])


def test_identical_rows_accept_all():
    b = W.c5_mixed(seed=8, rnd=0, B=6, V=2003)
    for i in range(b.B):
        n = b.keep_len[i]
        b.draft[b.d_offsets[i]: b.d_offsets[i] + n] = b.target[b.t_offsets[i]: b.t_offsets[i] + n]
    b.tokens = np.where(b.tokens >= 0, b.tokens, -1)
    # greedy requests need the target argmax as their drafted tokens for full acceptance
    for i in range(b.B):
        if b.temperature[i] == 0:
            t = decode_rows(b.target[b.t_offsets[i]: b.t_offsets[i] + b.keep_len[i]], "bf16")
            b.tokens[i, : b.keep_len[i]] = np.argmax(t, axis=1)
    out = run_ragged(b)
    assert np.array_equal(out[1], b.keep_len)
    compare(oracle(b), out[0], out[1], out[2], out[3], b.keep_len, batch=b)


def test_invalid_inputs_flag_and_poison():
    b = W.c5_mixed(seed=2, rnd=0, B=8, V=1999)
    ws = sv.workspace(sv.SV_OP_VERIFY, b.B, b.Kmax, b.V, sv.SV_BF16)
    tokens = b.tokens.copy()
    tokens[1, 0] = b.V + 5                        # out of range token
    kl = b.keep_len.copy()
    kl[2] = b.Kmax + 1                            # keep_len beyond Kmax
    temps = b.temperature.copy()
    temps[3] = np.nan                             # bad temperature
    temps[4] = -1.0
    out = sv.verify_ragged(dev_rows(b.target, "bf16"), i32(b.t_offsets), dev_rows(b.draft, "bf16"), i32(b.d_offsets),
                           i32(tokens), i32(kl), f32(temps), b.Kmax, seed=b.seed, ws=ws)
    st, bits = sv.sv_query_status(ws)
    assert st == sv.SV_ERR_DEVICE_INPUT
    assert bits & 1 and bits & 2 and bits & 4
    tok, alen = out[0].cpu().numpy(), out[1].cpu().numpy()
    flags = out[4].cpu().numpy()
    for i in (2, 3, 4):
        assert alen[i] == -1 and np.all(tok[i] == -1) and flags[i] & 4
    if tokens[1, 0] >= b.V:
        assert alen[1] == -1 and np.all(tok[1] == -1)
    ok = [0, 5, 6, 7]
    bb = W.c5_mixed(seed=2, rnd=0, B=8, V=1999)
    compare(oracle(bb), tok, alen, requests=ok, batch=bb)
    assert sv.sv_query_status(ws)[1] == 0           # cleared by the read


def test_ragged_row_counts_bound_every_request():
    """The packed arrays' row counts bound the last offsets: a request whose rows would run past
    t_rows (or d_rows) is flagged and reads nothing; the others verify as usual."""
    b = W.c5_mixed(seed=5, rnd=0, B=6, V=3001)
    tgt, dr = dev_rows(b.target, "bf16"), dev_rows(b.draft, "bf16")
    args = (i32(b.tokens), b.Kmax, i32(b.keep_len), f32(b.temperature), b.seed, b.round, None, sv.SV_BF16, b.B,
            b.Kmax, b.V)
    last = b.B - 1
    for short_t in (True, False):
        if not short_t and (b.temperature[last] == 0 or b.keep_len[last] == 0):
            continue                                  # the last request reads no draft row
        ws = sv.workspace(sv.SV_OP_VERIFY, b.B, b.Kmax, b.V, sv.SV_BF16)
        out = (torch.full((b.B, b.Kmax + 1), -7, dtype=torch.int32, device="cuda"),
               torch.full((b.B,), -7, dtype=torch.int32, device="cuda"),
               torch.empty((b.B, b.Kmax), device="cuda"), torch.empty((b.B, b.Kmax), device="cuda"),
               torch.zeros(b.B, dtype=torch.uint8, device="cuda"))
        t_rows = int(b.t_offsets[-1]) - (1 if short_t else 0)
        d_rows = int(b.d_offsets[-1]) - (0 if short_t else 1)
        sv.sv_verify_ragged(tgt, b.V, i32(b.t_offsets), t_rows, dr, b.V, i32(b.d_offsets), d_rows, *args, *out, ws)
        st, bits = sv.sv_query_status(ws)
        assert st == sv.SV_ERR_DEVICE_INPUT and bits == sv.SV_DEV_BAD_OFFSETS
        tok, alen = out[0].cpu().numpy(), out[1].cpu().numpy()
        assert alen[last] == -1 and np.all(tok[last] == -1) and out[4].cpu().numpy()[last] & sv.SV_FLAG_INVALID
        compare(oracle(b), tok, alen, requests=list(range(b.B - 1)), batch=b)


def test_sample_fixed_k_mixed_temperatures():
    """A fixed-K sampled call whose batch mixes greedy (T = 0) and sampled requests: the greedy
    ones follow the target argmax chain and do not need their draft rows."""
    b = W.make_batch("mixT", ["chat"] * 8, [3] * 8, [1.0, 0.0, 0.6, 0.0, 1.0, 2.0, 0.0, 0.6], 20011, "bf16", 31, 2,
                     {"chat": (3.0, 1.0)})
    tok, alen, p, q, fl = sv.verify_sample(dev_rows(b.target, "bf16"), dev_rows(b.draft, "bf16"), i32(b.tokens),
                                           f32(b.temperature), 3, seed=b.seed, round_=b.round,
                                           request_ids=i32(b.request_ids))
    torch.cuda.synchronize()
    compare(oracle(b), tok.cpu().numpy(), alen.cpu().numpy(), p.cpu().numpy(), q.cpu().numpy(), b.keep_len, batch=b)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_largest_draft_length(dt):
    """K = SV_MAX_DRAFT = 1023 drafted positions per request (2047 record rows per request)."""
    K = 1023
    b = W.make_batch("kmax", ["chat", "chat"], [K, K], [1.0, 0.0], 2053, dt, 41, 0, {"chat": (3.0, 0.05)})
    out = run_ragged(b)
    compare(oracle(b), out[0], out[1], out[2], out[3], b.keep_len, batch=b)
    tok, alen = sv.verify_greedy(dev_rows(b.target, dt)[: 2 * (K + 1)], K,
                                 draft_tokens=i32(np.ascontiguousarray(b.tokens)))
    bg = W.VerifyBatch("kmax-greedy", dt, 2, K, b.V, b.target, b.t_offsets, None, None, b.tokens, b.keep_len,
                       np.zeros(2, np.float32), 0, 0, np.arange(2, dtype=np.int32))
    compare(oracle(bg), tok.cpu().numpy(), alen.cpu().numpy(), batch=bg)


def test_largest_batch():
    """B = SV_MAX_BATCH = 4096 requests in one ragged call (the unit table at its largest)."""
    B = 4096
    kinds = ["chat"] * B
    rng = np.random.default_rng(9)
    Ks = [int(k) for k in rng.integers(0, 4, B)]
    temps = [float(t) for t in np.asarray([0.0, 0.6, 1.0], np.float32)[rng.integers(0, 3, B)]]
    b = W.make_batch("bmax", kinds, Ks, temps, 301, "bf16", 43, 0, {"chat": (3.0, 1.0)}, Kmax=3)
    out = run_ragged(b)
    compare(oracle(b), out[0], out[1], out[2], out[3], b.keep_len, batch=b)


def test_empty_batch_is_a_no_op():
    tok = torch.empty((0, 4), dtype=torch.int32, device="cuda")
    sv.sv_verify_greedy(None, 0, None, 0, None, sv.SV_BF16, 0, 3, 100, tok, tok, None)


# ------------------------------------------------------------------------ losslessness, sampled

def test_gpu_emissions_follow_the_target_distribution():
    """8192 verification rounds of one fixed (target, draft) row set on the GPU: the first
    emitted token follows p_0 and the mean accepted length matches sum_m prod_{k<m} beta_k."""
    from scipy.special import softmax
    from scipy.stats import chisquare
    from oracle.metrics import expected_accept_len
    V, K, T, B = 12, 3, 0.9, 2048
    rng = np.random.default_rng(21)
    t = rng.normal(0, 1.3, size=(K + 1, V)).astype(np.float32)
    d = (t[:K] + rng.normal(0, 0.9, size=(K, V))).astype(np.float32)
    tgt = np.tile(t, (B, 1))
    dr = np.tile(d, (B, 1))
    p0 = softmax(t[0].astype(np.float64) / T)
    betas = [float(np.sum(np.minimum(softmax(t[k].astype(np.float64) / T), softmax(d[k].astype(np.float64) / T))))
             for k in range(K)]
    first = np.zeros(V)
    lens = []
    for rnd in range(4):
        toks = np.stack([W.gumbel_max_tokens(np.random.default_rng([rnd, i]), d, T) for i in range(B)])
        out = sv.verify_sample(torch.from_numpy(tgt).cuda(), torch.from_numpy(dr).cuda(), i32(toks),
                               f32(np.full(B, T)), K, seed=77, round_=rnd)
        tok, alen = out[0].cpu().numpy(), out[1].cpu().numpy()
        first += np.bincount(tok[:, 0], minlength=V)
        lens += alen.tolist()
    n = len(lens)
    assert chisquare(first, p0 * n).pvalue > 1e-4
    lens = np.asarray(lens, float)
    assert abs(lens.mean() - expected_accept_len(betas)) < 4.5 * lens.std() / np.sqrt(n)


def test_draws_over_multi_chunk_pieces():
    """Enough (row, chunk) tasks that stream units span several chunks of a row; half the
    requests have draft = target (every drafted token accepted: bonus draws), half reject
    (residual draws)."""
    b = W.make_batch("pieces", ["chat"] * 12, [3] * 12, [1.0] * 12, 151936, "bf16", 42, 0, {"chat": (3.0, 1.0)})
    for i in range(0, b.B, 2):
        b.draft[b.d_offsets[i]: b.d_offsets[i] + 3] = b.target[b.t_offsets[i]: b.t_offsets[i] + 3]
    out = run_ragged(b)
    assert np.all(out[1][::2] == 3)
    compare(oracle(b), out[0], out[1], out[2], out[3], b.keep_len, batch=b)
    tok, alen, p, q, fl = sv.verify_sample(dev_rows(b.target, "bf16"), dev_rows(b.draft, "bf16"), i32(b.tokens),
                                           f32(b.temperature), 3, seed=b.seed, round_=b.round)
    torch.cuda.synchronize()
    compare(oracle(b), tok.cpu().numpy(), alen.cpu().numpy(), p.cpu().numpy(), q.cpu().numpy(), b.keep_len, batch=b)
