"""D-cut over a batch partitioned across ranks.

Verification is independent per request, so a data-parallel deployment splits the batch by
requests and each rank verifies its own.  The depth allocation is the one step that needs the
whole batch: D-cut ranks every drafted position of every request against every other and keeps
a global top-K, so the verify budget is shared by the batch, not set per request (AngelSpec
explainer, "D-cut: verification depth is a shared resource, not a per-request setting",
Figure 3 panels 3-4).  The exchange is one small all-gather of the drafter's confidences
(B_r x Dmax floats per rank, plus the draft lengths); every rank then runs the same schedule on
the concatenated batch and keeps its own requests' depths.  No logit crosses ranks.

The ranks may hold different numbers of requests.  Requests are concatenated in rank order, so
request j of rank r is request (sum of the earlier ranks' batch sizes) + j of the global batch,
and ties in the global ranking break on that global index.
"""
from __future__ import annotations

import torch


def gather_batch(alpha: torch.Tensor, draft_len: torch.Tensor | None, group=None):
    """All-gather every rank's confidences [B_r, Dmax] and draft lengths [B_r] (None: all Dmax).
    Returns (alpha_all [sum B_r, Dmax], draft_len_all [sum B_r], first request index of this
    rank, list of B_r)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    B, Dmax = alpha.shape
    dev = alpha.device
    sizes_t = torch.tensor([B, Dmax], dtype=torch.int64, device=dev)
    all_sizes = [torch.zeros_like(sizes_t) for _ in range(world)]
    dist.all_gather(all_sizes, sizes_t, group=group)
    sizes = [int(s[0].item()) for s in all_sizes]
    if any(int(s[1].item()) != Dmax for s in all_sizes):
        raise ValueError("every rank must pass the same Dmax")
    Bmax = max(sizes)
    if draft_len is None:
        draft_len = torch.full((B,), Dmax, dtype=torch.int32, device=dev)
    pad_a = torch.zeros((Bmax, Dmax), dtype=alpha.dtype, device=dev)
    pad_a[:B] = alpha
    pad_d = torch.zeros(Bmax, dtype=torch.int32, device=dev)
    pad_d[:B] = draft_len.to(torch.int32)
    got_a = [torch.empty_like(pad_a) for _ in range(world)]
    got_d = [torch.empty_like(pad_d) for _ in range(world)]
    dist.all_gather(got_a, pad_a, group=group)
    dist.all_gather(got_d, pad_d, group=group)
    alpha_all = torch.cat([got_a[r][: sizes[r]] for r in range(world)])
    dl_all = torch.cat([got_d[r][: sizes[r]] for r in range(world)])
    return alpha_all, dl_all, sum(sizes[:rank]), sizes


def global_schedule(alpha: torch.Tensor, cost_a: float, cost_b: float, budget: int, *, draft_len=None,
                    ratios=None, objective=None, cost_table=None, group=None, schedule=None):
    """D-cut of the whole partitioned batch, seen from one rank.

    alpha [B_r, Dmax] / draft_len [B_r] are this rank's requests; `budget` is the verify budget of
    the whole batch (0 = none).  Every rank must call this together (it all-gathers).  Returns
    this rank's (keep_len [B_r] int32, row_offsets [B_r + 1] int32, total_K, U_q48): keep_len and
    the global K and U(K) are the ones sv_schedule_depth computes for the concatenated batch;
    row_offsets pack this rank's kept target rows (n_i + 1 per request) for sv_verify_ragged.

    `schedule` is the scheduling call (default: the library's sv_schedule_depth through
    schedule_depth); it receives the concatenated batch on this rank's device and returns
    (keep_len, row_offsets, total_K, U_q48) for it.
    """
    if schedule is None:
        from . import SV_OBJ_THROUGHPUT, schedule_depth

        def schedule(a, ca, cb, bud, dl):
            return schedule_depth(a, ca, cb, bud, draft_len=dl, ratios=ratios,
                                  objective=SV_OBJ_THROUGHPUT if objective is None else objective,
                                  cost_table=cost_table)
    alpha_all, dl_all, start, _ = gather_batch(alpha, draft_len, group)
    keep_all, _, K, U = schedule(alpha_all, cost_a, cost_b, budget, dl_all)
    B = alpha.shape[0]
    keep = keep_all[start: start + B].to(torch.int32).contiguous()
    offs = torch.zeros(B + 1, dtype=torch.int32, device=keep.device)
    offs[1:] = torch.cumsum(keep + 1, 0).to(torch.int32)
    return keep, offs, K, U


# ------------------------------------------------------------------------------------------
# Vocabulary partition: the LM head split across ranks by vocabulary columns (the pages' TP
# serving, AngelSpec explainer "The numbers"; release article "Key Takeaways").  Verification's
# vocabulary-wide steps are sums and searches over fixed chunks of the vocabulary, so a rank that
# holds a contiguous range of chunks runs them on its range and the ranks exchange two small
# workspace regions: the chunk records (16 bytes per row and chunk) after the stream, and the
# draw weights' range sums (2 x 8 floats per request and chunk) before the draw.  The accept chain
# runs on every rank from the gathered records; the rank whose chunks hold the drawn token writes
# it.  The result matches sv_verify_sample's (sums grouped at the shard boundaries: float32
# rounding apart).
# ------------------------------------------------------------------------------------------

def chunk_ranges(nchunks: int, world: int) -> list[tuple[int, int]]:
    """Contiguous, balanced ranges of vocabulary chunks, one per rank (every rank at least one
    chunk: world <= nchunks)."""
    if world > nchunks:
        raise ValueError(f"{world} ranks for {nchunks} vocabulary chunks")
    return [(nchunks * r // world, nchunks * (r + 1) // world) for r in range(world)]


def gather_chunk_columns(region: torch.Tensor, ranges, rank: int, group=None) -> None:
    """region [rows, nchunks, item] (a view of a workspace region): rank r's columns
    ranges[r] are valid on rank r.  All-gathers them in place, so every rank holds every column."""
    import torch.distributed as dist
    world = len(ranges)
    width = max(b - a for a, b in ranges)
    c0, c1 = ranges[rank]
    local = torch.zeros((region.shape[0], width, region.shape[2]), dtype=region.dtype, device=region.device)
    local[:, : c1 - c0] = region[:, c0:c1]
    parts = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(parts, local, group=group)
    for r, (a, b) in enumerate(ranges):
        if r != rank:
            region[:, a:b] = parts[r][:, : b - a]


def vocab_parallel_verify_sample(target_local, draft_local, draft_tokens, temperature, K: int, V: int, *, seed=0,
                                 round_=0, request_ids=None, ws=None, group=None, stream=None):
    """sv_verify_sample with the vocabulary split across the group's ranks.  target_local
    [B*(K+1), V_r] and draft_local [B*K, V_r] hold this rank's columns: chunks
    chunk_ranges(nchunks, world)[rank] of the library's tiling (sv_vocab_chunks), i.e. columns
    [c0 * chunk_len, min(V, c1 * chunk_len)).  Returns (tokens, accept_len, p, q, flags), the same
    on every rank."""
    import torch.distributed as dist
    from . import (sv_vocab_chunks, sv_verify_regions, sv_verify_sample_phase, workspace, _dt, _rows,
                   SV_OP_VERIFY, SV_PHASE_STATS, SV_PHASE_ACCEPT, SV_PHASE_WEIGHTS, SV_PHASE_PICK)
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    dt = _dt(target_local)
    B = temperature.numel()
    dev = target_local.device
    cl, nc = sv_vocab_chunks(V, dt)
    ranges = chunk_ranges(nc, world)
    c0, c1 = ranges[rank]
    if ws is None:
        ws = workspace(SV_OP_VERIFY, B, K, V, dt, dev)
    out = (torch.full((B, K + 1), -1, dtype=torch.int32, device=dev),
           torch.empty(B, dtype=torch.int32, device=dev),
           torch.empty((B, K), dtype=torch.float32, device=dev),
           torch.empty((B, K), dtype=torch.float32, device=dev),
           torch.zeros(B, dtype=torch.uint8, device=dev))
    reg = sv_verify_regions(B, K, V, dt)
    w8 = ws.view(torch.uint8)
    rec = w8[reg["rec_offset"]: reg["rec_offset"] + reg["rec_bytes"]].view(B * (2 * K + 1), nc, 16)
    mass = w8[reg["mass_offset"]: reg["mass_offset"] + reg["mass_bytes"]].view(B, nc, 32)
    mass_p = w8[reg["mass_p_offset"]: reg["mass_p_offset"] + reg["mass_bytes"]].view(B, nc, 32)
    args = (target_local, _rows(target_local)[1], draft_local, _rows(draft_local)[1], draft_tokens, temperature, seed,
            round_, request_ids, dt, B, K, V, c0, c1)

    def phase(ph):
        sv_verify_sample_phase(*args, ph, *out, ws, stream)

    phase(SV_PHASE_STATS)
    gather_chunk_columns(rec, ranges, rank, group)
    phase(SV_PHASE_ACCEPT)
    phase(SV_PHASE_WEIGHTS)
    gather_chunk_columns(mass, ranges, rank, group)
    gather_chunk_columns(mass_p, ranges, rank, group)
    phase(SV_PHASE_PICK)
    # the drawn token is written by the rank that holds it (elsewhere -1); flags: that rank's
    # are a superset of the others'
    dist.all_reduce(out[0], op=dist.ReduceOp.MAX, group=group)
    fl = out[4].to(torch.int32)
    dist.all_reduce(fl, op=dist.ReduceOp.MAX, group=group)
    out[4].copy_(fl.to(torch.uint8))
    return out
