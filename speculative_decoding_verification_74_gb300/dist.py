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
