"""Benchmark: verified draft positions/s and achieved HBM GB/s of the verification hot path.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl sv|reference] [--workload c1..c5]
                  [--also c2,c4,c5]

One step = one verification round (plus the D-cut schedule for c4) over one batch of synthetic
logits already resident in HBM, through the library's C ABI.  Rotating input sets keep every
step's logits cold in L2: their logits exceed the 129 MB L2 twice over, and so do the rows the
other sets read again after their stream (the draw, a tree walk).  Rank 0 prints one JSON line: the
headline workload (default c3, B=64 K=16 V=151936 fp32, the largest stream) with its roofline,
end-to-end and CPU-baseline legs, and the other workloads (--also) measured the same way under
"other_workloads".

--impl reference times the fp64 CPU oracle on the host cores on a bounded sample of the same
workload (the only other place this file runs oracle code, besides the cpu_baseline leg).
Under torchrun each rank is an independent replica on its own GPU (weak scaling): requests
are independent, so there is no data-path collective; only the timing max-reduction.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import workloads as W  # noqa: E402
from synth import trees as TR  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    "c1": "greedy T=0 verify, B=4 K=3 V=32000 bf16, draft tokens fused from draft argmax",
    "c2": "stochastic MTP-style verify T=1.0, B=16 K=3 V=151936 bf16",
    "c3": "block-parallel DFly-style verify T=0.6, B=64 K=16 V=151936 fp32",
    "c4": "D-cut schedule (B=64 D=16 budget 384, c=1+0.05K) + ragged verify T=1.0 V=151936 bf16",
    "c5": "mixed round c64: 32 chat K=3 + 32 code K=16, T in {0,0.6,1}, V=151936 bf16",
    "t1": "token-tree verify T=1.0, B=64 trees of 16 nodes (8 shapes, 15 candidates each), V=151936 bf16",
}


def make_sets(workload: str, n_sets: int, base_seed: int):
    """Synthetic input sets (host numpy) of one workload."""
    sets = []
    for j in range(n_sets):
        seed = base_seed + j
        if workload == "c1":
            sets.append({"batch": W.c1_greedy(seed)})
        elif workload == "c2":
            sets.append({"batch": W.c2_mtp(seed)})
        elif workload == "c3":
            sets.append({"batch": W.c3_dfly(seed)})
        elif workload == "c4":
            s = W.c4_alpha(seed)
            b = W.c4_verify(s, np.full(64, 16, np.int32), seed=seed)
            sets.append({"batch": b, "sched": s})
        elif workload == "c5":
            sets.append({"batch": W.c5_mixed(seed=base_seed, rnd=j)})
        elif workload == "t1":
            sets.append({"batch": TR.t1_tree(seed)})
    return sets


def algorithmic_bytes(b, keep_len) -> int:
    """Each needed logit byte once: n_i + 1 target rows, plus n_i draft rows when the request
    samples (T > 0) or takes its drafted tokens from the draft argmax.  A tree of N nodes counts
    as n = N - 1: N target rows and, sampled, the draft rows of the N - 1 nodes that can have
    children (the walk's re-reads of a node's rows after a rejection are not counted)."""
    elt = 2 if b.dtype == "bf16" else 4
    rows = 0
    for i in range(b.B):
        n = int(keep_len[i])
        rows += n + 1
        if b.temperature[i] > 0 or b.tokens is None:
            rows += n
    return rows * b.V * elt


# -------------------------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    """Hash of the code that defines the verification kernel and its launch, with comments and
    whitespace removed (a recorded traffic figure is only used while this code is unchanged)."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_74_gb300", "csrc")
    for f in ("sv_device.cuh", "sv_internal.h", "sv_verify.cu"):
        with open(os.path.join(csrc, f)) as fh:
            code = re.sub(r"//[^\n]*", "", fh.read())
        h.update(f.encode() + " ".join(code.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per verification-kernel launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 10 ms, with the tool's timestamps, so that the
    samples taken inside a marked host-time window can be told apart."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.proc = None
        self.marks = {}
        self.path = f"/tmp/sv_clocks_{os.getpid()}.csv"
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "10", "-i", str(gpu_index)], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark(self, name: str):
        self.marks[name] = time.time()

    def _samples(self):
        import datetime
        out = []
        with open(self.path) as f:
            for ln in f:
                parts = [x.strip() for x in ln.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    sm, smax = float(parts[2].split()[0]), float(parts[3].split()[0])
                except ValueError:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    ts = None  # unreadable timestamp: counted as a sample of the whole run
                reasons = {nm for nm, v in zip(self.REASONS, parts[6:10]) if v.lower() == "active"}
                out.append((ts, sm, smax, reasons))
        return out

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        samples = self._samples()
        os.unlink(self.path)

        def within(a, b):
            if a not in self.marks or b not in self.marks:
                return []
            return [x for x in samples if x[0] is not None and self.marks[a] <= x[0] <= self.marks[b]]
        timed, load = within("timed0", "timed1"), within("load0", "load1")
        use = timed if len(timed) >= 3 else (timed + load) if (timed or load) else samples
        basis = ("samples inside the timed region" if len(timed) >= 3 else
                 "samples inside the timed region and during a replay of the timed graphs right after it (the "
                 "timed region is short next to the 10 ms sampling interval)" if (timed or load)
                 else "all samples of the run")
        if not timed and not load:
            timed = samples
        reasons = set()
        for x in timed + load:
            reasons |= x[3]
        return {"sm_mhz": float(np.median([x[1] for x in use])) if use else None,
                "sm_max_mhz": max(x[2] for x in samples) if samples else None,
                "reasons": sorted(reasons), "samples_timed": len(timed), "samples_load": len(load),
                "basis": basis}


# -------------------------------------------------------------------------------- GPU arm

class GpuWorkload:
    def __init__(self, workload, sets, device):
        import torch
        import speculative_decoding_verification_74_gb300 as sv
        self.sv, self.torch, self.dev = sv, torch, device
        self.workload = workload
        self.sets = []
        b0 = sets[0]["batch"]
        self.dt = sv.SV_BF16 if b0.dtype == "bf16" else sv.SV_F32
        self.tree = workload == "t1"
        self.B, self.V = b0.B, b0.V
        self.Kmax = b0.Nmax if self.tree else b0.Kmax  # trees: Nmax
        self.ws = sv.workspace(sv.SV_OP_TREE if self.tree else sv.SV_OP_VERIFY, self.B, self.Kmax, self.V, self.dt,
                               device)
        self.ws_sched = sv.workspace(sv.SV_OP_SCHEDULE, self.B, self.Kmax, 1, sv.SV_F32, device)
        for s in sets:
            self.sets.append(self._upload(s))
        if self.tree:
            self.out = (torch.empty((self.B, self.Kmax), dtype=torch.int32, device=device),
                        torch.empty((self.B, self.Kmax), dtype=torch.int32, device=device),
                        torch.empty(self.B, dtype=torch.int32, device=device),
                        torch.empty(self.B, dtype=torch.uint8, device=device))
        else:
            self.out = (torch.empty((self.B, self.Kmax + 1), dtype=torch.int32, device=device),
                        torch.empty(self.B, dtype=torch.int32, device=device),
                        torch.empty((self.B, self.Kmax), dtype=torch.float32, device=device),
                        torch.empty((self.B, self.Kmax), dtype=torch.float32, device=device),
                        torch.empty(self.B, dtype=torch.uint8, device=device))
        # what a caller reads back: emitted tokens and accepted lengths
        self.results = (self.out[1], self.out[2]) if self.tree else (self.out[0], self.out[1])
        self.sched_out = (torch.empty(self.B, dtype=torch.int32, device=device),
                          torch.empty(self.B + 1, dtype=torch.int32, device=device),
                          torch.empty(1, dtype=torch.int32, device=device),
                          torch.empty(1, dtype=torch.int64, device=device))

    def _t(self, a, dtype=None):
        torch = self.torch
        if a is None:
            return None
        if dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(self.dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def _upload(self, s):
        b = s["batch"]
        if self.tree:
            return {"b": b, "target": self._t(b.target, b.dtype), "draft": self._t(b.draft, b.dtype),
                    "t_off": self._t(b.node_offsets), "parent": self._t(b.parent), "tokens": self._t(b.tokens),
                    "temp": self._t(b.temperature), "rid": self._t(b.request_ids)}
        d = {"b": b,
             "target": self._t(b.target, b.dtype), "draft": self._t(b.draft, b.dtype),
             "t_off": self._t(b.t_offsets), "d_off": self._t(b.d_offsets),
             "tokens": self._t(b.tokens), "keep": self._t(b.keep_len), "temp": self._t(b.temperature),
             "rid": self._t(b.request_ids)}
        if "sched" in s:
            d["alpha"] = self._t(s["sched"].alpha)
            d["sched"] = s["sched"]
        return d

    def step(self, j, stream=None):
        sv = self.sv
        d = self.sets[j % len(self.sets)]
        b = d["b"]
        if self.tree:
            sv.sv_verify_tree(d["target"], b.V, d["draft"], b.V, d["t_off"], b.target.shape[0], d["parent"],
                              d["tokens"], d["temp"], b.seed, b.round, d["rid"], self.dt, self.B, self.Kmax, self.V,
                              *self.out, self.ws, stream)
        elif self.workload == "c1":
            sv.sv_verify_greedy(d["target"], b.V, d["draft"], b.V, None, self.dt, self.B, self.Kmax, self.V,
                                self.out[0], self.out[1], self.ws, stream)
        elif self.workload in ("c2", "c3"):
            sv.sv_verify_sample(d["target"], b.V, d["draft"], b.V, d["tokens"], d["temp"], b.seed, b.round,
                                d["rid"], self.dt, self.B, self.Kmax, self.V, *self.out, self.ws, stream)
        else:
            keep = d["keep"]
            if self.workload == "c4":
                s = d["sched"]
                sv.sv_schedule_depth(d["alpha"], self.Kmax, None, self.B, self.Kmax, s.cost_a, s.cost_b, s.budget,
                                     None, sv.SV_OBJ_THROUGHPUT, *self.sched_out, self.ws_sched, stream)
                keep = self.sched_out[0]
            sv.sv_verify_ragged(d["target"], b.V, d["t_off"], b.target.shape[0], d["draft"], b.V, d["d_off"],
                                b.draft.shape[0], d["tokens"], self.Kmax, keep, d["temp"], b.seed, b.round, d["rid"],
                                self.dt, self.B, self.Kmax, self.V, *self.out, self.ws, stream)

    def keep_len(self, j):
        """Kept positions of set j (runs the schedule once for c4)."""
        d = self.sets[j % len(self.sets)]
        if self.workload != "c4":
            return d["b"].keep_len
        self.step(j)
        self.torch.cuda.synchronize()
        return self.sched_out[0].cpu().numpy()


def rank_seed(base: int, rank: int) -> int:
    """Seed of a rank's input sets: every rank verifies its own independent requests."""
    return base + 7919 * rank


def job_totals(ms: float, positions: float, dist=None, device="cpu"):
    """Whole-job totals over the ranks: the slowest rank's time (max) and the positions all ranks
    verified (sum).  Without a process group, the local values."""
    if dist is None:
        return ms, positions
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    n = torch.tensor([positions], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


def cost_table_leg(gw, reps: int = 200) -> dict:
    """D-cut with a profiled latency table (c4 only, outside the timed region).

    Profiles the table once, as the D-cut pipeline does at startup: the ragged verification
    kernels of input set 0 (no target model) are timed on a (batch size x keep ratio) grid.
    The D-cut call is then timed with the linear cost and with the table: one CUDA graph
    each, `reps` replays between CUDA events."""
    import torch
    import speculative_decoding_verification_74_gb300 as sv
    from speculative_decoding_verification_74_gb300.cost_table import profile_cost_table
    d = gw.sets[0]
    b, D = d["b"], gw.Kmax
    keeps = {}

    def step(nb, K):
        if (nb, K) not in keeps:              # built on the first (untimed warm-up) call
            extra = K - nb
            keeps[(nb, K)] = torch.tensor([min(D, extra // nb + (1 if i < extra % nb else 0)) for i in range(nb)],
                                          dtype=torch.int32, device=gw.dev)
        sv.sv_verify_ragged(d["target"], b.V, d["t_off"], b.target.shape[0], d["draft"], b.V, d["d_off"],
                            b.draft.shape[0], d["tokens"], gw.Kmax, keeps[(nb, K)], d["temp"], b.seed, b.round,
                            d["rid"], gw.dt, nb, gw.Kmax, gw.V, *gw.out, gw.ws, None)

    grid = [16, 32, 48, 64]
    Ks, cs = profile_cost_table(step, grid, D, reps=5, warmup=2)
    s = d["sched"]
    calls = {
        "linear": lambda: sv.sv_schedule_depth(d["alpha"], gw.Kmax, None, gw.B, gw.Kmax, s.cost_a, s.cost_b,
                                               s.budget, None, sv.SV_OBJ_THROUGHPUT, *gw.sched_out, gw.ws_sched),
        "table": lambda: sv.sv_schedule_depth_table(d["alpha"], gw.Kmax, None, gw.B, gw.Kmax, Ks, cs, s.budget,
                                                    None, sv.SV_OBJ_THROUGHPUT, *gw.sched_out, gw.ws_sched),
    }
    us, chosen = {}, {}
    cap = torch.cuda.Stream()
    for name, fn in calls.items():
        fn()
        torch.cuda.synchronize()
        chosen[name] = int(gw.sched_out[2].item())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us[name] = e0.elapsed_time(e1) * 1e3 / reps
    return {"profiled_step": "ragged verification kernels of input set 0 (no target model), median of 5",
            "grid": {"batch_sizes": grid, "ratios": [0.25, 0.5, 0.75, 1.0], "depth": D},
            "knots_K": Ks, "knots_ms": cs, "chosen_K": chosen,
            "schedule_us": us, "timing": f"CUDA events over {reps} graph replays of one D-cut call"}


def rotation_sets(workload: str, b0) -> int:
    """How many input sets the timed steps rotate through.  The stream's copies are marked
    evict-first in L2, so the lines a step reads at a higher priority (the rows the draw reads
    again; a tree walk's rows) can outlive the stream of the next set.  So there are enough sets
    that the logits read exceed L2 twice over, and that the other sets' re-read rows (at most 2
    rows per request, 4 for a tree) exceed it twice over too: no step finds its own rows in L2
    from its set's previous turn."""
    set_bytes = algorithmic_bytes(b0, b0.keep_len if workload != "c4" else np.full(b0.B, 16))
    reread = b0.B * (4 if workload == "t1" else 2) * b0.V * (2 if b0.dtype == "bf16" else 4)
    n_sets = max(2, int(np.ceil(2.0 * L2_BYTES / max(1, set_bytes))), 1 + int(np.ceil(2.0 * L2_BYTES / reread)))
    return min(n_sets, 200)


def measure_workload(workload, steps, warm, rank, world, dev, dist, *, full: bool) -> dict:
    """One workload's measurement on this rank: K timed steps (CUDA graphs, rotating input sets
    larger than L2), per-kernel durations, and, with `full`, the end-to-end leg.  Returns the
    fields of a bench line (whole-job values where they are reduced over ranks)."""
    import torch
    import speculative_decoding_verification_74_gb300 as sv

    probe = make_sets(workload, 1, rank_seed(1000, rank))
    n_sets = rotation_sets(workload, probe[0]["batch"])
    sets = probe + make_sets(workload, n_sets - 1, rank_seed(1001, rank))
    gw = GpuWorkload(workload, sets, dev)

    keeps = [gw.keep_len(j) for j in range(len(gw.sets))]
    pos = [int(np.sum(k)) for k in keeps]
    trows = [int(np.sum(np.asarray(k) + 1)) for k in keeps]  # target rows verified (kept + bonus)
    byts = [algorithmic_bytes(gw.sets[j]["b"], keeps[j]) for j in range(len(gw.sets))]
    R = len(gw.sets)
    order = [j % R for j in range(steps)]          # the set each timed step reads
    tot_pos = sum(pos[j] for j in order)
    tot_rows = sum(trows[j] for j in order)
    tot_bytes = sum(byts[j] for j in order)

    # Steps are captured into CUDA graphs (kernels only, no host work): one graph per input set
    # and one graph running every set once in order.  The timed loop replays the latter K // R
    # times and single-set graphs for the remaining K % R steps, so exactly K steps run.
    stream = torch.cuda.current_stream()
    for j in range(R):
        gw.step(j)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    graphs, glaunch = [], []
    for j in range(R):
        g = torch.cuda.CUDAGraph()
        n0 = sv.sv_launch_count()
        with torch.cuda.graph(g, stream=cap):
            gw.step(j)
        glaunch.append(sv.sv_launch_count() - n0)
        graphs.append(g)
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all, stream=cap):
        for j in range(R):
            gw.step(j)
    for j in range(warm):
        graphs[j % R].replay()
    g_all.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = ClockSampler(dev.index or 0) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark("timed0")
    ev0.record(stream)
    for _ in range(steps // R):
        g_all.replay()
    for j in range(steps % R):
        graphs[j].replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark("timed1")
    ms = ev0.elapsed_time(ev1)
    launches = sum(glaunch[j] for j in order)
    if clocks:  # the same graphs for ~0.3 s more, so the sampler sees the clocks under this load
        clocks.mark("load0")
        t_end = time.time() + 0.3
        while time.time() < t_end:
            for _ in range(max(1, 1000 // R)):
                g_all.replay()
            torch.cuda.synchronize()
        clocks.mark("load1")
    clk = clocks.stop() if clocks else None
    _, job_rows = job_totals(ms, tot_rows, dist, dev)
    ms, job_pos = job_totals(ms, tot_pos, dist, dev)
    if dist:
        dist.barrier()

    # per-kernel durations: the same K steps replayed from graphs captured with the library's
    # CUDA-event brackets around each kernel (one graph at a time, collected after each replay)
    kms = [0.0] * sv.SV_NUM_KERNELS
    kn = [0] * sv.SV_NUM_KERNELS
    for j0 in range(R):
        idx = [j for j in order if j == j0]
        if not idx:
            continue
        sv.sv_profile_reset()
        sv.sv_profile_enable(True)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            gw.step(j0)
        sv.sv_profile_enable(False)
        g.replay()          # warm replay (not counted)
        torch.cuda.synchronize()
        for _ in idx:
            g.replay()
            a, n = sv.sv_profile_collect()
            kms = [x + y for x, y in zip(kms, a)]
            kn = [x + y for x, y in zip(kn, n)]
        sv.sv_profile_reset()
        del g

    e2e = None
    if full:
        # end to end through host buffers: H2D of the step's inputs from pinned memory, the C ABI
        # call, D2H of the emitted tokens and accepted lengths
        e2e = run_e2e(gw, warm, steps, stream)
        e2e_ms, e2e_pos = job_totals(e2e.pop("ms"), e2e.pop("positions"), dist, dev)
        e2e["value"] = e2e_pos / (e2e_ms * 1e-3)

    ctab = None
    if full and workload == "c4" and rank == 0:
        try:
            ctab = cost_table_leg(gw)
        except Exception as exc:  # context only, outside the timed region: never lose the bench line
            ctab = {"error": f"{type(exc).__name__}: {exc}"}

    peak, peak_kind = measured_peaks()
    kid = dominant_kernel(kms)
    k1_avg_ms = kms[kid] / max(1, kn[kid])
    k1_bytes = tot_bytes / steps
    achieved = k1_bytes / (k1_avg_ms * 1e-3) / 1e9
    out = {
        "value": job_pos / (ms * 1e-3), "ms_per_step": ms / steps,
        "config": {"workload": f"{workload}: {WORKLOADS[workload]}", "B": gw.B, "Kmax": gw.Kmax, "V": gw.V,
                   "logits": "bf16" if gw.dt == sv.SV_BF16 else "f32",
                   "arithmetic": "f32 (exp2, sums, probabilities); f64 for the D-cut objective",
                   "positions_per_step": tot_pos / steps, "logit_bytes_per_step": k1_bytes,
                   "l2": f"{len(gw.sets)} rotating input sets, {sum(byts) / 1e6:.0f} MB of logits read > 129 MB L2",
                   "parallelism": f"replicas x{world} (independent requests, no collective)"},
        "achieved_gbs_step": tot_bytes / (ms * 1e-3) / 1e9,
        "target_rows_per_s": job_rows / (ms * 1e-3),
        "roofline": {"bound": "hbm", "kernel": sv.KERNEL_NAMES[kid], "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": achieved / peak, "traffic": recorded_traffic(workload),
                     "avg_launch_us": k1_avg_ms * 1e3, "bytes_per_launch": k1_bytes,
                     "timing": "CUDA events on the launching stream around each launch of the kernel, inside "
                               "graph replays of the same K steps"},
        "kernels_us_per_step": {sv.KERNEL_NAMES[i]: kms[i] * 1e3 / steps for i in range(sv.SV_NUM_KERNELS) if kn[i]},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if e2e is not None:
        out["e2e"] = e2e
    if ctab is not None:
        out["cost_table"] = ctab
    del graphs, g_all, gw
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def dominant_kernel(kms) -> int:
    """The library kernel with the most time in the measured steps."""
    return int(np.argmax(kms))


def run_gpu(args, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    steps, warm = args.steps, args.warmup
    head = measure_workload(args.workload, steps, warm, rank, world, dev, dist, full=True)
    others = {}
    for w in args.also:
        if w == args.workload:
            continue
        m = measure_workload(w, steps, warm, rank, world, dev, dist, full=False)
        others[w] = {k: m[k] for k in ("value", "ms_per_step", "achieved_gbs_step", "roofline",
                                       "kernels_us_per_step", "gpu_launches", "clocks")}
        others[w]["config"] = m["config"]
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    cpu = cpu_baseline(args.workload) if world == 1 else None
    if cpu is not None:
        cpu["cpu"] = cpu_model()
    try:
        cpu_all = cpu_baseline_all_cores(args.workload) if world == 1 else None
    except Exception as exc:  # the all-core figure is context only: never lose the bench line
        cpu_all = {"error": f"{type(exc).__name__}: {exc}"}
    line = {
        "metric": "verified draft positions/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU",
        "value": head["value"], "unit": "positions/s", "n_gpus": world, "steps": steps, "warmup": warm,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded numpy generators in synth/)",
        "config": head["config"],
        "achieved_gbs_step": head["achieved_gbs_step"],
        "target_rows_per_s": head["target_rows_per_s"],
        "roofline": head["roofline"],
        "kernels_us_per_step": head["kernels_us_per_step"],
        "e2e": head["e2e"],
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "gpu_launches": head["gpu_launches"],
        "timed_loop": "CUDA graphs of the captured C ABI calls: one graph running every input set once, "
                      "replayed K // R times, plus single-set graphs for the K % R remaining steps",
        "clocks": head["clocks"],
    }
    if "cost_table" in head:
        line["cost_table"] = head["cost_table"]
    if others:
        line["other_workloads"] = others
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_e2e(gw, warm, steps, stream):
    import torch
    sv = gw.sv
    pinned = []
    names = ("target", "draft", "t_off", "d_off", "parent", "tokens", "keep", "temp", "rid", "alpha")
    for d in gw.sets[:2]:
        pinned.append({k: d[k].cpu().pin_memory() for k in names if d.get(k) is not None})
    h_out = [torch.empty(tuple(r.shape), dtype=torch.int32).pin_memory() for r in gw.results]
    # device staging buffers for one set (the step's inputs land here every step)
    stage = {k: torch.empty_like(gw.sets[0][k]) for k in pinned[0]}
    h2d = sum(v.numel() * v.element_size() for v in pinned[0].values())
    d2h = sum(v.numel() * v.element_size() for v in h_out)
    n = max(1, min(steps, 20))
    orig = gw.sets

    def one(j):
        src = pinned[j % 2]
        for k, v in src.items():
            stage[k].copy_(v, non_blocking=True)
        d = dict(orig[j % 2])
        d.update(stage)
        gw.sets = [d]
        gw.step(0)
        for h, r in zip(h_out, gw.results):
            h.copy_(r, non_blocking=True)

    for j in range(2):
        one(j)
    torch.cuda.synchronize()
    pos = [int(np.sum(gw.keep_len(j))) for j in range(2)] if gw.workload != "c4" else None
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    ev0.record(stream)
    for j in range(n):
        one(j)
    ev1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    gw.sets = orig
    if pos is None:
        pos = [int(np.sum(gw.keep_len(j))) for j in range(2)]
    tot = sum(pos[j % 2] for j in range(n))
    ms = ev0.elapsed_time(ev1)
    return {"value": tot / (ms * 1e-3), "positions": tot, "ms": ms, "unit": "positions/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n, "wall_s": wall,
            "note": "pinned host inputs copied to the device each step, C ABI call, tokens+lengths copied back"}


# -------------------------------------------------------------------------------- CPU oracle

def oracle_sets(workload):
    """Input sets for the oracle legs: the workload's own recipe and request shapes.  C3 keeps 8 of
    its 64 requests (each request is 33 fp32 rows of 151936; the oracle only ever takes a few per
    step, and a spawned worker per core holds its own copy)."""
    if workload == "c3":
        return [{"batch": W.c3_dfly(1000, B=8)}]
    return make_sets(workload, 1, 1000)


def oracle_step(workload, sets, j, req_slice):
    from oracle.verify import verify_batch
    from oracle.schedule import dcut_schedule
    s = sets[j % len(sets)]
    b = s["batch"]
    if workload == "t1":
        from oracle.tree import verify_tree_batch
        lo, hi = req_slice
        o = b.node_offsets
        verify_tree_batch(b.target, b.draft, o[lo:hi + 1], b.parent, b.tokens, b.temperature[lo:hi], b.seed, b.round,
                          b.request_ids[lo:hi], b.dtype)
        return int(np.sum(b.keep_len[lo:hi]))
    keep = b.keep_len
    if workload == "c4":
        sc = s["sched"]
        keep = dcut_schedule(sc.alpha, None, sc.cost_a, sc.cost_b, sc.budget)["keep_len"]
    lo, hi = req_slice
    sub = slice(lo, hi)
    verify_batch(b.target, b.t_offsets[lo:], b.draft, b.d_offsets[lo:] if b.d_offsets is not None else None,
                 None if b.tokens is None else b.tokens[sub], keep[sub], b.temperature[sub], b.seed, b.round,
                 b.request_ids[sub], b.dtype, b.Kmax)
    return int(np.sum(keep[sub]))


def cpu_baseline(workload, budget_s: float = 15.0):
    """The oracle, as it stands, on a bounded sample of the workload (single process)."""
    sets = oracle_sets(workload)
    b = sets[0]["batch"]
    t0 = time.perf_counter()
    pos = 0
    nreq = 0
    i = 0
    while time.perf_counter() - t0 < budget_s and nreq < 64 * b.B:
        pos += oracle_step(workload, sets, 0, (i % b.B, i % b.B + 1))
        nreq += 1
        i += 1
    dt = time.perf_counter() - t0
    return {"value": pos / dt, "unit": "positions/s", "cores": 1, "kind": "oracle",
            "sample": f"{nreq} requests of the {workload} batch verified one by one by the fp64 numpy oracle "
                      f"({dt:.1f} s, 1 thread)"}


def cpu_model() -> str:
    """The host CPU's model name (or its architecture when /proc/cpuinfo names none)."""
    import platform
    part = None
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
                if ln.lower().startswith("cpu part") and part is None:
                    part = ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return f"{platform.machine()} (CPU part {part})" if part else platform.machine()


_ORACLE_SETS = None


def _oracle_init(workload):
    global _ORACLE_SETS
    _ORACLE_SETS = (workload, oracle_sets(workload))


def _oracle_ready(_):
    return _ORACLE_SETS is not None


def _oracle_request(i):
    workload, sets = _ORACLE_SETS
    b = sets[0]["batch"]
    return oracle_step(workload, sets, 0, (i % b.B, i % b.B + 1))


def cpu_baseline_all_cores(workload, budget_s: float = 10.0):
    """The same oracle fanned out over requests on every host core (spawned worker processes,
    each holding its own copy of the inputs), timed from the moment every worker is ready."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_oracle_init, initargs=(workload,)) as pool:
        pool.map(_oracle_ready, range(cores), chunksize=1)
        t0 = time.perf_counter()
        pos, nreq, i = 0, 0, 0
        while time.perf_counter() - t0 < budget_s:
            batch = list(range(i, i + cores))
            pos += sum(pool.map(_oracle_request, batch, chunksize=1))
            nreq += len(batch)
            i += len(batch)
        dt = time.perf_counter() - t0
    return {"value": pos / dt, "unit": "positions/s", "cores": cores, "kind": "oracle", "cpu": cpu_model(),
            "sample": f"{nreq} requests of the {workload} batch verified by the fp64 numpy oracle in {cores} "
                      f"spawned worker processes, one request per task ({dt:.1f} s)"}


def run_reference(args, rank):
    if rank != 0:
        return
    sets = oracle_sets(args.workload)
    b = sets[0]["batch"]
    per_step = max(1, min(b.B, 4))
    for j in range(args.warmup):
        oracle_step(args.workload, sets, 0, ((j * per_step) % b.B, (j * per_step) % b.B + 1))
    t0 = time.perf_counter()
    pos = 0
    for j in range(args.steps):
        lo = (j * per_step) % b.B
        pos += oracle_step(args.workload, sets, 0, (lo, min(b.B, lo + per_step)))
    dt = time.perf_counter() - t0
    v = pos / dt
    line = {"impl": "reference", "metric": "verified draft positions/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU",
            "value": v, "unit": "positions/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy)",
            "config": {"workload": f"{args.workload}: {WORKLOADS[args.workload]}",
                       "sample": f"{per_step} requests per step"},
            "cpu_baseline": {"value": v, "unit": "positions/s", "cores": 1, "kind": "oracle",
                             "sample": f"{per_step} of {b.B} requests per step, fp64 numpy oracle, 1 thread"},
            "e2e": {"value": v, "unit": "positions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def check_world(gpus: int, world: int) -> None:
    """--gpus N must match the process group the launcher made (WORLD_SIZE): one rank per GPU."""
    if gpus != world:
        raise SystemExit(f"bench.py: --gpus {gpus} but WORLD_SIZE={world}; for N > 1 launch one rank per GPU, "
                         f"e.g. python -m torch.distributed.run --nproc-per-node {gpus} bench.py --gpus {gpus}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="sv", choices=["sv", "reference"])
    ap.add_argument("--workload", default="c3", choices=sorted(WORKLOADS),
                    help="headline workload (default c3, the largest stream)")
    ap.add_argument("--also", default="c2,c4,c5,t1",
                    help="comma-separated workloads measured after the headline and reported under "
                         "other_workloads ('' for none)")
    args = ap.parse_args()
    args.also = [w for w in args.also.split(",") if w]
    for w in args.also:
        if w not in WORKLOADS:
            raise SystemExit(f"bench.py: unknown workload {w!r} in --also")
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    check_world(args.gpus, world)
    if args.impl == "reference":
        run_reference(args, rank)
        return
    run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
