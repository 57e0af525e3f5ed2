// Verification kernel of libsv: one persistent launch per call streams every logit row the
// round needs, runs each request's accept chain once its rows are done, and draws the token at
// the accepted length while that request's rows are still in L2.
//
// Work is a global, ordered list of units, taken by the CTAs from a counter.  Segment j of the
// list holds, in order:
//   stream units of request j    a few consecutive (row, vocabulary chunk) tasks.  One producer
//                                lane issues 1-D bulk copies (cp.async.bulk) of 16 KB chunks into
//                                a 4-stage shared-memory ring; four consumer warps reduce each
//                                chunk.  A piece of a row (its chunks inside one unit) becomes one
//                                record {max m, sum of 2^(x k - rint(m k)) with k = log2(e)/T,
//                                first argmax, logit at the drafted token}.
//   the combine unit of j - D1   the request's accept chain, once its stream units are counted
//   the draw units of j - D2     one per vocabulary chunk of row a: sums, in 8 ranges, of the
//                                residual max(0, p_a - q_a) after a rejection and of p_a
//   the pick unit of j - D3      the draw: the crossing range among the 8 x chunks range sums,
//                                then a scan of that range
// The delays D1 < D2 < D3 (in requests) put about one to two grid-widths of units between the
// steps of a request, so that by the time a CTA takes a unit, what it waits for is usually done,
// and the draw reads row a while it is still in L2.
//
// The accept chain is the greedy test x_k == argmax, or the rejection test u_k q_k(x_k) <
// p_k(x_k); the first rejection is the accepted length (AngelSpec explainer, "MTP: fix position 2
// and 3", eq. L_e2e: one rejection voids every later position; AngelSpec release article, "Why one
// universal drafter underperforms": rejection-sampling verification in one target pass).  The
// draw is by inverse CDF in vocabulary order from norm(max(0, p_a - q_a)) after a rejection, or
// from p_n when every drafted token was accepted.
//
// Synchronisation.  Each step publishes with release semantics (a red.release count, or a
// st.release flag tagged with the call) and the producer lane of the CTA that takes the next step
// waits for it with acquire loads before it hands the step to its consumers.  Every wait is on
// work of a unit earlier in the list, which a running CTA took, so the grid cannot deadlock
// whatever the residency.  The four consumer warps of a CTA run independently (no CTA-wide barrier
// per chunk): piece partials meet in shared-memory slots guarded by mbarriers, and the accept
// chain and the pick synchronise the warps on an mbarrier too.  Every wait is bounded (~2 s, then
// SV_DEV_TIMEOUT, after which every other wait of the grid gives up).  Counters return to zero at
// the end of a call.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr float kLog2eF = 1.44269504088896340736f;

// request info, one uint16 per request, cached in shared memory by every CTA
constexpr uint16_t kInfoN = 0x3FF;
constexpr uint16_t kInfoNeedDraft = 1u << 10;
constexpr uint16_t kInfoSampled = 1u << 11;
constexpr uint16_t kInfoInvalid = 1u << 12;

constexpr int kMaxDelayRequests = 256;  // cap of each step delay (in requests)
constexpr int kSlots = 8;               // reduction slots (> the 4 stages a warp can lead by)

// log2(e) / T in float; every step uses this one value for a request's temperature.
__device__ __forceinline__ float kscale_of(float T) { return __fdiv_rn(kLog2eF, T); }

__device__ __forceinline__ int64_t target_row(const VerifyParams& p, int i, int k) {
  return (p.t_off ? static_cast<int64_t>(__ldg(p.t_off + i)) : static_cast<int64_t>(i) * (p.Kmax + 1)) + k;
}
__device__ __forceinline__ int64_t draft_row(const VerifyParams& p, int i, int k) {
  return (p.d_off ? static_cast<int64_t>(__ldg(p.d_off + i)) : static_cast<int64_t>(i) * p.Kmax) + k;
}

template <int DT>
__device__ __forceinline__ const char* row_ptr(const void* base, int64_t row, int64_t stride) {
  constexpr int kElt = DT == SV_BF16 ? 2 : 4;
  return reinterpret_cast<const char*>(base) + row * stride * kElt;
}

// A range [c0, c0 + len) of a row split into a head of plain loads, a 16-byte aligned interior of
// nvec vectors and a tail of plain loads; rows may start at any element.
struct ChunkSplit {
  int head, nvec, tail;
};
template <int kElt>
__device__ __forceinline__ ChunkSplit split_chunk(const char* row, int c0, int len) {
  const uintptr_t s = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(c0) * kElt;
  const uintptr_t e = s + static_cast<uintptr_t>(len) * kElt;
  const uintptr_t a = (s + 15u) & ~uintptr_t(15), z = e & ~uintptr_t(15);
  if (z <= a) return ChunkSplit{len, 0, 0};
  return ChunkSplit{static_cast<int>((a - s) / kElt), static_cast<int>((z - a) / 16), static_cast<int>((e - z) / kElt)};
}

__device__ __forceinline__ ChunkRecord ld_record(const ChunkRecord* r) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(r));
  ChunkRecord o;
  o.m = v.x;
  o.s = v.y;
  o.g = __float_as_int(v.z);
  o.xval = v.w;
  return o;
}

// hi + lo += x with the rounding error of the addition carried in lo (Knuth's TwoSum).
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float x) {
  const float s = __fadd_rn(hi, x);
  const float bb = __fsub_rn(s, hi);
  const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(x, bb));
  hi = s;
  lo = __fadd_rn(lo, err);
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Barrier of the four consumer warps on an mbarrier (one arrival per warp).  Bounded, and it gives
// up on an abort, so no warp is ever left waiting for one that has gone.  Every consumer warp
// must make the same sequence of calls.
struct ConsSync {
  uint64_t* bar;
  uint32_t phase;
  uint32_t* status;
  const volatile int* abort_flag;
  __device__ bool operator()() {
    const int lane = threadIdx.x & 31;
    __syncwarp();
    int ok = 1;
    if (lane == 0) {
      mbar_arrive(bar);
      ok = mbar_wait_or_abort(bar, phase, status, abort_flag) ? 1 : 0;
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    phase ^= 1u;
    return ok != 0;
  }
};

// ------------------------------------------------------------------------------------------
// per-request validation (every CTA computes the same info)
// ------------------------------------------------------------------------------------------
__device__ uint16_t request_info(const VerifyParams& p, int i, uint32_t* bad_out) {
  // every load is issued before any is used (one round trip)
  const int n = p.keep_len ? __ldg(p.keep_len + i) : p.Kmax;
  const float T = p.temperature ? __ldg(p.temperature + i) : 0.0f;
  const int ta = p.t_off ? __ldg(p.t_off + i) : 0, tb = p.t_off ? __ldg(p.t_off + i + 1) : 0;
  const int da = p.d_off ? __ldg(p.d_off + i) : 0, dbb = p.d_off ? __ldg(p.d_off + i + 1) : 0;
  uint32_t bad = 0;
  if (n < 0 || n > p.Kmax) bad |= SV_DEV_BAD_KEEP_LEN;
  if (!(T >= 0.0f) || isinf(T)) bad |= SV_DEV_BAD_TEMPERATURE;
  const bool sampled = T > 0.0f;
  const bool need_draft = (sampled || p.tokens == nullptr) && n > 0;  // n == 0: bonus row only
  if (sampled && n > 0 && p.tokens == nullptr) bad |= SV_DEV_BAD_TOKEN;
  if (need_draft && p.draft == nullptr) bad |= SV_DEV_NO_DRAFT_ROWS;
  if (!bad && p.t_off &&
      (tb - ta < n + 1 || ta < 0 || (p.t_rows >= 0 && static_cast<int64_t>(ta) + n + 1 > p.t_rows)))
    bad |= SV_DEV_BAD_OFFSETS;
  if (!bad && need_draft && p.d_off &&
      (dbb - da < n || da < 0 || (p.d_rows >= 0 && static_cast<int64_t>(da) + n > p.d_rows)))
    bad |= SV_DEV_BAD_OFFSETS;
  *bad_out = bad;
  if (bad) return kInfoInvalid;
  return static_cast<uint16_t>(n | (need_draft ? kInfoNeedDraft : 0) | (sampled ? kInfoSampled : 0));
}

__device__ __forceinline__ int rows_of(uint16_t inf) {
  if (inf & kInfoInvalid) return 0;
  const int n = inf & kInfoN;
  return n + 1 + ((inf & kInfoNeedDraft) ? n : 0);
}
__device__ __forceinline__ bool is_valid(uint16_t inf) { return !(inf & kInfoInvalid); }
__device__ __forceinline__ bool has_draw(uint16_t inf) { return !(inf & kInfoInvalid) && (inf & kInfoSampled); }

__device__ void write_invalid(const VerifyParams& p, int i, int tid, int nthreads) {
  for (int j = tid; j <= p.Kmax; j += nthreads) p.out_tokens[static_cast<int64_t>(i) * (p.Kmax + 1) + j] = -1;
  for (int j = tid; j < p.Kmax; j += nthreads) {
    if (p.out_p) p.out_p[static_cast<int64_t>(i) * p.Kmax + j] = NAN;
    if (p.out_q) p.out_q[static_cast<int64_t>(i) * p.Kmax + j] = NAN;
  }
  if (tid == 0) {
    p.out_accept_len[i] = -1;
    if (p.out_flags) p.out_flags[i] = SV_FLAG_INVALID;
  }
}

// ------------------------------------------------------------------------------------------
// shared state
// ------------------------------------------------------------------------------------------
enum : int32_t {
  kDescStream = 0,   // a chunk of a row
  kDescDrawT = 1,    // a chunk of target row a (a draft chunk follows in residual mode)
  kDescDrawD = 2,    // the draft chunk of a residual draw unit
  kDescSkip = 3,     // a draw unit of a request with nothing to draw
  kDescCombine = 4,  // the accept chain of request i
  kDescPick = 5,     // the draw of request i
  kDescEnd = 6
};
enum : int32_t { kPieceFirst = 1, kPieceLast = 2, kUnitLast = 4 };

// What the producer tells the consumers about one ring stage.
struct alignas(16) StageDesc {
  int32_t kind;
  int32_t i;       // request
  int32_t q;       // stream: row of the request (target rows 0..n, then its draft rows)
  int32_t c;       // vocabulary chunk
  int32_t flags;   // stream: kPieceFirst / kPieceLast / kUnitLast
  int32_t ntasks;  // stream: tasks of the unit (read on kUnitLast)
  int32_t mode;    // draw: kModeResidual or kModeBonus
  int32_t writer;  // consumer warp that merges this unit's partials and publishes its count
  float kscale;    // draw: the request's draw state
  float ct, cd, inv_st, inv_sd;
  int32_t pad[3];
  int64_t row_t, row_d;
};

// Per-row statistics of the request being combined (one entry per record row).
struct RowStatS {
  float s;     // sum of 2^(x k - rint(m k)) over the row (sampled rows)
  float m;     // row max
  int32_t g;   // first argmax (greedy rows)
  float xval;  // logit at the row's drafted token (sampled rows)
};

// One warp's part of a reduction: a row piece (m, s, g, and the drafted token's logit and chunk
// as seen by the warp that gathers it) or a draw unit's 2 x 8 range sums.
struct alignas(16) RedPart {
  float v[2 * kDrawRanges];
};

struct ConsumerSmem {
  RedPart part[kSlots][kConsumerWarps];
  // accept chain
  int a_min;
  uint32_t acc_flags;
  uint32_t bad;
  // pick
  ReqState st;
  float wsum[kConsumerWarps];
  int chunk, bonus;
  uint32_t flags;
  float base, thr;
  int pick_thread, last_pos;
};

// Dynamic shared memory: the ring, the stage descriptors, the row statistics of a combine, and
// the unit table (exclusive prefix of stream units per request, prefix counts of valid and of
// sampled requests, request info).
__host__ __device__ inline size_t verify_smem_bytes(int B, int Kmax) {
  size_t off = static_cast<size_t>(kStages) * kStageBytes + kStages * sizeof(StageDesc);
  off += static_cast<size_t>(2 * Kmax + 1) * sizeof(RowStatS);
  off += static_cast<size_t>(B + 1) * 4 + 2 * static_cast<size_t>(B + 1) * 2 + static_cast<size_t>(B) * 2;
  return (off + 15) & ~size_t(15);
}

// Consumer read of element e (chunk-relative) of a staged row: from the stage when it lies in the
// staged interior [head, head + nvec * kVec), else straight from the row.
template <int DT>
__device__ __forceinline__ float staged_elem(const unsigned char* sb, const char* row, int c0, int e, int head,
                                             int nvec) {
  constexpr int kVec = DT == SV_BF16 ? 8 : 4;
  if (e >= head && e < head + nvec * kVec) {
    if constexpr (DT == SV_BF16)
      return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(sb)[e - head]) << 16);
    else
      return reinterpret_cast<const float*>(sb)[e - head];
  }
  return load_logit<DT>(row, c0 + e);
}

// Contiguous ranges of a chunk: range r of nr covers [lo, hi).
__device__ __forceinline__ void draw_range(int len, int nr, int r, int* lo, int* hi) {
  const int seg = (len + nr - 1) / nr;
  *lo = min(len, r * seg);
  *hi = min(len, *lo + seg);
}

// ------------------------------------------------------------------------------------------
// accept chain of request i (the four consumer warps); every record of the request is complete
// and visible (the producer acquired its count).  Returns false after an abort.
// ------------------------------------------------------------------------------------------
__device__ bool combine_request(const VerifyParams& p, int i, RowStatS* rs, ConsumerSmem& cs, ConsSync& sync,
                                int tid, uint32_t tag) {
  const int lane = tid & 31, warp = tid >> 5;
  const int NC = p.nchunks, Kmax = p.Kmax, R = 2 * Kmax + 1;
  if (!sync()) return false;  // every warp is done with the shared state of the previous step
  uint32_t bad_in;
  const uint16_t info = request_info(p, i, &bad_in);  // valid: the request had a combine unit
  const int n = info & kInfoN;
  const bool sampled = info & kInfoSampled;
  const bool need_draft = info & kInfoNeedDraft;
  const float T = p.temperature ? __ldg(p.temperature + i) : 0.0f;
  const float kscale = sampled ? kscale_of(T) : 0.0f;
  const int nrows = n + 1 + (need_draft ? n : 0);
  const int32_t* toks = p.tokens ? p.tokens + static_cast<int64_t>(i) * p.tok_stride : nullptr;
  const ChunkRecord* recs = p.rec + static_cast<int64_t>(i) * R * NC;

  // 1. row statistics: one warp per row, one pass over the row's chunk records
  for (int q = warp; q < nrows; q += kConsumerWarps) {
    const bool is_target = q <= n;
    const int k = is_target ? q : q - n - 1;
    const int r = is_target ? k : Kmax + 1 + k;
    const ChunkRecord* rr = recs + static_cast<int64_t>(r) * NC;
    const int x = (sampled && k < n) ? __ldg(toks + k) : -1;  // drafted token of this row
    const int cx = (x >= 0 && x < p.V) ? x / p.chunk_len : -1;
    float m = -INFINITY, xval = NAN, S = 0.0f;
    int g = -1;
    ChunkRecord r0 = {-INFINITY, 0.0f, -1, NAN}, r1 = {-INFINITY, 0.0f, -1, NAN};
    if (lane < NC) r0 = ld_record(rr + lane);
    if (lane + 32 < NC) r1 = ld_record(rr + lane + 32);
    if (sampled) {
      // row max, then the piece sums rescaled to it, added with a compensated (TwoSum) tree
      m = fmaxf(r0.m, r1.m);
      for (int cc = lane + 64; cc < NC; cc += 32) m = fmaxf(m, ld_record(rr + cc).m);
      if (cx >= 0 && (cx & 31) == lane) xval = cx == lane ? r0.xval : cx == lane + 32 ? r1.xval : ld_record(rr + cx).xval;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      float hi = 0.0f, lo = 0.0f;
      if (m != -INFINITY) {
        const float C = exp_offset(m, kscale);
        if (r0.m != -INFINITY) two_sum_acc(hi, lo, r0.s * pow2_nonpos(exp_offset(r0.m, kscale) - C));
        if (r1.m != -INFINITY) two_sum_acc(hi, lo, r1.s * pow2_nonpos(exp_offset(r1.m, kscale) - C));
        for (int cc = lane + 64; cc < NC; cc += 32) {
          const ChunkRecord rc = ld_record(rr + cc);
          if (rc.m != -INFINITY) two_sum_acc(hi, lo, rc.s * pow2_nonpos(exp_offset(rc.m, kscale) - C));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xFFFFFFFFu, hi, o), l2 = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
        two_sum_acc(hi, lo, h2);
        lo += l2;
      }
      S = hi + lo;
    } else {
      merge_argmax(m, g, r0.m, r0.g);
      merge_argmax(m, g, r1.m, r1.g);
      for (int cc = lane + 64; cc < NC; cc += 32) {
        const ChunkRecord rc = ld_record(rr + cc);
        merge_argmax(m, g, rc.m, rc.g);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const int g2 = __shfl_xor_sync(0xFFFFFFFFu, g, o);
        merge_argmax(m, g, m2, g2);
      }
    }
    if (cx >= 0) xval = __shfl_sync(0xFFFFFFFFu, xval, cx & 31);
    if (lane == 0) {
      rs[r].s = S;
      rs[r].m = m;
      rs[r].g = g;
      rs[r].xval = xval;
    }
  }
  if (tid == 0) {
    cs.a_min = n;
    cs.acc_flags = 0;
    cs.bad = 0;
  }
  if (!sync()) return false;

  // 2. accept tests (each position independently; the first rejection is a min-reduction)
  const int rid = p.request_ids ? __ldg(p.request_ids + i) : i;
  auto tok = [&](int k) { return toks ? __ldg(toks + k) : rs[Kmax + 1 + k].g; };
  for (int k = tid; k < n; k += kConsumerThreads) {
    const int x = tok(k);
    bool acc;
    float pv, qv;
    if (x < 0 || x >= p.V) {
      atomicOr(&cs.bad, SV_DEV_BAD_TOKEN);
      acc = false;
      pv = qv = NAN;
    } else if (!sampled) {
      acc = (x == rs[k].g);
      pv = acc ? 1.0f : 0.0f;
      qv = 1.0f;
    } else {
      const RowStatS rt = rs[k], rd = rs[Kmax + 1 + k];
      // row sums are of 2^(x k - c(row max)): the drafted token's term uses the same offset
      pv = __fdiv_rn(exp2f(__fmaf_rn(rt.xval, kscale, -exp_offset(rt.m, kscale))), rt.s);
      qv = __fdiv_rn(exp2f(__fmaf_rn(rd.xval, kscale, -exp_offset(rd.m, kscale))), rd.s);
      const float u = philox_uniform_f(p.seed, static_cast<uint32_t>(k), static_cast<uint32_t>(rid), 0u, p.round);
      acc = u * qv < pv;
      if (qv == 0.0f) atomicOr(&cs.acc_flags, SV_FLAG_Q_ZERO);
    }
    if (p.out_p) p.out_p[static_cast<int64_t>(i) * Kmax + k] = pv;
    if (p.out_q) p.out_q[static_cast<int64_t>(i) * Kmax + k] = qv;
    if (!acc) atomicMin(&cs.a_min, k);
  }
  for (int k = n + tid; k < Kmax; k += kConsumerThreads) {
    if (p.out_p) p.out_p[static_cast<int64_t>(i) * Kmax + k] = NAN;
    if (p.out_q) p.out_q[static_cast<int64_t>(i) * Kmax + k] = NAN;
  }
  if (!sync()) return false;
  if (cs.bad) {
    if (tid == 0) atomicOr(p.status, cs.bad);
    write_invalid(p, i, tid, kConsumerThreads);
    if (tid == 0) {
      p.done[i] = 0;  // every stream unit of the request has counted itself
      if (sampled) {  // the request's draw units are scheduled: they find nothing to draw
        p.req[i].mode = kModeNone;
        __threadfence();
        st_release_u32(p.ready + i, tag + 1u);
      }
    }
    return true;
  }
  const int a = cs.a_min;

  // 3. emit: the accepted prefix (and, greedy, the target argmax at a); a sampled request's
  //    token at a is written by the pick
  for (int j = tid; j <= Kmax; j += kConsumerThreads) {
    if (j == a && sampled) continue;
    int v = -1;
    if (j < a) v = tok(j);
    else if (j == a) v = rs[a].g;
    p.out_tokens[static_cast<int64_t>(i) * (Kmax + 1) + j] = v;
  }
  if (tid == 0) {
    p.out_accept_len[i] = a;
    if (p.out_flags) p.out_flags[i] = static_cast<uint8_t>(cs.acc_flags);
    p.done[i] = 0;
    if (sampled) {
      ReqState st = {};
      st.mode = a < n ? kModeResidual : kModeBonus;
      st.a = a;
      st.flags = static_cast<int32_t>(cs.acc_flags);
      st.row_t = target_row(p, i, a);
      st.kscale = kscale;
      st.ct = exp_offset(rs[a].m, kscale);
      st.st = rs[a].s;
      st.inv_st = __frcp_rn(rs[a].s);
      if (a < n) {
        st.row_d = draft_row(p, i, a);
        st.cd = exp_offset(rs[Kmax + 1 + a].m, kscale);
        st.inv_sd = __frcp_rn(rs[Kmax + 1 + a].s);
      }
      st.u = philox_uniform_f(p.seed, static_cast<uint32_t>(a), static_cast<uint32_t>(rid), 1u, p.round);
      p.req[i] = st;
      __threadfence();
      st_release_u32(p.ready + i, tag + 1u);
    }
  }
  return true;
}

// ------------------------------------------------------------------------------------------
// the draw of request i (the four consumer warps); every draw unit's range sums are complete and
// visible (the producer acquired their count).  Returns false after an abort.
// ------------------------------------------------------------------------------------------
// Weight of vocabulary entry v of row a for the draw (target-only when !residual).
__device__ __forceinline__ float draw_weight(float tx, float dx, bool residual, const ReqState& st) {
  const float pv = ex2_approx(__fmaf_rn(tx, st.kscale, -st.ct));
  if (!residual) return pv;
  return fmaxf(0.0f, pv * st.inv_st - ex2_approx(__fmaf_rn(dx, st.kscale, -st.cd)) * st.inv_sd);
}

// Inverse-CDF pick inside one draw range by the consumer threads.  Thread t owns the contiguous
// entries [t*per, (t+1)*per) of the range.  Sets *y_out to the range-relative index of the first
// entry with cumsum > rem, or, if rounding keeps every partial sum at or below rem, the last entry
// with positive weight (-1 if none).
template <int DT>
__device__ bool block_pick(const char* trow, const char* drow, int c0, int len, bool residual, const ReqState& st,
                           float rem, ConsumerSmem& cs, ConsSync& sync, int tid, int* y_out) {
  constexpr int kElt = DT == SV_BF16 ? 2 : 4;
  // a draw range holds at most ceil(chunk / kDrawRanges) entries: kMaxPer per thread
  constexpr int kMaxPer = (kStageBytes / kElt / kDrawRanges + kConsumerThreads - 1) / kConsumerThreads;
  const int lane = tid & 31, warp = tid >> 5;
  const int per = (len + kConsumerThreads - 1) / kConsumerThreads;
  const int a = min(len, tid * per), b = min(len, a + per);
  const int cnt = b - a;
  // every load first (one round trip), then the weights
  float tx[kMaxPer], dx[kMaxPer], w[kMaxPer];
#pragma unroll
  for (int j = 0; j < kMaxPer; ++j) {
    tx[j] = j < cnt ? load_logit<DT>(trow, c0 + a + j) : -INFINITY;
    dx[j] = residual && j < cnt ? load_logit<DT>(drow, c0 + a + j) : -INFINITY;
  }
#pragma unroll
  for (int j = 0; j < kMaxPer; ++j) w[j] = j >= cnt ? 0.0f : draw_weight(tx[j], dx[j], residual, st);
  float sum = 0.0f;
  int lastpos = -1;
#pragma unroll
  for (int j = 0; j < kMaxPer; ++j) {
    sum += w[j];
    if (w[j] > 0.0f) lastpos = a + j;
  }
  float incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) cs.wsum[warp] = incl;
  if (tid == 0) {
    cs.pick_thread = kConsumerThreads;
    cs.last_pos = -1;
  }
  if (!sync()) return false;
  float excl = incl - sum;
  for (int v = 0; v < warp; ++v) excl += cs.wsum[v];
  if (cnt > 0 && sum > 0.0f && excl + sum > rem) atomicMin(&cs.pick_thread, tid);
  if (lastpos >= 0) atomicMax(&cs.last_pos, lastpos);
  if (!sync()) return false;
  if (tid == cs.pick_thread) {
    float run = excl;
    int y = -1;
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j) {
      run += w[j];
      if (y < 0 && w[j] > 0.0f && run > rem) y = a + j;
    }
    cs.last_pos = y >= 0 ? y : lastpos;
  }
  if (!sync()) return false;
  *y_out = cs.last_pos;
  return true;
}

// First index j in [0, cnt) whose running sum of w(j) (float, index order) exceeds thr, found by
// one warp.  Returns j (or the last j with w > 0 when rounding keeps every sum <= thr) and the sum
// of the entries before it in *before.
template <typename WF>
__device__ int warp_find(int cnt, float thr, WF w, float* before, int lane) {
  float run = 0.0f;
  int last_pos = -1;
  float before_last = 0.0f;
  for (int j0 = 0; j0 < cnt; j0 += 32) {
    const int j = j0 + lane;
    const float wj = j < cnt ? w(j) : 0.0f;
    float incl = wj;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, j < cnt && wj > 0.0f && run + incl > thr);
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, j < cnt && wj > 0.0f);
    if (hit) {
      const int src = __ffs(hit) - 1;
      *before = run + __shfl_sync(0xFFFFFFFFu, incl - wj, src);
      return j0 + src;
    }
    if (pos) {
      const int src = 31 - __clz(pos);
      last_pos = j0 + src;
      before_last = run + __shfl_sync(0xFFFFFFFFu, incl - wj, src);
    }
    run += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  *before = last_pos >= 0 ? before_last : 0.0f;
  return last_pos >= 0 ? last_pos : 0;
}

template <int DT>
__device__ bool pick_request(const VerifyParams& p, int i, ConsumerSmem& cs, ConsSync& sync, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  const int NC = p.nchunks, Kmax = p.Kmax;
  const int NE = NC * kDrawRanges;  // draw ranges of the request, in vocabulary order
  if (!sync()) return false;        // every warp is done with the shared state of the previous step
  if (tid == 0) {
    const ReqState* g = p.req + i;
    ReqState st;
    st.mode = __ldcg(&g->mode);
    st.a = __ldcg(&g->a);
    st.row_t = __ldcg(&g->row_t);
    st.row_d = __ldcg(&g->row_d);
    st.kscale = __ldcg(&g->kscale);
    st.ct = __ldcg(&g->ct);
    st.cd = __ldcg(&g->cd);
    st.inv_st = __ldcg(&g->inv_st);
    st.inv_sd = __ldcg(&g->inv_sd);
    st.st = __ldcg(&g->st);
    st.u = __ldcg(&g->u);
    st.flags = __ldcg(&g->flags);
    cs.st = st;
  }
  if (!sync()) return false;
  const ReqState st = cs.st;
  if (st.mode != kModeNone) {
    const bool residual_mode = st.mode == kModeResidual;
    const float* mass_r = p.mass + static_cast<int64_t>(i) * NE;
    const float* mass_p = p.mass_p + static_cast<int64_t>(i) * NE;
    const char* trow = row_ptr<DT>(p.target, st.row_t, p.t_row_stride);
    const char* drow = residual_mode ? row_ptr<DT>(p.draft, st.row_d, p.d_row_stride) : trow;

    // the crossing range (one warp)
    if (warp == 0) {
      auto r_at = [&](int e) { return __ldcg(mass_r + e); };
      auto p_at = [&](int e) { return __ldcg(mass_p + e); };
      int bonus = residual_mode ? 0 : 1;
      uint32_t flags = 0;
      float Z = 0.0f;
      if (!bonus) {
        for (int e = lane; e < NE; e += 32) Z += r_at(e);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xFFFFFFFFu, Z, o);
        if (!(Z > 0.0f)) {
          bonus = 1;  // residual mass 0 (not reachable in exact arithmetic): draw from p_a
          flags |= SV_FLAG_Z_ZERO;
        }
      }
      if (bonus) {
        Z = 0.0f;
        for (int e = lane; e < NE; e += 32) Z += p_at(e);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xFFFFFFFFu, Z, o);
      }
      const float thr = st.u * Z;
      float before = 0.0f;
      const int estar = bonus ? warp_find(NE, thr, p_at, &before, lane) : warp_find(NE, thr, r_at, &before, lane);
      if (lane == 0) {
        cs.chunk = estar;
        cs.base = before;
        cs.thr = thr;
        cs.bonus = bonus;
        cs.flags = flags;
      }
    }
    if (!sync()) return false;

    // the entry inside the crossing range (all consumer threads)
    const int estar = cs.chunk, cstar = estar / kDrawRanges;
    const bool residual = !cs.bonus;
    const int c0 = cstar * p.chunk_len;
    int lo, hi;
    draw_range(min(p.chunk_len, p.V - c0), kDrawRanges, estar - cstar * kDrawRanges, &lo, &hi);
    int y = -1;
    if (!block_pick<DT>(trow, residual ? drow : trow, c0 + lo, hi - lo, residual, st, cs.thr - cs.base, cs, sync,
                        tid, &y))
      return false;
    if (tid == 0) {
      if (y < 0) y = 0;  // only if every weight of the range flushed to zero; keep a valid token
      p.out_tokens[static_cast<int64_t>(i) * (Kmax + 1) + st.a] = c0 + lo + y;
      if (p.out_flags && cs.flags) p.out_flags[i] = static_cast<uint8_t>(st.flags | cs.flags);
    }
  }
  if (tid == 0) p.draw_done[i] = 0;  // every draw unit of the request has counted itself
  return true;
}

// ------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kVerifyThreads, 3) verify_kernel(const VerifyParams p) {
  constexpr int kElt = DT == SV_BF16 ? 2 : 4;
  constexpr int kVec = 16 / kElt;  // elements per 16-byte vector
  // -inf in every element of a padding vector
  constexpr uint32_t kPadWord = DT == SV_BF16 ? 0xFF80FF80u : 0xFF800000u;
  extern __shared__ __align__(128) unsigned char smem[];
  const int B = p.B, Kmax = p.Kmax, NC = p.nchunks, R = 2 * Kmax + 1;
  unsigned char* stages = smem;
  StageDesc* desc = reinterpret_cast<StageDesc*>(smem + kStages * kStageBytes);
  RowStatS* rs = reinterpret_cast<RowStatS*>(desc + kStages);     // [R]
  int* Stab = reinterpret_cast<int*>(rs + R);                      // [B + 1] stream-unit prefix
  uint16_t* Vtab = reinterpret_cast<uint16_t*>(Stab + B + 1);      // [B + 1] valid-request prefix
  uint16_t* Dtab = Vtab + B + 1;                                   // [B + 1] sampled-request prefix
  uint16_t* info = Dtab + B + 1;                                   // [B]
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t part_bar[kSlots];
  __shared__ __align__(8) uint64_t cons_bar;
  __shared__ ConsumerSmem cs;
  __shared__ int warp_tot[3][kVerifyThreads / 32];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int g_units = p.unit_tasks;
  // This call's tag: the draw-state flags it publishes hold tag + 1, so a flag left by an earlier
  // call (or any other stale value) never releases a draw unit.  The last CTA advances it.
  const uint32_t tag = *reinterpret_cast<volatile uint32_t*>(p.status + 3);

  // ---- prologue (all threads): barriers, per-request info and the unit table ----
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    for (int s = 0; s < kSlots; ++s) mbar_init(&part_bar[s], kConsumerWarps);
    mbar_init(&cons_bar, kConsumerWarps);
    abort_flag = 0;
    fence_proxy_async_smem();
  }
  {
    const int per = (B + kVerifyThreads - 1) / kVerifyThreads;
    const int lo = min(B, tid * per), hi = min(B, lo + per);
    int ls = 0, lv = 0, ld = 0;
    for (int i = lo; i < hi; ++i) {
      uint32_t bad;
      const uint16_t inf = request_info(p, i, &bad);
      info[i] = inf;
      if ((inf & kInfoInvalid) && i % static_cast<int>(gridDim.x) == static_cast<int>(blockIdx.x)) {
        atomicOr(p.status, bad);  // reported by one CTA; the request has no units
        write_invalid(p, i, 0, 1);
      }
      ls += (rows_of(inf) * NC + g_units - 1) / g_units;
      lv += is_valid(inf) ? 1 : 0;
      ld += has_draw(inf) ? 1 : 0;
    }
    int is = ls, iv = lv, id = ld;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ys = __shfl_up_sync(0xFFFFFFFFu, is, o), yv = __shfl_up_sync(0xFFFFFFFFu, iv, o),
                yd = __shfl_up_sync(0xFFFFFFFFu, id, o);
      if (lane >= o) {
        is += ys;
        iv += yv;
        id += yd;
      }
    }
    if (lane == 31) {
      warp_tot[0][warp] = is;
      warp_tot[1][warp] = iv;
      warp_tot[2][warp] = id;
    }
    __syncthreads();
    int bs = 0, bv = 0, bd = 0;
    for (int w = 0; w < warp; ++w) {
      bs += warp_tot[0][w];
      bv += warp_tot[1][w];
      bd += warp_tot[2][w];
    }
    int rs_ = bs + is - ls, rv_ = bv + iv - lv, rd_ = bd + id - ld;
    for (int i = lo; i < hi; ++i) {
      Stab[i] = rs_;
      Vtab[i] = static_cast<uint16_t>(rv_);
      Dtab[i] = static_cast<uint16_t>(rd_);
      rs_ += (rows_of(info[i]) * NC + g_units - 1) / g_units;
      rv_ += is_valid(info[i]) ? 1 : 0;
      rd_ += has_draw(info[i]) ? 1 : 0;
    }
    if (tid == kVerifyThreads - 1) {
      Stab[B] = bs + is;
      Vtab[B] = static_cast<uint16_t>(bv + iv);
      Dtab[B] = static_cast<uint16_t>(bd + id);
    }
  }
  __syncthreads();
  // Unit list: segment j (0 <= j < B + D3) holds the stream units of request j (j < B), the
  // combine unit of request j - D1, the draw units (one per chunk) of request j - D2 and the pick
  // unit of request j - D3 (those that exist).  The delays are in requests: about 1.25, 2 and 3
  // grid-widths of stream units.
  const int64_t S_tot = max(static_cast<int64_t>(Stab[B]), int64_t(1));
  const int64_t w_units = p.delay_units;
  auto delay = [&](int64_t units) {
    return static_cast<int>(min(static_cast<int64_t>(kMaxDelayRequests), (units * B + S_tot - 1) / S_tot));
  };
  const int D1 = 1 + delay(w_units + w_units / 4);
  const int D2 = D1 + 1 + delay(3 * w_units / 4);
  const int D3 = D2 + 1 + delay(w_units);
  auto clampB = [&](int j) { return min(max(j, 0), B); };
  auto seg_start = [&](int j) -> int64_t {
    return static_cast<int64_t>(Stab[min(j, B)]) + Vtab[clampB(j - D1)] + static_cast<int64_t>(NC) * Dtab[clampB(j - D2)] +
           Dtab[clampB(j - D3)];
  };
  const int NSEG = B + D3;
  const int64_t U = seg_start(NSEG);

  if (warp == kConsumerWarps) {
    // ---------------- producer warp: one lane takes units and issues the bulk copies ----------------
    if (lane == 0) {
      uint32_t it = 0;  // stages filled so far
      bool aborted = false;
      int jlo = 0;      // units are taken in increasing order: segments too
      int64_t u = blockIdx.x;
      int64_t nxt = static_cast<int64_t>(gridDim.x) + atomicAdd(p.status + 1, 1u);
      // Fill the next stage with descriptor d and (when src is given) a bulk copy of chunk c.
      auto fill = [&](const StageDesc& d, const char* src, int c) -> bool {
        const int stage = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        if (!mbar_wait_or_abort(&empty_bar[stage], ph ^ 1u, p.status, &abort_flag)) return false;
        desc[stage] = d;
        int nvec = 0;
        if (src != nullptr) {
          const int c0 = c * p.chunk_len;
          const ChunkSplit sp = split_chunk<kElt>(src, c0, min(p.chunk_len, p.V - c0));
          nvec = sp.nvec;
          if (nvec > 0) {
            mbar_arrive_expect_tx(&full_bar[stage], static_cast<uint32_t>(nvec) * 16u);
            bulk_g2s(stages + stage * kStageBytes, src + static_cast<int64_t>(c0 + sp.head) * kElt,
                     static_cast<uint32_t>(nvec) * 16u, &full_bar[stage]);
          }
        }
        if (nvec == 0) mbar_arrive(&full_bar[stage]);
        ++it;
        return true;
      };
      while (u < U && !aborted) {
        int lo = jlo, hi = NSEG - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (seg_start(mid) <= u) lo = mid;
          else hi = mid - 1;
        }
        jlo = lo;
        const int j = lo;
        int64_t o = u - seg_start(j);
        StageDesc d = {};
        d.writer = static_cast<int32_t>(u & (kConsumerWarps - 1));
        const int su = j < B ? Stab[j + 1] - Stab[j] : 0;
        const int ic = j - D1, id = j - D2, ip = j - D3;
        const int nc_ = (ic >= 0 && ic < B && is_valid(info[ic])) ? 1 : 0;
        const int nd = (id >= 0 && id < B && has_draw(info[id])) ? NC : 0;
        if (o < su) {
          // stream unit: tasks [t0, t1) of request j, task t = (row t / NC, chunk t % NC)
          const int i = j;
          const int n = info[i] & kInfoN;
          const int64_t tasks = static_cast<int64_t>(rows_of(info[i])) * NC;
          const int64_t t0 = o * g_units, t1 = min(t0 + g_units, tasks);
          for (int64_t t = t0; t < t1 && !aborted; ++t) {
            const int q = static_cast<int>(t / NC), c = static_cast<int>(t - static_cast<int64_t>(q) * NC);
            d.kind = kDescStream;
            d.i = i;
            d.q = q;
            d.c = c;
            d.flags = ((t == t0 || c == 0) ? kPieceFirst : 0) | ((t == t1 - 1 || c == NC - 1) ? kPieceLast : 0) |
                      (t == t1 - 1 ? kUnitLast : 0);
            d.ntasks = static_cast<int>(t1 - t0);
            const char* src = q <= n ? row_ptr<DT>(p.target, target_row(p, i, q), p.t_row_stride)
                                     : row_ptr<DT>(p.draft, draft_row(p, i, q - n - 1), p.d_row_stride);
            aborted = !fill(d, src, c);
          }
        } else if ((o -= su) < nc_) {
          // combine unit: once every stream unit of the request has counted itself
          const uint32_t total = static_cast<uint32_t>(rows_of(info[ic])) * static_cast<uint32_t>(NC);
          if (!flag_wait(p.done + ic, total, p.status, &abort_flag)) {
            aborted = true;
            break;
          }
          d.kind = kDescCombine;
          d.i = ic;
          aborted = !fill(d, nullptr, 0);
        } else if ((o -= nc_) < nd) {
          // draw unit: chunk o of row a, once the request's accept chain has published
          const int c = static_cast<int>(o);
          if (!flag_wait(p.ready + id, tag + 1u, p.status, &abort_flag)) {
            aborted = true;
            break;
          }
          const ReqState* g = p.req + id;
          d.i = id;
          d.c = c;
          d.mode = __ldcg(&g->mode);
          d.kscale = __ldcg(&g->kscale);
          d.ct = __ldcg(&g->ct);
          d.cd = __ldcg(&g->cd);
          d.inv_st = __ldcg(&g->inv_st);
          d.inv_sd = __ldcg(&g->inv_sd);
          d.row_t = __ldcg(&g->row_t);
          d.row_d = __ldcg(&g->row_d);
          if (d.mode == kModeNone) {
            d.kind = kDescSkip;
            aborted = !fill(d, nullptr, c);
          } else {
            d.kind = kDescDrawT;
            aborted = !fill(d, row_ptr<DT>(p.target, d.row_t, p.t_row_stride), c);
            if (!aborted && d.mode == kModeResidual) {
              d.kind = kDescDrawD;
              aborted = !fill(d, row_ptr<DT>(p.draft, d.row_d, p.d_row_stride), c);
            }
          }
        } else {
          // pick unit: once every draw unit of the request has counted itself
          if (!flag_wait(p.draw_done + ip, static_cast<uint32_t>(NC), p.status, &abort_flag)) {
            aborted = true;
            break;
          }
          d.kind = kDescPick;
          d.i = ip;
          aborted = !fill(d, nullptr, 0);
        }
        u = nxt;
        if (u < U) nxt = static_cast<int64_t>(gridDim.x) + atomicAdd(p.status + 1, 1u);
      }
      if (!aborted) {
        StageDesc d = {};
        d.kind = kDescEnd;
        aborted = !fill(d, nullptr, 0);
      }
      if (aborted) abort_flag = 1;
      // drain: every issued copy must land before the CTA may exit
      const uint32_t issued = it;
      for (uint32_t s = 0; s < kStages && s < issued; ++s) {
        const uint32_t last = issued - 1 - ((issued - 1 - s) % kStages);  // last fill of stage s
        mbar_wait(&full_bar[s], (last / kStages) & 1u, p.status);
      }
      // the last CTA to finish taking units resets the unit counter for the next call
      __threadfence();
      if (atomicAdd(p.status + 2, 1u) == gridDim.x - 1) {
        p.status[1] = 0;
        p.status[2] = 0;
        p.status[3] = tag + 1u;  // no producer reads a flag of this call any more
      }
    }
    return;
  }

  // ---------------- consumer warps (each runs on its own; no CTA-wide barrier) ----------------
  uint32_t it = 0;  // stages consumed (the same sequence in every consumer warp)
  uint32_t ev = 0;  // reduction events: stream pieces and draw units
  ConsSync sync{&cons_bar, 0u, p.status, &abort_flag};
  // lane 0 of a writer warp: a count to publish (red.release) once its stores have had a stage
  // to land; always before the warp could block
  uint32_t* pend_ptr = nullptr;
  uint32_t pend_val = 0;
  auto flush = [&]() {
    if (lane == 0 && pend_ptr != nullptr) {
      red_release_add(pend_ptr, pend_val);
      pend_ptr = nullptr;
    }
  };
  // Bounded wait of this warp for a barrier phase; publishes a pending count before blocking.
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    int ok = 1;
    if (lane == 0 && !mbar_test_wait(bar, parity)) {
      if (pend_ptr != nullptr) {
        red_release_add(pend_ptr, pend_val);
        pend_ptr = nullptr;
      }
      ok = mbar_wait_or_abort(bar, parity, p.status, &abort_flag) ? 1 : 0;
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok != 0;
  };
  auto release_stage = [&](int stage) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[stage]);
  };
  auto next_stage = [&](int* stage_out) -> bool {
    const int stage = it % kStages;
    const uint32_t ph = (it / kStages) & 1u;
    if (!warp_wait(&full_bar[stage], ph)) return false;
    ++it;
    *stage_out = stage;
    return true;
  };

  // per-piece state (the same in every warp: every warp sees every stage)
  const char* rowp = nullptr;
  bool sampled = false;
  int i_cur = 0, rec_row = 0, c_first = 0, g = -1, tok = -1, cx_piece = -1;
  float kscale = 0.0f, m = -INFINITY, sacc = 0.0f, xval_piece = NAN;
  float cofs = 0.0f;  // exp_offset(m, kscale) of the running max (sampled rows)

  for (;;) {
    int stage;
    if (!next_stage(&stage)) break;
    flush();  // the stores a pending count covers were issued a stage ago
    const StageDesc d = desc[stage];
    if (d.kind == kDescEnd) break;

    if (d.kind == kDescStream) {
      const int c = d.c;
      if (d.flags & kPieceFirst) {
        const uint16_t inf = info[d.i];
        const int n = inf & kInfoN;
        const bool is_target = d.q <= n;
        const int k = is_target ? d.q : d.q - n - 1;
        i_cur = d.i;
        rec_row = is_target ? k : Kmax + 1 + k;
        sampled = inf & kInfoSampled;
        kscale = sampled ? kscale_of(__ldg(p.temperature + d.i)) : 0.0f;
        tok = (tid == 0 && sampled && p.tokens != nullptr && k < n)
                  ? __ldg(p.tokens + static_cast<int64_t>(d.i) * p.tok_stride + k) : -1;
        rowp = is_target ? row_ptr<DT>(p.target, target_row(p, d.i, k), p.t_row_stride)
                         : row_ptr<DT>(p.draft, draft_row(p, d.i, k), p.d_row_stride);
        c_first = c;
        m = -INFINITY;
        sacc = 0.0f;
        g = -1;
        xval_piece = NAN;
        cx_piece = -1;
        cofs = 0.0f;
      }
      const int c0 = c * p.chunk_len;
      const int len = min(p.chunk_len, p.V - c0);
      const ChunkSplit sp = split_chunk<kElt>(rowp, c0, len);
      const int head = sp.head, nvec = sp.nvec, tail = sp.tail;
      const int v0 = c0 + head;         // vocabulary index of the first staged element
      const int te = v0 + nvec * kVec;  // first tail element
      const unsigned char* sb = stages + stage * kStageBytes;
      uint4 raw[kVecPerThread];
      if (nvec == kVecPerThread * kConsumerThreads) {  // a full chunk: no predicates
#pragma unroll
        for (int j = 0; j < kVecPerThread; ++j) raw[j] = lds128(sb + (tid + j * kConsumerThreads) * 16);
      } else {
#pragma unroll
        for (int j = 0; j < kVecPerThread; ++j) {
          const int v = tid + j * kConsumerThreads;
          raw[j] = v < nvec ? lds128(sb + v * 16) : make_uint4(kPadWord, kPadWord, kPadWord, kPadWord);
        }
      }
      if (tid == 0 && tok >= v0 && tok < te) {
        if constexpr (DT == SV_BF16)
          xval_piece = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(sb)[tok - v0]) << 16);
        else
          xval_piece = reinterpret_cast<const float*>(sb)[tok - v0];
        cx_piece = c;
      }
      release_stage(stage);

      // head / tail elements outside the 16-byte aligned interior: plain loads
      const bool has_head = tid < head, has_tail = tid < tail;
      const float head_x = has_head ? load_logit<DT>(rowp, c0 + tid) : -INFINITY;
      const float tail_x = has_tail ? load_logit<DT>(rowp, te + tid) : -INFINITY;
      if (tid == 0 && tok >= c0 && tok < c0 + len && !(tok >= v0 && tok < te)) {
        xval_piece = load_logit<DT>(rowp, tok);
        cx_piece = c;
      }

      if (!sampled) {
        // running first argmax (elements visited in increasing vocabulary order)
        if (has_head && (g < 0 || head_x > m)) {
          m = head_x;
          g = c0 + tid;
        }
#pragma unroll
        for (int j = 0; j < kVecPerThread; ++j) {
          const int v = tid + j * kConsumerThreads;
          if (v < nvec) {
            // the vector's first argmax by a pairwise tree (the left element wins ties), then one
            // merge into the running argmax: a short dependency chain per vector
            float x[kVec];
            if constexpr (DT == SV_BF16) {
              const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                x[2 * e] = bf16_lo(w[e]);
                x[2 * e + 1] = bf16_hi(w[e]);
              }
            } else {
              x[0] = __uint_as_float(raw[j].x);
              x[1] = __uint_as_float(raw[j].y);
              x[2] = __uint_as_float(raw[j].z);
              x[3] = __uint_as_float(raw[j].w);
            }
            int ix[kVec];
#pragma unroll
            for (int e = 0; e < kVec; ++e) ix[e] = e;
#pragma unroll
            for (int step = 1; step < kVec; step <<= 1)
#pragma unroll
              for (int e = 0; e + step < kVec; e += 2 * step)
                if (x[e + step] > x[e]) {
                  x[e] = x[e + step];
                  ix[e] = ix[e + step];
                }
            if (g < 0 || x[0] > m) {
              m = x[0];
              g = v0 + v * kVec + ix[0];
            }
          }
        }
        if (has_tail && (g < 0 || tail_x > m)) {
          m = tail_x;
          g = te + tid;
        }
      } else {
        // chunk max (packed bf16x2 max where possible), then rescale the running sum once
        float mc;
        if constexpr (DT == SV_BF16) {
          uint32_t w = bf16x2_max(bf16x2_max(raw[0].x, raw[0].y), bf16x2_max(raw[0].z, raw[0].w));
#pragma unroll
          for (int j = 1; j < kVecPerThread; ++j)
            w = bf16x2_max(w, bf16x2_max(bf16x2_max(raw[j].x, raw[j].y), bf16x2_max(raw[j].z, raw[j].w)));
          mc = fmaxf(bf16_lo(w), bf16_hi(w));
        } else {
          mc = -INFINITY;
#pragma unroll
          for (int j = 0; j < kVecPerThread; ++j)
            mc = fmaxf(mc, fmaxf(fmaxf(__uint_as_float(raw[j].x), __uint_as_float(raw[j].y)),
                                 fmaxf(__uint_as_float(raw[j].z), __uint_as_float(raw[j].w))));
        }
        mc = fmaxf(mc, fmaxf(head_x, tail_x));
        if (mc > m) {  // new running max: move the running sum to the new offset (exact)
          const float cnew = exp_offset(mc, kscale);
          sacc = (m == -INFINITY) ? 0.0f : sacc * pow2_nonpos(cofs - cnew);
          m = mc;
          cofs = cnew;
        }
        if (m != -INFINITY) {
          // terms 2^(x k - c): one fused multiply-add per logit, done on pairs of logits in
          // packed f32x2 registers; padding (-inf) adds 2^-inf = 0
          const f32x2 k2 = f2_pack(kscale, kscale), nc2 = f2_pack(-cofs, -cofs);
          f32x2 acc2[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};  // two independent chains
#pragma unroll
          for (int j = 0; j < kVecPerThread; ++j) {
            if constexpr (DT == SV_BF16) {
              const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                acc2[e & 1] = f2_add(acc2[e & 1], f2_exp2_offset(f2_pack(bf16_lo(w[e]), bf16_hi(w[e])), k2, nc2));
            } else {
              acc2[0] = f2_add(acc2[0], f2_exp2_offset(f2_pack(__uint_as_float(raw[j].x),
                                                               __uint_as_float(raw[j].y)), k2, nc2));
              acc2[1] = f2_add(acc2[1], f2_exp2_offset(f2_pack(__uint_as_float(raw[j].z),
                                                               __uint_as_float(raw[j].w)), k2, nc2));
            }
          }
          float a0, a1, a2, a3;
          f2_unpack(acc2[0], a0, a1);
          f2_unpack(acc2[1], a2, a3);
          float acc = (a0 + a1) + (a2 + a3);
          if (has_head) acc += ex2_approx(__fmaf_rn(head_x, kscale, -cofs));
          if (has_tail) acc += ex2_approx(__fmaf_rn(tail_x, kscale, -cofs));
          sacc += acc;
        }
      }

      if (d.flags & kPieceLast) {
        // the warp's part of the piece; the unit's writer warp merges the four parts and writes
        // the piece's records: the merged one at the first chunk, empty ones (max -inf, with the
        // drafted token's logit where it lies) at the others
        const uint32_t e = ev++;
        const int slot = static_cast<int>(e % kSlots);
        float pm, ps = 0.0f;
        int pg = -1;
        if (sampled) {
          // common offset of the warp's max, then plain sums (every rescale is a power of two)
          float M = m;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
          float sc = (m == -INFINITY) ? 0.0f : sacc * pow2_nonpos(cofs - exp_offset(M, kscale));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sc += __shfl_xor_sync(0xFFFFFFFFu, sc, o);
          pm = M;
          ps = sc;
        } else {
          float m3 = m;
          int g3 = g;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m3, o);
            const int g2 = __shfl_xor_sync(0xFFFFFFFFu, g3, o);
            merge_argmax(m3, g3, m2, g2);
          }
          pm = m3;
          pg = g3;
        }
        if (lane == 0) {
          RedPart& rp = cs.part[slot][warp];
          rp.v[0] = pm;
          rp.v[1] = ps;
          rp.v[2] = __int_as_float(pg);
          rp.v[3] = xval_piece;  // meaningful in warp 0 only
          rp.v[4] = __int_as_float(cx_piece);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&part_bar[slot]);
        if (warp == d.writer) {
          if (!warp_wait(&part_bar[slot], (e / kSlots) & 1u)) break;
          if (lane < kConsumerWarps) {
            const RedPart& rp = cs.part[slot][lane];
            float mm = rp.v[0];
            float ss = rp.v[1];
            int gg = __float_as_int(rp.v[2]);
            const float xv = cs.part[slot][0].v[3];
            const int cxp = __float_as_int(cs.part[slot][0].v[4]);
            const unsigned kMask = (1u << kConsumerWarps) - 1u;
            if (sampled) {
              float MM = mm;
#pragma unroll
              for (int o = kConsumerWarps / 2; o > 0; o >>= 1) MM = fmaxf(MM, __shfl_xor_sync(kMask, MM, o));
              float s2 = (mm == -INFINITY) ? 0.0f : ss * pow2_nonpos(exp_offset(mm, kscale) - exp_offset(MM, kscale));
#pragma unroll
              for (int o = kConsumerWarps / 2; o > 0; o >>= 1) s2 += __shfl_xor_sync(kMask, s2, o);
              mm = MM;
              ss = MM == -INFINITY ? 0.0f : s2;
              gg = -1;
            } else {
#pragma unroll
              for (int o = kConsumerWarps / 2; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(kMask, mm, o);
                const int g2 = __shfl_xor_sync(kMask, gg, o);
                merge_argmax(mm, gg, m2, g2);
              }
              ss = 0.0f;
            }
            if (lane == 0) {
              ChunkRecord* rec_base = p.rec + (static_cast<int64_t>(i_cur) * R + rec_row) * NC;
              __stcg(reinterpret_cast<float4*>(rec_base + c_first),
                     make_float4(mm, ss, __int_as_float(gg), cxp == c_first ? xv : NAN));
              for (int cc = c_first + 1; cc <= c; ++cc)
                __stcg(reinterpret_cast<float4*>(rec_base + cc),
                       make_float4(-INFINITY, 0.0f, __int_as_float(-1), cxp == cc ? xv : NAN));
              if (d.flags & kUnitLast) {  // every record of the unit was written by this lane
                pend_ptr = p.done + i_cur;
                pend_val = static_cast<uint32_t>(d.ntasks);
              }
            }
          }
          __syncwarp();
        }
      }
    } else if (d.kind == kDescDrawT) {
      // ---- draw unit: chunk c of row a; residual mode also holds the draft chunk in the next stage
      const bool residual = d.mode == kModeResidual;
      const int i = d.i, c = d.c;
      int stage_d = stage;
      if (residual && !next_stage(&stage_d)) break;
      const ReqState st = {d.mode, 0, d.row_t, d.row_d, d.kscale, d.ct, d.cd, d.inv_st, d.inv_sd, 0.0f, 0.0f, 0};
      const char* trow = row_ptr<DT>(p.target, d.row_t, p.t_row_stride);
      const char* drow = residual ? row_ptr<DT>(p.draft, d.row_d, p.d_row_stride) : trow;
      const int c0 = c * p.chunk_len;
      const int len = min(p.chunk_len, p.V - c0);
      const ChunkSplit spt = split_chunk<kElt>(trow, c0, len);
      const ChunkSplit spd = residual ? split_chunk<kElt>(drow, c0, len) : spt;
      const unsigned char* sbt = stages + stage * kStageBytes;
      const unsigned char* sbd = stages + stage_d * kStageBytes;
      constexpr int kFull = kVecPerThread * kConsumerThreads;
      float accr[kDrawRanges], accp[kDrawRanges];
      if (spt.nvec == kFull && spd.nvec == kFull) {
        // full chunks: range r is every thread's vector r
#pragma unroll
        for (int j = 0; j < kVecPerThread; ++j) {
          const uint4 wt = lds128(sbt + (tid + j * kConsumerThreads) * 16);
          const uint4 wd = residual ? lds128(sbd + (tid + j * kConsumerThreads) * 16) : wt;
          const uint32_t t4[4] = {wt.x, wt.y, wt.z, wt.w}, d4[4] = {wd.x, wd.y, wd.z, wd.w};
          float sr = 0.0f, sp = 0.0f;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float tx[2], dx[2];
            if constexpr (DT == SV_BF16) {
              tx[0] = bf16_lo(t4[e]);
              tx[1] = bf16_hi(t4[e]);
              dx[0] = bf16_lo(d4[e]);
              dx[1] = bf16_hi(d4[e]);
            } else {
              tx[0] = __uint_as_float(t4[e]);
              dx[0] = __uint_as_float(d4[e]);
            }
#pragma unroll
            for (int h = 0; h < (DT == SV_BF16 ? 2 : 1); ++h) {
              const float pv = ex2_approx(__fmaf_rn(tx[h], st.kscale, -st.ct));
              sp += pv;
              if (residual)
                sr += fmaxf(0.0f, pv * st.inv_st - ex2_approx(__fmaf_rn(dx[h], st.kscale, -st.cd)) * st.inv_sd);
            }
          }
          accr[j] = sr;
          accp[j] = sp;
        }
      } else {
        // any other chunk: warp w sums ranges 2w and 2w + 1 element by element (the other ranges
        // of its part stay zero)
#pragma unroll
        for (int r = 0; r < kDrawRanges; ++r) accr[r] = accp[r] = 0.0f;
#pragma unroll
        for (int r = 0; r < kDrawRanges; ++r) {
          if (r / 2 != warp) continue;
          int lo, hi;
          draw_range(len, kDrawRanges, r, &lo, &hi);
          float sr = 0.0f, sp = 0.0f;
          for (int e = lo + lane; e < hi; e += 32) {
            const float tx = staged_elem<DT>(sbt, trow, c0, e, spt.head, spt.nvec);
            const float pv = ex2_approx(__fmaf_rn(tx, st.kscale, -st.ct));
            sp += pv;
            if (residual) {
              const float dx = staged_elem<DT>(sbd, drow, c0, e, spd.head, spd.nvec);
              sr += fmaxf(0.0f, pv * st.inv_st - ex2_approx(__fmaf_rn(dx, st.kscale, -st.cd)) * st.inv_sd);
            }
          }
          accr[r] = sr;
          accp[r] = sp;
        }
      }
      release_stage(stage);
      if (residual) release_stage(stage_d);
#pragma unroll
      for (int r = 0; r < kDrawRanges; ++r) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          accr[r] += __shfl_xor_sync(0xFFFFFFFFu, accr[r], o);
          accp[r] += __shfl_xor_sync(0xFFFFFFFFu, accp[r], o);
        }
      }
      const uint32_t e = ev++;
      const int slot = static_cast<int>(e % kSlots);
      if (lane == 0) {
        RedPart& rp = cs.part[slot][warp];
#pragma unroll
        for (int r = 0; r < kDrawRanges; ++r) {
          rp.v[r] = accr[r];
          rp.v[kDrawRanges + r] = accp[r];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&part_bar[slot]);
      if (warp == d.writer) {
        if (!warp_wait(&part_bar[slot], (e / kSlots) & 1u)) break;
        if (lane == 0) {
          float* mr = p.mass + (static_cast<int64_t>(i) * NC + c) * kDrawRanges;
          float* mp = p.mass_p + (static_cast<int64_t>(i) * NC + c) * kDrawRanges;
#pragma unroll
          for (int r = 0; r < kDrawRanges; ++r) {
            float sr = 0.0f, sp = 0.0f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
              sr += cs.part[slot][w].v[r];
              sp += cs.part[slot][w].v[kDrawRanges + r];
            }
            if (residual) mr[r] = sr;
            mp[r] = sp;
          }
          pend_ptr = p.draw_done + i;
          pend_val = 1u;
        }
        __syncwarp();
      }
    } else if (d.kind == kDescSkip) {
      // a draw unit of a request with nothing to draw (its input was invalid)
      release_stage(stage);
      if (warp == d.writer && lane == 0) {
        pend_ptr = p.draw_done + d.i;
        pend_val = 1u;
      }
    } else if (d.kind == kDescCombine) {
      release_stage(stage);
      flush();
      if (!combine_request(p, d.i, rs, cs, sync, tid, tag)) break;
    } else if (d.kind == kDescPick) {
      release_stage(stage);
      flush();
      if (!pick_request<DT>(p, d.i, cs, sync, tid)) break;
    } else {
      release_stage(stage);  // not reached: a lone draft chunk always follows its target chunk
    }
  }
  flush();
}

// Per-device launch set-up, done once per device (and dtype) under a lock: function attributes
// belong to the device that was current when they were set.
constexpr int kMaxDevices = 64;
struct DeviceLaunchState {
  bool ready[2];  // attributes of the bf16 / fp32 kernels set
  int num_sms;
};
DeviceLaunchState g_dev_state[kMaxDevices] = {};
std::mutex g_dev_mu;

template <int DT>
cudaError_t device_setup(int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const int di = DT == SV_BF16 ? 0 : 1;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceLaunchState& ds = g_dev_state[dev];
  if (!ds.ready[di]) {
    if (ds.num_sms == 0 && (e = cudaDeviceGetAttribute(&ds.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    const size_t max_dyn = verify_smem_bytes(SV_MAX_BATCH, SV_MAX_DRAFT);
    if ((e = cudaFuncSetAttribute(verify_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(max_dyn))) != cudaSuccess)
      return e;
    ds.ready[di] = true;
  }
  *num_sms = ds.num_sms;
  return cudaSuccess;
}

template <int DT>
cudaError_t launch_verify_t(VerifyParams p, cudaStream_t stream) {
  cudaError_t e;
  int num_sms = 0;
  if ((e = device_setup<DT>(&num_sms)) != cudaSuccess) return e;
  const size_t dyn = verify_smem_bytes(p.B, p.Kmax);
  int nb = 0;  // resident CTAs per SM at this shared-memory size
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, verify_kernel<DT>, kVerifyThreads, dyn)) != cudaSuccess)
    return e;
  const int64_t cap = static_cast<int64_t>(num_sms) * (nb > 0 ? nb : 1);
  // Upper bound of the stream tasks (the kept lengths and temperatures live on the device).
  const bool drafts = p.draft != nullptr && (p.temperature != nullptr || p.tokens == nullptr);
  const int64_t rows = static_cast<int64_t>(p.B) * (drafts ? 2 * p.Kmax + 1 : p.Kmax + 1);
  const int64_t tasks = rows * p.nchunks;
  // Units of a few chunks: enough units per CTA (~24) to balance the grid, few piece reductions.
  const int64_t g = std::max<int64_t>(1, std::min<int64_t>(4, tasks / (cap * 24)));
  const int64_t units =
      (tasks + g - 1) / g + p.B + (p.temperature != nullptr ? static_cast<int64_t>(p.B) * (p.nchunks + 1) : 0);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cap, units)));
  p.unit_tasks = static_cast<int32_t>(g);
  p.delay_units = grid;
  prof_before(SV_KERNEL_VERIFY, stream);
  verify_kernel<DT><<<grid, kVerifyThreads, dyn, stream>>>(p);
  prof_after(SV_KERNEL_VERIFY, stream);
  return cudaGetLastError();
}

}  // namespace

// Fixed 16 KB chunks: every chunk but the last of a row is full (no predicated loads).
void vocab_tiling(int V, sv_dtype dt, int* chunk_len, int* nchunks) {
  const int elt = dt == SV_BF16 ? 2 : 4;
  const int cl = kStageBytes / elt;
  *chunk_len = cl;
  *nchunks = (V + cl - 1) / cl;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

VerifyLayout verify_layout(int B, int Kmax, int nchunks) {
  VerifyLayout L;
  const size_t R = 2 * static_cast<size_t>(Kmax) + 1;
  size_t off = 0;
  L.status = off;
  off = align256(off + 256);
  L.counters = off;  // at a fixed place and size: calls of any batch size share the same zeroed counters
  off = align256(off + 3 * sizeof(uint32_t) * static_cast<size_t>(SV_MAX_BATCH));
  L.req = off;
  off = align256(off + sizeof(ReqState) * B);
  L.mass = off;
  off = align256(off + sizeof(float) * B * static_cast<size_t>(nchunks) * kDrawRanges);
  L.mass_p = off;
  off = align256(off + sizeof(float) * B * static_cast<size_t>(nchunks) * kDrawRanges);
  L.rec = off;
  off = align256(off + sizeof(ChunkRecord) * B * R * static_cast<size_t>(nchunks));
  L.total = off;
  return L;
}

int launch_verify(const VerifyParams& p, sv_dtype dt, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return static_cast<int>(dt == SV_BF16 ? launch_verify_t<SV_BF16>(p, s) : launch_verify_t<SV_F32>(p, s));
}

}  // namespace sv
