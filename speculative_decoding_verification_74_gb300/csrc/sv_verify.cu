// Verification kernels of libsv.
//
// row_stats  One streaming pass over every logit row a round needs.  A persistent grid walks
//            (request, row, vocabulary chunk) tasks in request-major order; per CTA one
//            producer lane issues 1-D bulk copies (cp.async.bulk) of 16 KB chunks into a
//            4-stage shared-memory ring and eight consumer warps reduce each chunk to
//            {max, sum 2^((x-max) log2(e)/T), first argmax, logit at the drafted token}.
//            The CTA that finishes a request's last chunk (atomic counter, no waiting)
//            merges its chunks and runs the accept chain: the greedy test x_k == argmax,
//            or the rejection test u_k q_k(x_k) < p_k(x_k), first rejection = accepted
//            length (AngelSpec explainer, "MTP: fix position 2 and 3", eq. L_e2e: one
//            rejection voids every later position; AngelSpec release article, "Why one
//            universal drafter underperforms": rejection-sampling verification in one pass).
// sample     For sampled requests: the draw at the accepted length a, from
//            norm(max(0, p_a - q_a)) after a rejection or from p_n when every drafted token
//            was accepted (the bonus row), by inverse CDF in vocabulary order.  Residual
//            requests re-read their two rows once (chunk sums, then a scan of the chunk that
//            holds the crossing); bonus requests reuse row_stats' chunk sums and scan one
//            chunk.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr double kLog2e = 1.4426950408889634074;

// request info, one uint16 per request, cached in shared memory by every row_stats CTA
constexpr uint16_t kInfoN = 0x3FF;
constexpr uint16_t kInfoNeedDraft = 1u << 10;
constexpr uint16_t kInfoSampled = 1u << 11;
constexpr uint16_t kInfoInvalid = 1u << 12;

enum : int { kSkip = 0, kLoad = 1, kDummy = 2 };

__device__ __forceinline__ float kscale_of(float T) {
  return static_cast<float>(kLog2e / static_cast<double>(T));
}

__device__ __forceinline__ int slot_kind(uint16_t info, int r, int c, int Kmax) {
  if (info & kInfoInvalid) return (r == 0 && c == 0) ? kDummy : kSkip;
  const int n = info & kInfoN;
  if (r <= Kmax) return r <= n ? kLoad : kSkip;
  return ((info & kInfoNeedDraft) && (r - Kmax - 1) < n) ? kLoad : kSkip;
}

__device__ __forceinline__ uint32_t expected_tasks(uint16_t info, int nchunks) {
  if (info & kInfoInvalid) return 1u;
  const uint32_t n = info & kInfoN;
  const uint32_t rows = n + 1u + ((info & kInfoNeedDraft) ? n : 0u);
  return rows * static_cast<uint32_t>(nchunks);
}

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

// A chunk [c0, c0 + len) of a row split into a head of plain loads, a 16-byte aligned interior of
// nvec vectors (bulk-copied) and a tail of plain loads; rows may start at any element.
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

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// ------------------------------------------------------------------------------------------
// per-request validation (every row_stats CTA computes the same info; CTA 0 reports errors)
// ------------------------------------------------------------------------------------------
__device__ uint16_t request_info(const VerifyParams& p, int i, uint32_t* bad_out) {
  const int n = p.keep_len ? __ldg(p.keep_len + i) : p.Kmax;
  const float T = p.temperature ? __ldg(p.temperature + i) : 0.0f;
  uint32_t bad = 0;
  if (n < 0 || n > p.Kmax) bad |= SV_DEV_BAD_KEEP_LEN;
  if (!(T >= 0.0f) || isinf(T)) bad |= SV_DEV_BAD_TEMPERATURE;
  const bool sampled = T > 0.0f;
  const bool need_draft = (sampled || p.tokens == nullptr) && n > 0;  // n == 0: bonus row only
  if (sampled && n > 0 && p.tokens == nullptr) bad |= SV_DEV_BAD_TOKEN;
  if (need_draft && p.draft == nullptr) bad |= SV_DEV_NO_DRAFT_ROWS;
  if (!bad && p.t_off && (__ldg(p.t_off + i + 1) - __ldg(p.t_off + i) < n + 1 || __ldg(p.t_off + i) < 0))
    bad |= SV_DEV_BAD_OFFSETS;
  if (!bad && need_draft && p.d_off &&
      (__ldg(p.d_off + i + 1) - __ldg(p.d_off + i) < n || __ldg(p.d_off + i) < 0))
    bad |= SV_DEV_BAD_OFFSETS;
  *bad_out = bad;
  if (bad) return kInfoInvalid;
  return static_cast<uint16_t>(n | (need_draft ? kInfoNeedDraft : 0) | (sampled ? kInfoSampled : 0));
}

__device__ void write_invalid(const VerifyParams& p, int i, int tid, int nthreads) {
  for (int j = tid; j <= p.Kmax; j += nthreads) p.out_tokens[static_cast<int64_t>(i) * (p.Kmax + 1) + j] = -1;
  for (int j = tid; j < p.Kmax; j += nthreads) {
    if (p.out_p) p.out_p[static_cast<int64_t>(i) * p.Kmax + j] = NAN;
    if (p.out_q) p.out_q[static_cast<int64_t>(i) * p.Kmax + j] = NAN;
  }
  if (tid == 0) {
    p.out_accept_len[i] = -1;
    if (p.out_flags) p.out_flags[i] = SV_FLAG_INVALID;
    p.req[i].mode = kModeNone;
  }
}

// ------------------------------------------------------------------------------------------
// combine: merge a request's chunk records into row statistics, run the accept chain, emit.
// Runs on the 256 consumer threads of the CTA that completed the request.
// ------------------------------------------------------------------------------------------
struct CombineSmem {
  int a_min;
  uint32_t flags;
  uint32_t bad;
};

__device__ void combine_request(const VerifyParams& p, int i, uint16_t info, int tid, CombineSmem* cs) {
  const int lane = tid & 31, warp = tid >> 5;
  const int Kmax = p.Kmax, NC = p.nchunks, R = p.rows_per_req;
  if (info & kInfoInvalid) {
    write_invalid(p, i, tid, kConsumerThreads);
    if (tid == 0) p.cnt_stats[i] = 0;
    named_bar(1, kConsumerThreads);
    return;
  }
  const int n = info & kInfoN;
  const bool sampled = info & kInfoSampled;
  const bool need_draft = info & kInfoNeedDraft;
  const float T = p.temperature ? __ldg(p.temperature + i) : 0.0f;
  const float kscale = sampled ? kscale_of(T) : 0.0f;
  const int nrows = n + 1 + (need_draft ? n : 0);
  const int rid = p.request_ids ? __ldg(p.request_ids + i) : i;

  // 1. row statistics
  for (int q = warp; q < nrows; q += kConsumerWarps) {
    const int r = q <= n ? q : Kmax + 1 + (q - n - 1);
    const ChunkRecord* rr = p.rec + (static_cast<int64_t>(i) * R + r) * NC;
    float m = -INFINITY;
    int g = -1;
    for (int c = lane; c < NC; c += 32) {
      const ChunkRecord rc = ld_record(rr + c);
      if (sampled) m = fmaxf(m, rc.m);
      else merge_argmax(m, g, rc.m, rc.g);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
      const int g2 = __shfl_xor_sync(0xFFFFFFFFu, g, o);
      if (sampled) m = fmaxf(m, m2);
      else merge_argmax(m, g, m2, g2);
    }
    double s = 0.0;
    if (sampled && m != -INFINITY) {
      for (int c = lane; c < NC; c += 32) {
        const ChunkRecord rc = ld_record(rr + c);
        if (rc.m != -INFINITY) s += static_cast<double>(rc.s) * static_cast<double>(exp2f((rc.m - m) * kscale));
      }
      s = warp_sum_d(s);
    }
    if (lane == 0) {
      RowStat rs;
      rs.s = s;
      rs.m = m;
      rs.g = g;
      p.rowstat[static_cast<int64_t>(i) * R + r] = rs;
    }
  }
  if (tid == 0) {
    cs->a_min = n;
    cs->flags = 0;
    cs->bad = 0;
  }
  named_bar(1, kConsumerThreads);

  // 2. accept tests (each position independently; the first rejection is a min-reduction)
  const RowStat* rs = p.rowstat + static_cast<int64_t>(i) * R;
  for (int k = tid; k < n; k += kConsumerThreads) {
    const int x = p.tokens ? __ldg(p.tokens + static_cast<int64_t>(i) * p.tok_stride + k) : rs[Kmax + 1 + k].g;
    bool acc;
    double pv, qv;
    if (x < 0 || x >= p.V) {
      atomicOr(&cs->bad, SV_DEV_BAD_TOKEN);
      acc = false;
      pv = qv = NAN;
    } else if (!sampled) {
      acc = (x == rs[k].g);
      pv = acc ? 1.0 : 0.0;
      qv = 1.0;
    } else {
      const int cx = x / p.chunk_len;
      const float xt = ld_record(p.rec + (static_cast<int64_t>(i) * R + k) * NC + cx).xval;
      const float xd = ld_record(p.rec + (static_cast<int64_t>(i) * R + Kmax + 1 + k) * NC + cx).xval;
      const RowStat rt = rs[k], rd = rs[Kmax + 1 + k];
      pv = exp2(static_cast<double>(xt - rt.m) * static_cast<double>(kscale)) / rt.s;
      qv = exp2(static_cast<double>(xd - rd.m) * static_cast<double>(kscale)) / rd.s;
      const double u = philox_uniform(p.seed, static_cast<uint32_t>(k), static_cast<uint32_t>(rid), 0u, p.round);
      acc = u * qv < pv;
      if (qv == 0.0) atomicOr(&cs->flags, SV_FLAG_Q_ZERO);
    }
    if (p.out_p) p.out_p[static_cast<int64_t>(i) * Kmax + k] = static_cast<float>(pv);
    if (p.out_q) p.out_q[static_cast<int64_t>(i) * Kmax + k] = static_cast<float>(qv);
    if (!acc) atomicMin(&cs->a_min, k);
  }
  for (int k = n + tid; k < Kmax; k += kConsumerThreads) {
    if (p.out_p) p.out_p[static_cast<int64_t>(i) * Kmax + k] = NAN;
    if (p.out_q) p.out_q[static_cast<int64_t>(i) * Kmax + k] = NAN;
  }
  named_bar(1, kConsumerThreads);

  // 3. emit
  if (cs->bad) {
    if (tid == 0) atomicOr(p.status, cs->bad);
    write_invalid(p, i, tid, kConsumerThreads);
  } else {
    const int a = cs->a_min;
    for (int j = tid; j <= Kmax; j += kConsumerThreads) {
      int v = -1;
      if (j < a) v = p.tokens ? __ldg(p.tokens + static_cast<int64_t>(i) * p.tok_stride + j) : rs[Kmax + 1 + j].g;
      else if (j == a && !sampled) v = rs[a].g;
      p.out_tokens[static_cast<int64_t>(i) * (Kmax + 1) + j] = v;
    }
    if (tid == 0) {
      p.out_accept_len[i] = a;
      if (p.out_flags) p.out_flags[i] = static_cast<uint8_t>(cs->flags);
      ReqState st;
      st.mode = kModeNone;
      st.a = a;
      st.flags = static_cast<int32_t>(cs->flags);
      st.pad = 0;
      if (sampled) {
        st.mode = a < n ? kModeResidual : kModeBonus;
        st.row_t = target_row(p, i, a);
        st.row_d = a < n ? draft_row(p, i, a) : 0;
        st.kscale = kscale;
        st.mt = rs[a].m;
        st.st = rs[a].s;
        st.inv_st = static_cast<float>(1.0 / rs[a].s);
        st.md = a < n ? rs[Kmax + 1 + a].m : 0.0f;
        st.inv_sd = a < n ? static_cast<float>(1.0 / rs[Kmax + 1 + a].s) : 0.0f;
        st.rec_row_t = i * R + a;
        st.u = philox_uniform(p.seed, static_cast<uint32_t>(a), static_cast<uint32_t>(rid), 1u, p.round);
      } else {
        st.row_t = st.row_d = 0;
        st.kscale = st.mt = st.md = st.inv_st = st.inv_sd = 0.0f;
        st.rec_row_t = 0;
        st.st = st.u = 0.0;
      }
      p.req[i] = st;
    }
  }
  if (tid == 0) p.cnt_stats[i] = 0;
  named_bar(1, kConsumerThreads);
}

// ------------------------------------------------------------------------------------------
// row_stats kernel
// ------------------------------------------------------------------------------------------
struct StatsRed {
  float m[kConsumerWarps];
  float s[kConsumerWarps];
  int g[kConsumerWarps];
  int last;
  int stop;  // uniform copy of the abort flag, written before a barrier
};

template <int DT>
__global__ void __launch_bounds__(kStatsThreads, 3) row_stats_kernel(const VerifyParams p) {
  constexpr int kElt = DT == SV_BF16 ? 2 : 4;
  constexpr int kVec = 16 / kElt;  // elements per 16-byte vector
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* stages = smem;
  uint16_t* info = reinterpret_cast<uint16_t*>(smem + kStages * kStageBytes);
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ StatsRed red[2];
  __shared__ CombineSmem cs;
  __shared__ volatile int abort_flag;
  __shared__ float xval_s;

  const int tid = threadIdx.x;
  const int B = p.B, Kmax = p.Kmax, NC = p.nchunks, R = p.rows_per_req;

  // prologue: request table + barriers
  for (int i = tid; i < B; i += blockDim.x) {
    uint32_t bad;
    info[i] = request_info(p, i, &bad);
    if (bad && blockIdx.x == 0) atomicOr(p.status, bad);
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    abort_flag = 0;
    fence_proxy_async_smem();
  }
  __syncthreads();

  const int64_t per_req = static_cast<int64_t>(R) * NC;
  const int64_t total = per_req * B;

  if (tid >= kConsumerThreads) {
    // ---------------- producer warp: one lane issues the bulk copies ----------------
    if (tid == kConsumerThreads) {
      const uint64_t pol = policy_evict_first();
      uint32_t it = 0;
      for (int64_t s = blockIdx.x; s < total; s += gridDim.x) {
        const int i = static_cast<int>(s / per_req);
        const int rem = static_cast<int>(s - static_cast<int64_t>(i) * per_req);
        const int r = rem / NC, c = rem - (rem / NC) * NC;
        const int kind = slot_kind(info[i], r, c, Kmax);
        if (kind == kSkip) continue;
        if (abort_flag) break;
        const int stage = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        ++it;
        if (!mbar_wait(&empty_bar[stage], ph ^ 1u, p.status)) {
          abort_flag = 1;
          break;
        }
        if (kind == kDummy) {
          mbar_arrive(&full_bar[stage]);
          continue;
        }
        const int64_t row = r <= Kmax ? target_row(p, i, r) : draft_row(p, i, r - Kmax - 1);
        const char* src = r <= Kmax ? row_ptr<DT>(p.target, row, p.t_row_stride)
                                    : row_ptr<DT>(p.draft, row, p.d_row_stride);
        const int c0 = c * p.chunk_len;
        const ChunkSplit sp = split_chunk<kElt>(src, c0, min(p.chunk_len, p.V - c0));
        if (sp.nvec == 0) {
          mbar_arrive(&full_bar[stage]);
        } else {
          mbar_arrive_expect_tx(&full_bar[stage], static_cast<uint32_t>(sp.nvec) * 16u);
          bulk_g2s(stages + stage * kStageBytes, src + static_cast<int64_t>(c0 + sp.head) * kElt,
                   static_cast<uint32_t>(sp.nvec) * 16u, &full_bar[stage], pol);
        }
      }
      // drain: every issued copy must land before the CTA may exit
      const uint32_t issued = it;
      for (uint32_t s = 0; s < kStages && s < issued; ++s) {
        const uint32_t last = issued - 1 - ((issued - 1 - s) % kStages);  // last issue on stage s
        mbar_wait(&full_bar[s], (last / kStages) & 1u, p.status);
      }
    }
    pdl_trigger();
    return;
  }

  // ---------------- consumer warps ----------------
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t it = 0;
  int buf = 0;
  for (int64_t s = blockIdx.x; s < total; s += gridDim.x) {
    const int i = static_cast<int>(s / per_req);
    const int rem = static_cast<int>(s - static_cast<int64_t>(i) * per_req);
    const int r = rem / NC, c = rem - (rem / NC) * NC;
    const uint16_t inf = info[i];
    const int kind = slot_kind(inf, r, c, Kmax);
    if (kind == kSkip) continue;
    const int stage = it % kStages;
    const uint32_t ph = (it / kStages) & 1u;
    ++it;

    const bool sampled = inf & kInfoSampled;
    const int n = inf & kInfoN;
    const int k_row = r <= Kmax ? r : r - Kmax - 1;
    float kscale = 0.0f;
    if (sampled) kscale = kscale_of(__ldg(p.temperature + i));
    int tok = -1;
    if (tid == 0 && kind == kLoad && sampled && k_row < n)
      tok = __ldg(p.tokens + static_cast<int64_t>(i) * p.tok_stride + k_row);

    const int c0 = c * p.chunk_len;
    const int len = kind == kLoad ? min(p.chunk_len, p.V - c0) : 0;
    const char* rowp = nullptr;
    if (kind == kLoad) {
      const int64_t row = r <= Kmax ? target_row(p, i, r) : draft_row(p, i, r - Kmax - 1);
      rowp = r <= Kmax ? row_ptr<DT>(p.target, row, p.t_row_stride) : row_ptr<DT>(p.draft, row, p.d_row_stride);
    }
    const ChunkSplit sp = kind == kLoad ? split_chunk<kElt>(rowp, c0, len) : ChunkSplit{0, 0, 0};
    const int head = sp.head, nvec = sp.nvec, tail = sp.tail;
    const int v0 = c0 + head;                      // vocabulary index of the first staged element
    const int t0 = v0 + nvec * kVec;               // first tail element

    // A timed-out wait does not leave the loop here: every consumer thread must reach the same
    // named barriers; the abort decision is taken uniformly after them.
    if (!mbar_wait(&full_bar[stage], ph, p.status)) abort_flag = 1;
    const unsigned char* sb = stages + stage * kStageBytes;
    uint4 raw[kVecPerThread];
#pragma unroll
    for (int j = 0; j < kVecPerThread; ++j) {
      const int v = tid + j * kConsumerThreads;
      raw[j] = v < nvec ? lds128(sb + v * 16) : make_uint4(0, 0, 0, 0);
    }
    float xval = NAN;
    if (tid == 0 && tok >= v0 && tok < t0) {
      if constexpr (DT == SV_BF16)
        xval = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(sb)[tok - v0]) << 16);
      else
        xval = reinterpret_cast<const float*>(sb)[tok - v0];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[stage]);

    // head / tail elements outside the 16-byte aligned interior: plain loads
    const bool has_head = tid < head, has_tail = tid < tail;
    const float head_x = has_head ? load_logit<DT>(rowp, c0 + tid) : 0.0f;
    const float tail_x = has_tail ? load_logit<DT>(rowp, t0 + tid) : 0.0f;
    if (tid == 0 && kind == kLoad && tok >= c0 && tok < c0 + len && !(tok >= v0 && tok < t0))
      xval = load_logit<DT>(rowp, tok);

    float m = -INFINITY, sacc = 0.0f;
    int g = -1;
    if (!sampled) {
      if (has_head) { m = head_x; g = c0 + tid; }
#pragma unroll
      for (int j = 0; j < kVecPerThread; ++j) {
        const int v = tid + j * kConsumerThreads;
        if (v < nvec) {
          const int base = v0 + v * kVec;
          if constexpr (DT == SV_BF16) {
            const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
              if (g < 0 || lo > m) { m = lo; g = base + 2 * e; }
              if (hi > m) { m = hi; g = base + 2 * e + 1; }
            }
          } else {
            const float w[4] = {__uint_as_float(raw[j].x), __uint_as_float(raw[j].y),
                                __uint_as_float(raw[j].z), __uint_as_float(raw[j].w)};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (g < 0 || w[e] > m) { m = w[e]; g = base + e; }
          }
        }
      }
      if (has_tail && (g < 0 || tail_x > m)) { m = tail_x; g = t0 + tid; }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const int g2 = __shfl_xor_sync(0xFFFFFFFFu, g, o);
        merge_argmax(m, g, m2, g2);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kVecPerThread; ++j) {
        if (tid + j * kConsumerThreads < nvec) {
          if constexpr (DT == SV_BF16) {
            m = fmaxf(m, fmaxf(fmaxf(bf16_lo(raw[j].x), bf16_hi(raw[j].x)), fmaxf(bf16_lo(raw[j].y), bf16_hi(raw[j].y))));
            m = fmaxf(m, fmaxf(fmaxf(bf16_lo(raw[j].z), bf16_hi(raw[j].z)), fmaxf(bf16_lo(raw[j].w), bf16_hi(raw[j].w))));
          } else {
            m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(raw[j].x), __uint_as_float(raw[j].y)),
                               fmaxf(__uint_as_float(raw[j].z), __uint_as_float(raw[j].w))));
          }
        }
      }
      if (has_head) m = fmaxf(m, head_x);
      if (has_tail) m = fmaxf(m, tail_x);
      if (m != -INFINITY) {
        if (has_head) sacc += ex2_approx((head_x - m) * kscale);
#pragma unroll
        for (int j = 0; j < kVecPerThread; ++j) {
          if (tid + j * kConsumerThreads < nvec) {
            if constexpr (DT == SV_BF16) {
              const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                sacc += ex2_approx((bf16_lo(w[e]) - m) * kscale);
                sacc += ex2_approx((bf16_hi(w[e]) - m) * kscale);
              }
            } else {
              sacc += ex2_approx((__uint_as_float(raw[j].x) - m) * kscale);
              sacc += ex2_approx((__uint_as_float(raw[j].y) - m) * kscale);
              sacc += ex2_approx((__uint_as_float(raw[j].z) - m) * kscale);
              sacc += ex2_approx((__uint_as_float(raw[j].w) - m) * kscale);
            }
          }
        }
        if (has_tail) sacc += ex2_approx((tail_x - m) * kscale);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, sacc, o);
        merge_ms(m, sacc, m2, s2, kscale);
      }
    }
    if (lane == 0) {
      red[buf].m[warp] = m;
      red[buf].s[warp] = sacc;
      red[buf].g[warp] = g;
    }
    if (tid == 0) xval_s = xval;
    named_bar(1, kConsumerThreads);
    if (warp == 0) {
      float mm = lane < kConsumerWarps ? red[buf].m[lane] : -INFINITY;
      float ss = lane < kConsumerWarps ? red[buf].s[lane] : 0.0f;
      int gg = lane < kConsumerWarps ? red[buf].g[lane] : -1;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, mm, o);
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, ss, o);
        const int g2 = __shfl_xor_sync(0xFFFFFFFFu, gg, o);
        if (sampled) merge_ms(mm, ss, m2, s2, kscale);
        else merge_argmax(mm, gg, m2, g2);
      }
      if (lane == 0) {
        if (kind == kLoad) {
          float4 rec;
          rec.x = mm;
          rec.y = sampled ? ss : 0.0f;
          rec.z = __int_as_float(sampled ? -1 : gg);
          rec.w = xval_s;
          __stcg(reinterpret_cast<float4*>(p.rec + (static_cast<int64_t>(i) * R + r) * NC + c), rec);
        }
        __threadfence();
        const uint32_t old = atomicAdd(p.cnt_stats + i, 1u);
        red[buf].last = (old + 1u == expected_tasks(inf, NC)) ? 1 : 0;
        red[buf].stop = abort_flag;
        __threadfence();
      }
    }
    named_bar(1, kConsumerThreads);
    if (red[buf].last) combine_request(p, i, inf, tid, &cs);
    if (red[buf].stop) break;
    buf ^= 1;
  }
  pdl_trigger();
}

// ------------------------------------------------------------------------------------------
// sample kernel: grid (nchunks, B)
// ------------------------------------------------------------------------------------------
struct SampleSmem {
  ReqState st;
  float wsum[kSampleThreads / 32];
  float seg_excl[kSampleThreads];
  int pick_thread;
  int last_pos;
  int last;
  int chunk;
  double base;
  double Z;
  int use_bonus_row;
  uint32_t flags;
};

// weight of vocabulary entry v (index inside the chunk) for the draw
template <int DT>
__device__ __forceinline__ float draw_weight(const unsigned char* tb, const unsigned char* db, int v, bool residual,
                                             const ReqState& st) {
  float t, d = 0.0f;
  if constexpr (DT == SV_BF16) {
    t = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(tb)[v]) << 16);
    if (residual) d = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(db)[v]) << 16);
  } else {
    t = reinterpret_cast<const float*>(tb)[v];
    if (residual) d = reinterpret_cast<const float*>(db)[v];
  }
  const float pv = ex2_approx((t - st.mt) * st.kscale);
  if (!residual) return pv;
  return fmaxf(0.0f, pv * st.inv_st - ex2_approx((d - st.md) * st.kscale) * st.inv_sd);
}

// Copy `len` elements of a row chunk into shared memory (16-byte vectors + scalar tail).
template <int DT>
__device__ void stage_chunk(unsigned char* dst, const char* src, int len, int tid) {
  constexpr int kElt = DT == SV_BF16 ? 2 : 4;
  const int nvec = (reinterpret_cast<uintptr_t>(src) & 15u) ? 0 : ((len * kElt) >> 4);
  for (int v = tid; v < nvec; v += kSampleThreads)
    reinterpret_cast<uint4*>(dst)[v] = __ldg(reinterpret_cast<const uint4*>(src) + v);
  for (int e = nvec * (16 / kElt) + tid; e < len; e += kSampleThreads) {
    if constexpr (DT == SV_BF16)
      reinterpret_cast<uint16_t*>(dst)[e] = __ldg(reinterpret_cast<const uint16_t*>(src) + e);
    else
      reinterpret_cast<float*>(dst)[e] = __ldg(reinterpret_cast<const float*>(src) + e);
  }
}

// Inverse-CDF pick inside one staged chunk: first v with base + cumsum_{w<=v} > thr.
template <int DT>
__device__ int scan_pick(const unsigned char* tb, const unsigned char* db, int len, bool residual,
                         const ReqState& st, double base, double thr, int tid, SampleSmem* sm) {
  const int seg = (len + kSampleThreads - 1) / kSampleThreads;
  const int lo = min(len, tid * seg), hi = min(len, lo + seg);
  float ssum = 0.0f;
  int lastpos = -1;
  for (int v = lo; v < hi; ++v) {
    const float w = draw_weight<DT>(tb, db, v, residual, st);
    ssum += w;
    if (w > 0.0f) lastpos = v;
  }
  // block exclusive scan of segment sums (sequential over warps' totals; deterministic)
  const int lane = tid & 31, warp = tid >> 5;
  float incl = ssum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm->wsum[warp] = incl;
  if (tid == 0) {
    sm->pick_thread = kSampleThreads;
    sm->last_pos = -1;
  }
  __syncthreads();
  float wbase = 0.0f;
  for (int w = 0; w < warp; ++w) wbase += sm->wsum[w];
  const float excl = wbase + incl - ssum;
  const float rem = static_cast<float>(thr - base);
  if (hi > lo && ssum > 0.0f && excl + ssum > rem) atomicMin(&sm->pick_thread, tid);
  if (lastpos >= 0) atomicMax(&sm->last_pos, lastpos);
  __syncthreads();
  int y = -1;
  if (tid == sm->pick_thread) {
    float run = excl;
    for (int v = lo; v < hi; ++v) {
      const float w = draw_weight<DT>(tb, db, v, residual, st);
      run += w;
      if (run > rem && w > 0.0f) {
        y = v;
        break;
      }
    }
    if (y < 0) y = lastpos;  // rounding: stay on the last positive weight of this segment
    sm->last_pos = y;
  }
  __syncthreads();
  return sm->last_pos;  // pick (or the last positive entry of the chunk if no segment crossed)
}

template <int DT>
__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const VerifyParams p) {
  constexpr int kElt = DT == SV_BF16 ? 2 : 4;
  __shared__ __align__(16) unsigned char tbuf[kStageBytes];
  __shared__ __align__(16) unsigned char dbuf[kStageBytes];
  __shared__ SampleSmem sm;
  pdl_wait();
  const int tid = threadIdx.x;
  const int i = blockIdx.y, c = blockIdx.x;
  const int NC = p.nchunks;
  if (tid == 0) sm.st = p.req[i];
  __syncthreads();
  const ReqState& st = sm.st;
  if (st.mode == kModeNone) return;
  if (st.mode == kModeBonus && c != 0) return;

  bool residual = st.mode == kModeResidual;
  if (residual) {
    // chunk residual mass
    const int c0 = c * p.chunk_len, len = min(p.chunk_len, p.V - c0);
    const char* trow = row_ptr<DT>(p.target, st.row_t, p.t_row_stride) + static_cast<int64_t>(c0) * kElt;
    const char* drow = row_ptr<DT>(p.draft, st.row_d, p.d_row_stride) + static_cast<int64_t>(c0) * kElt;
    stage_chunk<DT>(tbuf, trow, len, tid);
    stage_chunk<DT>(dbuf, drow, len, tid);
    __syncthreads();
    float acc = 0.0f;
    for (int v = tid; v < len; v += kSampleThreads) acc += draw_weight<DT>(tbuf, dbuf, v, true, st);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if ((tid & 31) == 0) sm.wsum[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
      float tot = 0.0f;
      for (int w = 0; w < kSampleThreads / 32; ++w) tot += sm.wsum[w];
      __stcg(p.mass + static_cast<int64_t>(i) * NC + c, tot);
      __threadfence();
      const uint32_t old = atomicAdd(p.cnt_sample + i, 1u);
      sm.last = (old + 1u == static_cast<uint32_t>(NC)) ? 1 : 0;
      __threadfence();
    }
    __syncthreads();
    if (!sm.last) return;
  }

  // ---- one CTA per request from here on ----
  if (tid == 0) {
    sm.flags = 0;
    sm.use_bonus_row = residual ? 0 : 1;
    double Z = 0.0;
    if (residual) {
      for (int cc = 0; cc < NC; ++cc) Z += static_cast<double>(__ldcg(p.mass + static_cast<int64_t>(i) * NC + cc));
      if (!(Z > 0.0)) {
        sm.flags |= SV_FLAG_Z_ZERO;
        sm.use_bonus_row = 1;  // draw from p_a instead
      }
    }
    if (sm.use_bonus_row) {
      Z = 0.0;
      const ChunkRecord* rr = p.rec + static_cast<int64_t>(st.rec_row_t) * NC;
      for (int cc = 0; cc < NC; ++cc) {
        const ChunkRecord rc = ld_record(rr + cc);
        if (rc.m != -INFINITY)
          Z += static_cast<double>(rc.s) * static_cast<double>(exp2f((rc.m - st.mt) * st.kscale));
      }
    }
    const double thr = st.u * Z;
    double base = 0.0;
    int cstar = -1;
    int last_pos_chunk = -1;
    for (int cc = 0; cc < NC; ++cc) {
      double w;
      if (sm.use_bonus_row) {
        const ChunkRecord rc = ld_record(p.rec + static_cast<int64_t>(st.rec_row_t) * NC + cc);
        w = rc.m != -INFINITY ? static_cast<double>(rc.s) * static_cast<double>(exp2f((rc.m - st.mt) * st.kscale)) : 0.0;
      } else {
        w = static_cast<double>(__ldcg(p.mass + static_cast<int64_t>(i) * NC + cc));
      }
      if (w > 0.0) last_pos_chunk = cc;
      if (base + w > thr && w > 0.0) {
        cstar = cc;
        break;
      }
      base += w;
    }
    if (cstar < 0) {  // rounding pushed the threshold past the end: last chunk with mass
      cstar = last_pos_chunk < 0 ? 0 : last_pos_chunk;
      base = thr;     // pick the first positive weight of that chunk
    }
    sm.chunk = cstar;
    sm.base = base;
    sm.Z = Z;
  }
  __syncthreads();
  residual = !sm.use_bonus_row;
  const int cstar = sm.chunk;
  const int c0 = cstar * p.chunk_len, len = min(p.chunk_len, p.V - c0);
  stage_chunk<DT>(tbuf, row_ptr<DT>(p.target, st.row_t, p.t_row_stride) + static_cast<int64_t>(c0) * kElt, len, tid);
  if (residual)
    stage_chunk<DT>(dbuf, row_ptr<DT>(p.draft, st.row_d, p.d_row_stride) + static_cast<int64_t>(c0) * kElt, len, tid);
  __syncthreads();
  const double thr = st.u * sm.Z;
  // when the chunk search fell off the end, base == thr: any positive weight crosses
  const int yloc = scan_pick<DT>(tbuf, dbuf, len, residual, st, sm.base, thr, tid, &sm);
  if (tid == 0) {
    // yloc < 0 only if every weight of the chosen chunk flushed to zero (a chunk mass below the
    // float range); keep the output a valid token.
    const int y = c0 + (yloc >= 0 ? yloc : 0);
    p.out_tokens[static_cast<int64_t>(i) * (p.Kmax + 1) + st.a] = y;
    if (p.out_flags && sm.flags) p.out_flags[i] = static_cast<uint8_t>(st.flags | sm.flags);
    if (residual || st.mode == kModeResidual) p.cnt_sample[i] = 0;
  }
}

int g_stats_blocks_per_sm[2] = {0, 0};
int g_num_sms = 0;

template <int DT>
cudaError_t launch_verify_t(const VerifyParams& p, bool sampled, cudaStream_t stream) {
  const size_t dyn = static_cast<size_t>(kStages) * kStageBytes + ((static_cast<size_t>(p.B) * 2 + 15) & ~size_t(15));
  cudaError_t e;
  if (g_num_sms == 0) {
    int dev;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  }
  const int di = DT == SV_BF16 ? 0 : 1;
  {
    const size_t max_dyn = static_cast<size_t>(kStages) * kStageBytes + SV_MAX_BATCH * 2;
    if (g_stats_blocks_per_sm[di] == 0) {
      if ((e = cudaFuncSetAttribute(row_stats_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(max_dyn))) != cudaSuccess)
        return e;
      int nb = 0;
      if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, row_stats_kernel<DT>, kStatsThreads,
                                                             static_cast<size_t>(kStages) * kStageBytes + 1024)) != cudaSuccess)
        return e;
      g_stats_blocks_per_sm[di] = nb > 0 ? nb : 1;
    }
  }
  const int64_t slots = static_cast<int64_t>(p.B) * p.rows_per_req * p.nchunks;
  const int64_t cap = static_cast<int64_t>(g_num_sms) * g_stats_blocks_per_sm[di];
  const int grid = static_cast<int>(slots < cap ? slots : cap);
  prof_before(SV_KERNEL_ROW_STATS, stream);
  row_stats_kernel<DT><<<grid, kStatsThreads, dyn, stream>>>(p);
  prof_after(SV_KERNEL_ROW_STATS, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (!sampled) return cudaSuccess;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.nchunks), static_cast<unsigned>(p.B), 1);
  cfg.blockDim = dim3(kSampleThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // Programmatic dependent launch lets the sample grid's launch overlap the row_stats tail; it
  // is left out while instrumentation puts an event between the two kernels.
  cfg.numAttrs = prof_enabled() ? 0 : 1;
  prof_before(SV_KERNEL_SAMPLE, stream);
  e = cudaLaunchKernelEx(&cfg, sample_kernel<DT>, p);
  prof_after(SV_KERNEL_SAMPLE, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

void vocab_tiling(int V, sv_dtype dt, int* chunk_len, int* nchunks) {
  const int elt = dt == SV_BF16 ? 2 : 4;
  const int vec = 16 / elt;
  const int stage_elems = kStageBytes / elt;
  int nc = (V + stage_elems - 1) / stage_elems;
  if (nc < 1) nc = 1;
  int cl = (V + nc - 1) / nc;
  cl = (cl + vec - 1) / vec * vec;
  if (cl > stage_elems) cl = stage_elems;
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
  L.cnt_stats = off;
  off = align256(off + sizeof(uint32_t) * B);
  L.cnt_sample = off;
  off = align256(off + sizeof(uint32_t) * B);
  L.req = off;
  off = align256(off + sizeof(ReqState) * B);
  L.rowstat = off;
  off = align256(off + sizeof(RowStat) * B * R);
  L.mass = off;
  off = align256(off + sizeof(float) * B * static_cast<size_t>(nchunks));
  L.rec = off;
  off = align256(off + sizeof(ChunkRecord) * B * R * static_cast<size_t>(nchunks));
  L.total = off;
  return L;
}

int launch_verify(const VerifyParams& p, sv_dtype dt, bool sampled, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return static_cast<int>(dt == SV_BF16 ? launch_verify_t<SV_BF16>(p, sampled, s)
                                        : launch_verify_t<SV_F32>(p, sampled, s));
}

}  // namespace sv
