// Verification kernels of libsv.
//
// row_stats  One streaming pass over every logit row a round needs.  A persistent grid walks
//            (request, row, vocabulary chunk) tasks in request-major order, one contiguous range
//            per CTA; one producer lane issues 1-D bulk copies (cp.async.bulk) of <= 16 KB chunks
//            into a shared-memory ring (4 stages at 3 CTAs per SM for fp32 rows, 3 stages at 4
//            CTAs per SM for bf16) and four consumer warps, each waiting on a stage itself,
//            reduce each chunk.  A
//            piece of a row (its chunks inside one CTA's range) becomes one record {max m,
//            sum of 2^(x k - rint(m k)) with k = log2(e)/T, first argmax, logit at the drafted
//            token}.  The kernel only streams and writes records: no atomics, no fences, no
//            waiting on other CTAs.
// combine    Launched behind row_stats with programmatic dependent launch, grid (vocabulary
//            chunks, B) for short sampled requests, else (1, B).  Every CTA of request i merges the
//            request's records into row statistics and runs the accept chain: the greedy test
//            x_k == argmax, or the rejection test u_k q_k(x_k) < p_k(x_k); the first rejection
//            is the accepted length (AngelSpec explainer, "MTP: fix position 2 and 3", eq.
//            L_e2e: one rejection voids every later position; AngelSpec release article, "Why
//            one universal drafter underperforms": rejection-sampling verification in one pass).
//            CTA 0 writes the outputs; each CTA of a short sampled request then sums its chunk of
//            the residual max(0, p_a - q_a) after a rejection and of the target weights p_a, in 8
//            per-warp ranges.
// mass       For longer requests the same range sums come from a separate grid (chunks, B) that
//            reads the draw state the combine leaves.
// pick       One CTA per request: the token at the accepted length a, drawn from
//            norm(max(0, p_a - q_a)) after a rejection or from p_n when every drafted token was
//            accepted (the bonus row), by inverse CDF in vocabulary order: a warp finds the
//            crossing range among the 8 x chunks range sums, the whole CTA scans that range.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr float kLog2eF = 1.44269504088896340736f;

// request info, one uint16 per request, cached in shared memory by every row_stats CTA
constexpr uint16_t kInfoN = 0x3FF;
constexpr uint16_t kInfoNeedDraft = 1u << 10;
constexpr uint16_t kInfoSampled = 1u << 11;
constexpr uint16_t kInfoInvalid = 1u << 12;

// log2(e) / T in float; every kernel uses this one value for a request's temperature.
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

// ------------------------------------------------------------------------------------------
// per-request validation (every row_stats CTA computes the same info; CTA 0 reports errors)
// ------------------------------------------------------------------------------------------
__device__ uint16_t request_info(const VerifyParams& p, int i, uint32_t* bad_out) {
  // every load is issued before any is used (one round trip)
  const float T = p.temperature ? __ldg(p.temperature + i) : 0.0f;
  const int ta = p.t_off ? __ldg(p.t_off + i) : 0, tb = p.t_off ? __ldg(p.t_off + i + 1) : 0;
  const int da = p.d_off ? __ldg(p.d_off + i) : 0, dbb = p.d_off ? __ldg(p.d_off + i + 1) : 0;
  // a tree of N nodes streams N target rows and (sampled) the draft rows of nodes 0..N-2 (node
  // N - 1 is a leaf): the rows of a chain of N - 1 positions
  const int n = p.tree ? tb - ta - 1 : (p.keep_len ? __ldg(p.keep_len + i) : p.Kmax);
  uint32_t bad = 0;
  if (n < 0 || n > p.Kmax) bad |= SV_DEV_BAD_KEEP_LEN;
  if (!(T >= 0.0f) || isinf(T)) bad |= SV_DEV_BAD_TEMPERATURE;
  const bool sampled = T > 0.0f;
  const bool need_draft = (sampled || (p.tokens == nullptr && !p.tree)) && n > 0;  // n == 0: bonus row only
  if (sampled && n > 0 && p.tokens == nullptr && !p.tree) bad |= SV_DEV_BAD_TOKEN;
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
// row_stats kernel
// ------------------------------------------------------------------------------------------
// Rows are numbered request by request (row_start[i] = first row of request i, built in every
// CTA's prologue); inside a request its n_i + 1 target rows come first, then its n_i draft rows
// when it reads them.  The (row, chunk) tasks are split into one contiguous range per CTA, so a
// CTA keeps running per-thread statistics across consecutive chunks of a row and reduces across
// threads only where a row ends.  The first chunk of each (CTA, row) piece receives the merged
// record; the other chunks of the piece receive an empty record (max -inf) that still carries
// the drafted token's logit when the token lies in that chunk.
struct RowRef {
  int i;        // request
  int k;        // position inside the request
  int rec_row;  // record row: k for target rows, Kmax + 1 + k for draft rows
  bool is_target;
};

// Request holding row r: the largest i in [0, B) with row_start[i] <= r (a request without rows
// shares its start with the next request and is never the largest).
__device__ __forceinline__ int find_request(const int* row_start, int B, int r) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (row_start[mid] <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void locate_row(const int* row_start, const uint16_t* info, int Kmax, int row, int& i,
                                           RowRef& rr) {
  while (row >= row_start[i + 1]) ++i;  // rows are visited in increasing order
  const int q = row - row_start[i];
  const int n = info[i] & kInfoN;
  rr.i = i;
  rr.is_target = q <= n;
  rr.k = rr.is_target ? q : q - n - 1;
  rr.rec_row = rr.is_target ? rr.k : Kmax + 1 + rr.k;
}

// Address of vocabulary entry 0 of a row when the arrays hold the columns from v_begin on (a
// vocabulary shard; v_begin = 0 for whole rows): only entries >= v_begin are ever read through it.
template <int DT>
__device__ __forceinline__ const char* shard_row(const char* row, const VerifyParams& p) {
  constexpr int kElt = DT == SV_BF16 ? 2 : 4;
  return row - p.v_begin * kElt;
}

template <int DT>
__device__ __forceinline__ const char* row_base(const VerifyParams& p, const RowRef& rr) {
  return shard_row<DT>(rr.is_target ? row_ptr<DT>(p.target, target_row(p, rr.i, rr.k), p.t_row_stride)
                                    : row_ptr<DT>(p.draft, draft_row(p, rr.i, rr.k), p.d_row_stride), p);
}

// Closed-form plan: every request has U record rows (its K + 1 target rows, then its K draft
// rows when U == 2K + 1).
__device__ __forceinline__ void locate_row_uniform(int U, int Kmax, int row, RowRef& rr) {
  rr.i = row / U;
  const int q = row - rr.i * U;
  rr.is_target = q <= Kmax;
  rr.k = rr.is_target ? q : q - Kmax - 1;
  rr.rec_row = rr.is_target ? rr.k : Kmax + 1 + rr.k;
}

__device__ __forceinline__ int rows_of(uint16_t inf) {
  if (inf & kInfoInvalid) return 0;
  const int n = inf & kInfoN;
  return n + 1 + ((inf & kInfoNeedDraft) ? n : 0);
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

struct StatsRed {
  float m[kConsumerWarps];
  float s[kConsumerWarps];
  int g[kConsumerWarps];
  int stop;  // snapshot of the abort flag, taken before the barrier
};

template <int DT>
__global__ void __launch_bounds__(kStatsThreads, StreamShape<DT>::kCtasPerSm) row_stats_kernel(const VerifyParams p) {
  constexpr int kStages = StreamShape<DT>::kStages;
  constexpr int kElt = DT == SV_BF16 ? 2 : 4;
  constexpr int kVec = 16 / kElt;  // elements per 16-byte vector
  // -inf in every element of a padding vector
  constexpr uint32_t kPadWord = DT == SV_BF16 ? 0xFF80FF80u : 0xFF800000u;
  extern __shared__ __align__(128) unsigned char smem[];
  const int B = p.B, Kmax = p.Kmax, NC = p.nchunks, R = p.rows_per_req;
  const int c_lo = p.c_begin, c_hi = p.c_end, NCo = c_hi - c_lo;  // this call's chunks of every row
  unsigned char* stages = smem;
  int* row_start = reinterpret_cast<int*>(smem + kStages * kStageBytes);        // [B + 1]
  uint16_t* info = reinterpret_cast<uint16_t*>(row_start + ((B + 4) & ~3));     // [B]
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ StatsRed red[2];
  __shared__ int warp_tot[kStatsThreads / 32 + 1];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  // ---- prologue: barriers, and (ragged calls) per-request info and the row prefix ----
  const bool uniform = p.uniform_rows > 0;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    abort_flag = 0;
    fence_proxy_async_smem();
  }
  if (!uniform) {  // every CTA computes the same table; the combine reports invalid requests
    const int per = (B + kStatsThreads - 1) / kStatsThreads;
    const int lo = min(B, tid * per), hi = min(B, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) {
      uint32_t bad;
      info[i] = request_info(p, i, &bad);
      local += rows_of(info[i]);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    int run = base + incl - local;
    for (int i = lo; i < hi; ++i) {
      row_start[i] = run;
      run += rows_of(info[i]);
    }
    if (tid == kStatsThreads - 1) row_start[B] = base + incl;
  }
  __syncthreads();
  const int64_t rows_total = uniform ? static_cast<int64_t>(B) * p.uniform_rows : row_start[B];
  const int64_t T = rows_total * NCo;
  const int64_t t0 = T * blockIdx.x / gridDim.x, t1 = T * (blockIdx.x + 1) / gridDim.x;
  if (t0 >= t1) {
    pdl_trigger();
    return;
  }
  auto locate = [&](int row, int& i, RowRef& rr) {
    if (uniform) locate_row_uniform(p.uniform_rows, Kmax, row, rr);
    else locate_row(row_start, info, Kmax, row, i, rr);
  };

  if (tid >= kConsumerThreads) {
    // ---------------- producer warp: one lane issues the bulk copies ----------------
    if (tid == kConsumerThreads) {
      int row = static_cast<int>(t0 / NCo), c = c_lo + static_cast<int>(t0 - static_cast<int64_t>(row) * NCo);
      int i = uniform ? 0 : find_request(row_start, B, row);
      RowRef rr;
      locate(row, i, rr);
      const char* src = row_base<DT>(p, rr);
      uint32_t it = 0;
      // test hook: the chosen CTA issues nothing, so its consumers' first wait runs out
      const bool stall = p.stall_cta == static_cast<int>(blockIdx.x) + 1;
      const uint64_t pol_last = policy_evict_last(), pol_first = policy_evict_first();
      for (int64_t t = t0; t < t1 && !stall; ++t) {
        if (abort_flag) break;
        const int stage = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        ++it;
        if (!mbar_wait(&empty_bar[stage], ph ^ 1u, p.status, p.wait_limit_ns)) {
          abort_flag = 1;
          break;
        }
        const int c0 = c * p.chunk_len;
        const ChunkSplit sp = split_chunk<kElt>(src, c0, min(p.chunk_len, p.V - c0));
        if (sp.nvec == 0) {
          mbar_arrive(&full_bar[stage]);
        } else {
          mbar_arrive_expect_tx(&full_bar[stage], static_cast<uint32_t>(sp.nvec) * 16u);
          // The stream's lines are marked first to be evicted from L2: it reads each of them once,
          // and the chunk records and the draw's re-reads keep their lines (an A/B on GB300:
          // C4 65.0 -> 59.0, C5 78.3 -> 75.6, C3 213.1 -> 210.7 us per step).  A tree's root rows
          // are marked last instead: every walk starts there and re-reads them at each rejection.
          bulk_g2s_hint(stages + stage * kStageBytes, src + static_cast<int64_t>(c0 + sp.head) * kElt,
                        static_cast<uint32_t>(sp.nvec) * 16u, &full_bar[stage],
                        (p.tree && rr.k == 0) ? pol_last : pol_first);
        }
        if (++c == c_hi && t + 1 < t1) {
          c = c_lo;
          locate(++row, i, rr);
          src = row_base<DT>(p, rr);
        }
      }
      // drain: every issued copy must land before the CTA may exit
      const uint32_t issued = it;
      for (uint32_t s = 0; s < kStages && s < issued; ++s) {
        const uint32_t last = issued - 1 - ((issued - 1 - s) % kStages);  // last issue on stage s
        mbar_wait(&full_bar[s], (last / kStages) & 1u, p.status, p.wait_limit_ns);
      }
    }
    pdl_trigger();
    return;
  }

  // ---------------- consumer warps ----------------
  int row = static_cast<int>(t0 / NCo), c = c_lo + static_cast<int>(t0 - static_cast<int64_t>(row) * NCo);
  int i = uniform ? 0 : find_request(row_start, B, row);
  RowRef rr;
  locate(row, i, rr);
  int stage = 0;     // ring slot of the next chunk
  uint32_t ph = 0u;  // its phase parity
  int buf = 0;
  bool row_open = false;
  // per-row state
  const char* rowp = nullptr;
  bool sampled = false;
  float kscale = 0.0f, m = -INFINITY, sacc = 0.0f, xfirst = NAN;
  float cofs = 0.0f;  // exp_offset(m, kscale) of the running max (sampled rows)
  int g = -1, tok = -1, c_first = 0;
  for (int64_t t = t0; t < t1; ++t) {
    if (!row_open) {
      int n;
      if (uniform) {  // invalid temperatures give garbage statistics; the combine rejects the request
        const float T = p.temperature ? __ldg(p.temperature + rr.i) : 0.0f;
        sampled = T > 0.0f;
        kscale = sampled ? kscale_of(T) : 0.0f;
        n = Kmax;
      } else {
        const uint16_t inf = info[rr.i];
        sampled = inf & kInfoSampled;
        kscale = sampled ? kscale_of(__ldg(p.temperature + rr.i)) : 0.0f;
        n = inf & kInfoN;
      }
      tok = (tid == 0 && sampled && p.tokens != nullptr && rr.k < n)
                ? __ldg(p.tokens + static_cast<int64_t>(rr.i) * p.tok_stride + rr.k) : -1;
      rowp = row_base<DT>(p, rr);
      c_first = c;
      m = -INFINITY;
      sacc = 0.0f;
      g = -1;
      xfirst = NAN;
      row_open = true;
    }
    const int c0 = c * p.chunk_len;
    const int len = min(p.chunk_len, p.V - c0);
    const ChunkSplit sp = split_chunk<kElt>(rowp, c0, len);
    const int head = sp.head, nvec = sp.nvec, tail = sp.tail;
    const int v0 = c0 + head;         // vocabulary index of the first staged element
    const int te = v0 + nvec * kVec;  // first tail element

    // Every consumer warp waits for the stage itself (backed-off polling; the barrier's phase
    // completion orders its shared-memory reads after the bulk copy), so no warp waits on another
    // (an A/B on GB300: C3's stream 191.7 -> 185.9 us, C5's 60.1 -> 59.3 us against one warp
    // polling while the others slept in a named barrier).  After a timeout the remaining tasks run
    // on whatever the stage holds; the loop leaves at the next row end, where every consumer
    // thread reads the same abort snapshot.
    if (!abort_flag && !mbar_wait(&full_bar[stage], ph, p.status, p.wait_limit_ns)) abort_flag = 1;
    const unsigned char* sb = stages + stage * kStageBytes;
    uint64_t* const empty_here = &empty_bar[stage];
    if (++stage == kStages) {
      stage = 0;
      ph ^= 1u;
    }
    uint4 raw[kVecPerThread];
    if (DT == SV_BF16 && nvec == kVecPerThread * kConsumerThreads) {  // a full bf16 chunk: no predicates
#pragma unroll
      for (int j = 0; j < kVecPerThread; ++j) raw[j] = lds128(sb + (tid + j * kConsumerThreads) * 16);
    } else {
#pragma unroll
      for (int j = 0; j < kVecPerThread; ++j) {
        const int v = tid + j * kConsumerThreads;
        raw[j] = v < nvec ? lds128(sb + v * 16) : make_uint4(kPadWord, kPadWord, kPadWord, kPadWord);
      }
    }
    float xval = NAN;
    if (tid == 0 && tok >= v0 && tok < te) {
      if constexpr (DT == SV_BF16)
        xval = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(sb)[tok - v0]) << 16);
      else
        xval = reinterpret_cast<const float*>(sb)[tok - v0];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_here);

    // head / tail elements outside the 16-byte aligned interior: plain loads (none for a chunk
    // that is all interior, the common case: the same in every thread)
    const bool edges = head != 0 || tail != 0;
    const bool has_head = edges && tid < head, has_tail = edges && tid < tail;
    float head_x = -INFINITY, tail_x = -INFINITY;
    if (edges) {
      if (has_head) head_x = load_logit<DT>(rowp, c0 + tid);
      if (has_tail) tail_x = load_logit<DT>(rowp, te + tid);
      if (tid == 0 && tok >= c0 && tok < c0 + len && !(tok >= v0 && tok < te)) xval = load_logit<DT>(rowp, tok);
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
      if (edges) mc = fmaxf(mc, fmaxf(head_x, tail_x));
      if (mc > m) {  // new running max: move the running sum to the new offset (exact)
        const float cnew = exp_offset(mc, kscale);
        sacc = (m == -INFINITY) ? 0.0f : sacc * pow2_nonpos(cofs - cnew);
        m = mc;
        cofs = cnew;
      }
      if (m != -INFINITY) {
        // terms 2^(x k - c): one fused multiply-add per logit, done on pairs of logits in
        // packed f32x2 registers; even and odd positions keep separate sums.  Padding vectors
        // hold -inf, whose term is 2^-inf = 0: bf16 needs no predicate per vector (fp32 keeps
        // one, which measured faster there).
        const f32x2 k2 = f2_pack(kscale, kscale), nc2 = f2_pack(-cofs, -cofs);
        f32x2 acc2[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};  // two independent chains
#pragma unroll
        for (int j = 0; j < kVecPerThread; ++j) {
          if constexpr (DT == SV_BF16) {
            const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              acc2[e & 1] = f2_add(acc2[e & 1], f2_exp2_offset(f2_pack(bf16_lo(w[e]), bf16_hi(w[e])), k2, nc2));
          } else if (tid + j * kConsumerThreads < nvec) {
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
        if (edges) {
          if (has_head) acc += ex2_approx(__fmaf_rn(head_x, kscale, -cofs));
          if (has_tail) acc += ex2_approx(__fmaf_rn(tail_x, kscale, -cofs));
        }
        sacc += acc;
      }
    }

    ChunkRecord* rec_row = p.rec + (static_cast<int64_t>(rr.i) * R + rr.rec_row) * NC;
    if (tid == 0) {
      if (c == c_first) {
        xfirst = xval;
      } else {
        // empty record: this chunk's statistics live in the piece's first record
        __stcg(reinterpret_cast<float4*>(rec_row + c), make_float4(-INFINITY, 0.0f, __int_as_float(-1), xval));
      }
    }

    const bool row_end = (c == c_hi - 1) || (t + 1 == t1);
    if (row_end) {
      // reduce the piece across threads and write its record
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        if (sampled) {
          const float s2 = __shfl_xor_sync(0xFFFFFFFFu, sacc, o);
          merge_ms(m, sacc, m2, s2, kscale);
        } else {
          const int g2 = __shfl_xor_sync(0xFFFFFFFFu, g, o);
          merge_argmax(m, g, m2, g2);
        }
      }
      if (lane == 0) {
        red[buf].m[warp] = m;
        red[buf].s[warp] = sacc;
        red[buf].g[warp] = g;
      }
      if (tid == 0) red[buf].stop = abort_flag;
      // red[] is double-buffered: a warp writes red[buf] again two row ends later, after the
      // next barrier, by which time warp 0 has read it.
      named_bar(1, kConsumerThreads);
      if (warp == 0) {
        float mm = lane < kConsumerWarps ? red[buf].m[lane] : -INFINITY;
        float ss = lane < kConsumerWarps ? red[buf].s[lane] : 0.0f;
        int gg = lane < kConsumerWarps ? red[buf].g[lane] : -1;
#pragma unroll
        for (int o = kConsumerWarps / 2; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xFFFFFFFFu, mm, o);
          const float s2 = __shfl_xor_sync(0xFFFFFFFFu, ss, o);
          const int g2 = __shfl_xor_sync(0xFFFFFFFFu, gg, o);
          if (sampled) merge_ms(mm, ss, m2, s2, kscale);
          else merge_argmax(mm, gg, m2, g2);
        }
        if (lane == 0)
          __stcg(reinterpret_cast<float4*>(rec_row + c_first),
                 make_float4(mm, sampled ? ss : 0.0f, __int_as_float(sampled ? -1 : gg), xfirst));
      }
      const int stop = red[buf].stop;
      buf ^= 1;
      row_open = false;
      if (stop) break;
    }
    if (++c == c_hi && t + 1 < t1) {
      c = c_lo;
      locate(++row, i, rr);
    }
  }
  pdl_trigger();
}

// ------------------------------------------------------------------------------------------
// combine (grid (chunks or 1, B)), mass (grid (chunks, B)) and pick (grid B) kernels, chained
// behind row_stats with programmatic dependent launch
// ------------------------------------------------------------------------------------------
// Per-row statistics in shared memory (one entry per record row of the request).
struct RowStatS {
  float s;     // sum of 2^(x k - rint(m k)) over the row (sampled rows)
  float m;     // row max
  int32_t g;   // first argmax (greedy rows)
  float xval;  // logit at the row's drafted token (sampled rows)
};

constexpr size_t kFinMaxStagedBytes = 48 * 1024;  // chunk records staged in shared memory up to this
constexpr int kFinMaxDynSmem = 96 * 1024;
constexpr int kCombineThreads = 256, kCombineWarps = kCombineThreads / 32;
constexpr int kMassThreads = 256, kMassWarps = kMassThreads / 32;
static_assert(kCombineWarps == kDrawRanges && kMassWarps == kDrawRanges, "one draw range per warp");
// Requests with at most this many chunk records (rows x chunks) get their draw weights summed by
// the combine kernel's CTAs, which each merge the request's records again; longer requests use
// the separate mass kernel, which reads the draw state the combine leaves.
constexpr int kFuseDrawMaxRecords = 256;
constexpr int kPickThreads = 256, kPickWarps = kPickThreads / 32;
constexpr int kPickStaged = 2048;  // range masses staged in shared memory up to this many

struct CombineSmem {
  int a_min;
  uint32_t acc_flags;
  uint32_t bad;
};

struct PickSmem {
  ReqState st;
  float wsum[kPickWarps];
  int chunk;        // crossing draw range (chunk * kDrawRanges + range)
  int bonus;        // draw from the target row (bonus, or residual mass 0)
  uint32_t flags;
  float base;       // mass before the crossing range
  float thr;        // u' * Z
  int pick_thread;  // first thread whose entries hold the crossing
  int last_pos;     // broadcast of the pick
  float mass[2 * kPickStaged];
};

// weight of vocabulary entry v of a row pair for the draw (target-only when !residual)
template <int DT>
__device__ __forceinline__ float draw_weight(const char* trow, const char* drow, int64_t v, bool residual,
                                             const ReqState& st) {
  const float pv = ex2_approx(__fmaf_rn(load_logit<DT>(trow, v), st.kscale, -st.ct));
  if (!residual) return pv;
  return fmaxf(0.0f, pv * st.inv_st - ex2_approx(__fmaf_rn(load_logit<DT>(drow, v), st.kscale, -st.cd)) * st.inv_sd);
}

// Contiguous ranges of a chunk, one per warp: warp w of nw covers [lo, hi).
__device__ __forceinline__ void warp_range(int len, int nw, int w, int* lo, int* hi) {
  const int seg = (len + nw - 1) / nw;
  *lo = min(len, w * seg);
  *hi = min(len, *lo + seg);
}

// Sums over [c0 + lo, c0 + hi) by one warp: *sum_r of the residual max(0, p - q) (residual only)
// and *sum_p of the target weights.  Vectors are loaded in batches of kBatch per lane, every
// load of a batch issued before any is used.
constexpr int kBatch = 4;
template <int DT>
__device__ void warp_range_sum(const char* trow, const char* drow, int c0, int lo, int hi, bool residual,
                               const ReqState& st, int lane, float* sum_r, float* sum_p) {
  constexpr int kElt = DT == SV_BF16 ? 2 : 4;
  constexpr int kVec = 16 / kElt;
  float acc_r = 0.0f, acc_p = 0.0f;
  auto add = [&](float tx, float dx) {
    const float pv = ex2_approx(__fmaf_rn(tx, st.kscale, -st.ct));
    acc_p += pv;
    if (residual) acc_r += fmaxf(0.0f, pv * st.inv_st - ex2_approx(__fmaf_rn(dx, st.kscale, -st.cd)) * st.inv_sd);
  };
  const int len = hi - lo;
  const ChunkSplit a = split_chunk<kElt>(trow, c0 + lo, len);
  const ChunkSplit b = residual ? split_chunk<kElt>(drow, c0 + lo, len) : a;
  if (a.nvec > 0 && a.head == b.head) {
    const int v0 = c0 + lo + a.head;
    const uint4* tv = reinterpret_cast<const uint4*>(trow + static_cast<int64_t>(v0) * kElt);
    const uint4* dv = reinterpret_cast<const uint4*>(drow + static_cast<int64_t>(v0) * kElt);
    const bool hh = lane < a.head, ht = lane < a.tail;
    if (hh) add(load_logit<DT>(trow, c0 + lo + lane), residual ? load_logit<DT>(drow, c0 + lo + lane) : 0.0f);
    if (ht)
      add(load_logit<DT>(trow, v0 + a.nvec * kVec + lane),
          residual ? load_logit<DT>(drow, v0 + a.nvec * kVec + lane) : 0.0f);
    for (int base = 0; base < a.nvec; base += 32 * kBatch) {
      uint4 tw[kBatch], dw[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int v = base + lane + 32 * u;
        tw[u] = v < a.nvec ? __ldg(tv + v) : make_uint4(0, 0, 0, 0);
        dw[u] = (residual && v < a.nvec) ? __ldg(dv + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (base + lane + 32 * u >= a.nvec) break;
        if constexpr (DT == SV_BF16) {
          const uint32_t t4[4] = {tw[u].x, tw[u].y, tw[u].z, tw[u].w}, d4[4] = {dw[u].x, dw[u].y, dw[u].z, dw[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            add(bf16_lo(t4[e]), bf16_lo(d4[e]));
            add(bf16_hi(t4[e]), bf16_hi(d4[e]));
          }
        } else {
          add(__uint_as_float(tw[u].x), __uint_as_float(dw[u].x));
          add(__uint_as_float(tw[u].y), __uint_as_float(dw[u].y));
          add(__uint_as_float(tw[u].z), __uint_as_float(dw[u].z));
          add(__uint_as_float(tw[u].w), __uint_as_float(dw[u].w));
        }
      }
    }
  } else {
#pragma unroll 4
    for (int e = lane; e < len; e += 32)
      add(load_logit<DT>(trow, c0 + lo + e), residual ? load_logit<DT>(drow, c0 + lo + e) : 0.0f);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    acc_r += __shfl_xor_sync(0xFFFFFFFFu, acc_r, o);
    acc_p += __shfl_xor_sync(0xFFFFFFFFu, acc_p, o);
  }
  *sum_r = acc_r;
  *sum_p = acc_p;
}

// Inverse-CDF pick inside one draw range by a whole kPickThreads CTA.  Thread t owns the
// contiguous entries [t*per, (t+1)*per) of the range.  Returns the range-relative index of the
// first entry with cumsum > rem, or, if rounding keeps every partial sum at or below rem, the last
// entry with positive weight (-1 if none).
template <int DT>
__device__ int block_pick(const char* trow, const char* drow, int c0, int len, bool residual, const ReqState& st,
                          float rem, PickSmem* sm, int tid) {
  // a draw range holds at most ceil(chunk / kDrawRanges) entries: kMaxPer per thread
  constexpr int kMaxPer = (kStageBytes / 2 / kDrawRanges + kPickThreads - 1) / kPickThreads;
  const int lane = tid & 31, warp = tid >> 5;
  const int per = (len + kPickThreads - 1) / kPickThreads;
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
  for (int j = 0; j < kMaxPer; ++j) {
    const float pv = ex2_approx(__fmaf_rn(tx[j], st.kscale, -st.ct));
    w[j] = j >= cnt ? 0.0f
           : residual ? fmaxf(0.0f, pv * st.inv_st - ex2_approx(__fmaf_rn(dx[j], st.kscale, -st.cd)) * st.inv_sd)
                      : pv;
  }
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
  if (lane == 31) sm->wsum[warp] = incl;
  if (tid == 0) {
    sm->pick_thread = kPickThreads;
    sm->last_pos = -1;
  }
  __syncthreads();
  float excl = incl - sum;
  for (int v = 0; v < warp; ++v) excl += sm->wsum[v];
  if (cnt > 0 && sum > 0.0f && excl + sum > rem) atomicMin(&sm->pick_thread, tid);
  if (lastpos >= 0) atomicMax(&sm->last_pos, lastpos);
  __syncthreads();
  if (tid == sm->pick_thread) {
    float run = excl;
    int y = -1;
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j) {
      run += w[j];
      if (y < 0 && w[j] > 0.0f && run > rem) y = a + j;
    }
    sm->last_pos = y >= 0 ? y : lastpos;
  }
  __syncthreads();
  return sm->last_pos;
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

// Shared-memory plan of the combine kernel: row statistics, then (when they fit) the request's
// staged chunk records, then its drafted tokens.
struct FinLayout {
  size_t rec_off, tok_off, bytes;
  bool staged;
};
__host__ __device__ inline FinLayout fin_layout(int R, int NC, int Kmax) {
  FinLayout L;
  const size_t rows = static_cast<size_t>(R) * sizeof(RowStatS);
  const size_t recs = static_cast<size_t>(R) * NC * sizeof(ChunkRecord);
  L.staged = recs <= kFinMaxStagedBytes;
  L.rec_off = rows;
  L.tok_off = rows + (L.staged ? recs : 0);
  L.bytes = L.tok_off + ((static_cast<size_t>(Kmax) * 4 + 15) & ~size_t(15));
  return L;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---- combine: grid (chunks, B) when the draw weights are fused in, (1, B) otherwise -------
// Every CTA of request i merges the request's records and runs its accept chain (the CTAs agree
// without communicating: same inputs, same order of operations); CTA 0 writes the outputs and
// the draw state.  With the draw weights fused in, each CTA of a sampled request then sums its
// vocabulary chunk of the residual max(0, p_a - q_a) after a rejection, and of the target
// weights p_a (the bonus draw, or the fallback when the residual mass is zero).
template <int DT>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const VerifyParams p) {
  extern __shared__ __align__(16) unsigned char fin_dyn[];
  __shared__ CombineSmem sm;
  __shared__ ReqState sst;
  __shared__ float uacc[SV_MAX_DRAFT + 1], uprime[SV_MAX_DRAFT + 1];
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blockIdx.y, c = blockIdx.x;
  const int NC = p.nchunks, R = p.rows_per_req, Kmax = p.Kmax;
  const FinLayout FL = fin_layout(R, NC, Kmax);
  RowStatS* rs = reinterpret_cast<RowStatS*>(fin_dyn);                        // [R]
  ChunkRecord* rec_s = reinterpret_cast<ChunkRecord*>(fin_dyn + FL.rec_off);  // [R * NC] if staged
  int32_t* tok_s = reinterpret_cast<int32_t*>(fin_dyn + FL.tok_off);          // [Kmax]
  const ChunkRecord* rec_g = p.rec + static_cast<int64_t>(i) * R * NC;
  const int32_t* toks = p.tokens ? p.tokens + static_cast<int64_t>(i) * p.tok_stride : nullptr;

  // round 1: everything the combine reads, requested at once (records of all 2*Kmax+1 record
  // rows and all Kmax tokens; entries past n are ignored)
  if (FL.staged)
    for (int j = tid; j < R * NC; j += kCombineThreads) cp_async16(rec_s + j, rec_g + j);
  if (toks)
    for (int j = tid; j < Kmax; j += kCombineThreads) cp_async4(tok_s + j, toks + j);
  uint32_t bad_in;
  const uint16_t info = request_info(p, i, &bad_in);
  const float T = p.temperature ? __ldg(p.temperature + i) : 0.0f;
  const int rid = p.request_ids ? __ldg(p.request_ids + i) : i;
  // the uniforms of every accept test and of the draw at every position depend only on the keys:
  // computed while the records are in flight
  for (int k = tid; k <= Kmax; k += kCombineThreads) {
    uacc[k] = philox_uniform_f(p.seed, static_cast<uint32_t>(k), static_cast<uint32_t>(rid), 0u, p.round);
    uprime[k] = philox_uniform_f(p.seed, static_cast<uint32_t>(k), static_cast<uint32_t>(rid), 1u, p.round);
  }
  cp_async_wait_all();
  __syncthreads();
  if (c > 0 && !(info & kInfoSampled)) return;  // nothing to draw: CTA 0 does all the work
  if (info & kInfoInvalid) {
    if (c == 0) {
      if (tid == 0) {
        atomicOr(p.status, bad_in);
        p.req[i].mode = kModeNone;
      }
      write_invalid(p, i, tid, kCombineThreads);
    }
    return;
  }
  const int n = info & kInfoN;
  const bool sampled = info & kInfoSampled;
  const bool need_draft = info & kInfoNeedDraft;
  const float kscale = sampled ? kscale_of(T) : 0.0f;
  const int nrows = n + 1 + (need_draft ? n : 0);
  const ChunkRecord* recs = FL.staged ? rec_s : rec_g;
  auto tok = [&](int k) { return toks ? tok_s[k] : rs[Kmax + 1 + k].g; };

  // 1. row statistics: one warp per row, one pass over the row's chunk records
  for (int q = warp; q < nrows; q += kCombineWarps) {
    const bool is_target = q <= n;
    const int k = is_target ? q : q - n - 1;
    const int r = is_target ? k : Kmax + 1 + k;
    const ChunkRecord* rr = recs + static_cast<int64_t>(r) * NC;
    const int x = (sampled && k < n) ? tok_s[k] : -1;  // drafted token of this row
    const int cx = (x >= 0 && x < p.V) ? x / p.chunk_len : -1;
    float m = -INFINITY, xval = NAN, S = 0.0f;
    int g = -1;
    if (sampled) {
      // row max, then the piece sums rescaled to it, added with a compensated (TwoSum) tree
      for (int cc = lane; cc < NC; cc += 32) {
        const ChunkRecord rc = FL.staged ? rr[cc] : ld_record(rr + cc);
        m = fmaxf(m, rc.m);
        if (cc == cx) xval = rc.xval;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      float hi = 0.0f, lo = 0.0f;
      if (m != -INFINITY) {
        const float C = exp_offset(m, kscale);
        for (int cc = lane; cc < NC; cc += 32) {
          const ChunkRecord rc = FL.staged ? rr[cc] : ld_record(rr + cc);
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
      for (int cc = lane; cc < NC; cc += 32) {
        const ChunkRecord rc = FL.staged ? rr[cc] : ld_record(rr + cc);
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
    sm.a_min = n;
    sm.acc_flags = 0;
    sm.bad = 0;
  }
  __syncthreads();

  // 2. accept tests (each position independently; the first rejection is a min-reduction)
  for (int k = tid; k < n; k += kCombineThreads) {
    const int x = tok(k);
    bool acc;
    float pv, qv;
    if (x < 0 || x >= p.V) {
      atomicOr(&sm.bad, SV_DEV_BAD_TOKEN);
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
      const float u = uacc[k];
      acc = u * qv < pv;
      if (qv == 0.0f) atomicOr(&sm.acc_flags, SV_FLAG_Q_ZERO);
    }
    if (c == 0) {
      if (p.out_p) p.out_p[static_cast<int64_t>(i) * Kmax + k] = pv;
      if (p.out_q) p.out_q[static_cast<int64_t>(i) * Kmax + k] = qv;
    }
    if (!acc) atomicMin(&sm.a_min, k);
  }
  if (c == 0)
    for (int k = n + tid; k < Kmax; k += kCombineThreads) {
      if (p.out_p) p.out_p[static_cast<int64_t>(i) * Kmax + k] = NAN;
      if (p.out_q) p.out_q[static_cast<int64_t>(i) * Kmax + k] = NAN;
    }
  __syncthreads();
  if (sm.bad) {
    if (c == 0) {
      if (tid == 0) {
        atomicOr(p.status, sm.bad);
        p.req[i].mode = kModeNone;
      }
      write_invalid(p, i, tid, kCombineThreads);
    }
    return;
  }
  const int a = sm.a_min;

  // 3. emit (CTA 0): the accepted prefix (and, greedy, the target argmax at a); a sampled
  //    request's token at a is written by the pick kernel
  if (c == 0)
    for (int j = tid; j <= Kmax; j += kCombineThreads) {
      if (j == a && sampled) continue;
      int v = -1;
      if (j < a) v = tok(j);
      else if (j == a) v = rs[a].g;
      p.out_tokens[static_cast<int64_t>(i) * (Kmax + 1) + j] = v;
    }
  if (tid == 0) {
    if (c == 0) {
      p.out_accept_len[i] = a;
      if (p.out_flags) p.out_flags[i] = static_cast<uint8_t>(sm.acc_flags);
    }
    ReqState st = {};
    st.mode = kModeNone;
    if (sampled) {
      st.mode = a < n ? kModeResidual : kModeBonus;
      st.a = a;
      st.flags = static_cast<int32_t>(sm.acc_flags);
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
      st.u = uprime[a];
    }
    if (c == 0) p.req[i] = st;
    sst = st;
  }
  __syncthreads();
  if (!p.fuse_draw || sst.mode == kModeNone) return;

  // 4. this CTA's vocabulary chunk of the draw weights (row a of the request)
  const bool residual = sst.mode == kModeResidual;
  const char* trow = row_ptr<DT>(p.target, sst.row_t, p.t_row_stride);
  const char* drow = residual ? row_ptr<DT>(p.draft, sst.row_d, p.d_row_stride) : trow;
  const int c0 = c * p.chunk_len, len = min(p.chunk_len, p.V - c0);
  int lo, hi;
  warp_range(len, kCombineWarps, warp, &lo, &hi);
  float wr, wp;
  warp_range_sum<DT>(trow, drow, c0, lo, hi, residual, sst, lane, &wr, &wp);
  if (lane == 0) {
    const int64_t e = (static_cast<int64_t>(i) * NC + c) * kDrawRanges + warp;
    p.mass[e] = wr;
    p.mass_p[e] = wp;
  }
}

// ---- mass: one light CTA per (request, chunk) --------------------------------------------
// Chunk sums of the residual max(0, p_a - q_a) after a rejection, and of the target weights
// of row a (the bonus draw, or the fallback when the residual mass is zero).
template <int DT>
__global__ void __launch_bounds__(kMassThreads) mass_kernel(const VerifyParams p) {
  __shared__ ReqState st;
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blockIdx.y, c = p.c_begin + blockIdx.x, NC = p.nchunks;  // this call's chunks
  if (tid == 0) st = p.req[i];
  __syncthreads();
  if (st.mode == kModeNone) return;
  const bool residual = st.mode == kModeResidual;
  const char* trow = shard_row<DT>(row_ptr<DT>(p.target, st.row_t, p.t_row_stride), p);
  const char* drow = residual ? shard_row<DT>(row_ptr<DT>(p.draft, st.row_d, p.d_row_stride), p) : trow;
  const int c0 = c * p.chunk_len, len = min(p.chunk_len, p.V - c0);
  int lo, hi;
  warp_range(len, kMassWarps, warp, &lo, &hi);
  float wr, wp;
  warp_range_sum<DT>(trow, drow, c0, lo, hi, residual, st, lane, &wr, &wp);
  if (lane == 0) {
    const int64_t e = (static_cast<int64_t>(i) * NC + c) * kDrawRanges + warp;
    p.mass[e] = wr;
    p.mass_p[e] = wp;
  }
}

// ---- pick: one CTA per request -------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kPickThreads) pick_kernel(const VerifyParams p) {
  __shared__ PickSmem sm;
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blockIdx.x, NC = p.nchunks, Kmax = p.Kmax;
  const int NE = NC * kDrawRanges;  // draw ranges of the request, in vocabulary order
  const float* mass_r = p.mass + static_cast<int64_t>(i) * NE;
  const float* mass_p = p.mass_p + static_cast<int64_t>(i) * NE;
  const bool staged = NE <= kPickStaged;
  // one round trip: the draw state and every range mass of the request (unused for requests
  // without a draw)
  if (tid == 0) sm.st = p.req[i];
  if (staged) {
    for (int j = tid; j < NE; j += kPickThreads) {
      sm.mass[j] = mass_r[j];
      sm.mass[kPickStaged + j] = mass_p[j];
    }
  }
  __syncthreads();
  const ReqState& st = sm.st;
  if (st.mode == kModeNone) return;
  const bool residual_mode = st.mode == kModeResidual;
  const char* trow = shard_row<DT>(row_ptr<DT>(p.target, st.row_t, p.t_row_stride), p);
  const char* drow = residual_mode ? shard_row<DT>(row_ptr<DT>(p.draft, st.row_d, p.d_row_stride), p) : trow;

  // the crossing range (one warp)
  if (warp == 0) {
    auto r_at = [&](int e) { return staged ? sm.mass[e] : mass_r[e]; };
    auto p_at = [&](int e) { return staged ? sm.mass[kPickStaged + e] : mass_p[e]; };
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
      sm.chunk = estar;
      sm.base = before;
      sm.thr = thr;
      sm.bonus = bonus;
      sm.flags = flags;
    }
  }
  __syncthreads();

  // the entry inside the crossing range (whole CTA), by the call that holds its chunk (a vocabulary
  // shard that does not leaves the token to the one that does)
  const int estar = sm.chunk, cstar = estar / kDrawRanges;
  if (cstar < p.c_begin || cstar >= p.c_end) return;
  const bool residual = !sm.bonus;
  const int c0 = cstar * p.chunk_len;
  int lo, hi;
  warp_range(min(p.chunk_len, p.V - c0), kDrawRanges, estar - cstar * kDrawRanges, &lo, &hi);
  int y = block_pick<DT>(trow, residual ? drow : trow, c0 + lo, hi - lo, residual, st, sm.thr - sm.base, &sm, tid);
  if (tid == 0) {
    if (y < 0) y = 0;  // only if every weight of the range flushed to zero; keep a valid token
    p.out_tokens[static_cast<int64_t>(i) * (Kmax + 1) + st.a] = c0 + lo + y;
    if (p.out_flags && sm.flags) p.out_flags[i] = static_cast<uint8_t>(st.flags | sm.flags);
  }
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
    const size_t max_dyn =
        static_cast<size_t>(StreamShape<DT>::kStages) * kStageBytes + (SV_MAX_BATCH + 4) * 4 + SV_MAX_BATCH * 2;
    if ((e = cudaFuncSetAttribute(row_stats_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(max_dyn))) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(combine_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kFinMaxDynSmem)) != cudaSuccess)
      return e;
    ds.ready[di] = true;
  }
  *num_sms = ds.num_sms;
  return cudaSuccess;
}

// Launch `kernel` behind the previous kernel on the stream with programmatic dependent launch
// (its launch overlaps the previous grid's tail; it waits in griddepcontrol.wait).  Left out
// while instrumentation puts events between kernels.
template <typename K>
cudaError_t launch_pdl(K kernel, dim3 grid, int threads, size_t smem, cudaStream_t stream, int prof_id,
                       const VerifyParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = prof_enabled() ? 0 : 1;
  prof_before(prof_id, stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
  prof_after(prof_id, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_row_stats_t(const VerifyParams& p, cudaStream_t stream) {
  const size_t table =
      p.uniform_rows > 0 ? 0 : static_cast<size_t>((p.B + 4) & ~3) * 4 + ((static_cast<size_t>(p.B) * 2 + 15) & ~size_t(15));
  const size_t dyn = static_cast<size_t>(StreamShape<DT>::kStages) * kStageBytes + table;
  cudaError_t e;
  int num_sms = 0;
  if ((e = device_setup<DT>(&num_sms)) != cudaSuccess) return e;
  int nb = 0;  // resident CTAs per SM at this table size (the grid is persistent)
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, row_stats_kernel<DT>, kStatsThreads, dyn)) != cudaSuccess)
    return e;
  // one contiguous task range per CTA; with a known task count (fixed-K calls) every CTA gets the
  // same number of (row, chunk) tasks, so the grid's CTAs finish together
  const int nco = p.c_end - p.c_begin;  // chunks of every row this call streams
  const int64_t slots = static_cast<int64_t>(p.B) * p.rows_per_req * nco;
  const int64_t tasks = p.uniform_rows > 0 ? static_cast<int64_t>(p.B) * p.uniform_rows * nco : slots;
  const int64_t cap = static_cast<int64_t>(num_sms) * (nb > 0 ? nb : 1);
  const int64_t per_cta = (tasks + cap - 1) / cap;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cap, (tasks + per_cta - 1) / per_cta)));
  prof_before(SV_KERNEL_ROW_STATS, stream);
  row_stats_kernel<DT><<<grid, kStatsThreads, dyn, stream>>>(p);
  prof_after(SV_KERNEL_ROW_STATS, stream);
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_verify_t(const VerifyParams& p, bool sampled, cudaStream_t stream) {
  cudaError_t e;
  if ((e = launch_row_stats_t<DT>(p, stream)) != cudaSuccess) return e;

  const size_t csmem = fin_layout(p.rows_per_req, p.nchunks, p.Kmax).bytes;
  if ((e = launch_pdl(combine_kernel<DT>, dim3(p.fuse_draw ? p.nchunks : 1, p.B), kCombineThreads, csmem, stream,
                      SV_KERNEL_COMBINE, p)) != cudaSuccess)
    return e;
  if (!sampled) return cudaSuccess;
  if (!p.fuse_draw &&
      (e = launch_pdl(mass_kernel<DT>, dim3(p.c_end - p.c_begin, p.B), kMassThreads, 0, stream, SV_KERNEL_MASS, p)) !=
          cudaSuccess)
    return e;
  return launch_pdl(pick_kernel<DT>, dim3(p.B), kPickThreads, 0, stream, SV_KERNEL_PICK, p);
}

// One step of a sampled verification over a vocabulary shard (row f4): the stream of this
// shard's chunks, the accept chain over every chunk's records, this shard's draw weights, or the
// draw.
template <int DT>
cudaError_t launch_phase_t(const VerifyParams& p, int phase, cudaStream_t stream) {
  switch (phase) {
    case SV_PHASE_STATS:
      return launch_row_stats_t<DT>(p, stream);
    case SV_PHASE_ACCEPT: {
      const size_t csmem = fin_layout(p.rows_per_req, p.nchunks, p.Kmax).bytes;
      return launch_pdl(combine_kernel<DT>, dim3(1, p.B), kCombineThreads, csmem, stream, SV_KERNEL_COMBINE, p);
    }
    case SV_PHASE_WEIGHTS:
      return launch_pdl(mass_kernel<DT>, dim3(p.c_end - p.c_begin, p.B), kMassThreads, 0, stream, SV_KERNEL_MASS, p);
    default:
      return launch_pdl(pick_kernel<DT>, dim3(p.B), kPickThreads, 0, stream, SV_KERNEL_PICK, p);
  }
}

}  // namespace

// Vocabulary chunks of at most one 16 KB stage.  bf16 rows are cut into full stages (and one short
// chunk at the end), which the stream reduces without predicates (an A/B on GB300: C5 75.8 -> 73.8
// us per step against equal chunks of 8000); fp32 rows into equal chunks.
void vocab_tiling(int V, sv_dtype dt, int* chunk_len, int* nchunks) {
  const int elt = dt == SV_BF16 ? 2 : 4;
  const int vec = 16 / elt;
  const int stage_elems = kStageBytes / elt;
  int nc = (V + stage_elems - 1) / stage_elems;
  if (nc < 1) nc = 1;
  int cl = (V + nc - 1) / nc;
  cl = (cl + vec - 1) / vec * vec;
  if (cl > stage_elems || (dt == SV_BF16 && nc > 1)) cl = stage_elems;
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

int launch_stats(const VerifyParams& p, sv_dtype dt, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return static_cast<int>(dt == SV_BF16 ? launch_row_stats_t<SV_BF16>(p, s) : launch_row_stats_t<SV_F32>(p, s));
}

int launch_phase(const VerifyParams& p_in, sv_dtype dt, int phase, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  VerifyParams p = p_in;
  p.fuse_draw = 0;  // the draw weights come from the shards' own weights step
  return static_cast<int>(dt == SV_BF16 ? launch_phase_t<SV_BF16>(p, phase, s) : launch_phase_t<SV_F32>(p, phase, s));
}

int launch_verify(const VerifyParams& p_in, sv_dtype dt, bool sampled, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  VerifyParams p = p_in;
  p.fuse_draw = sampled && static_cast<int64_t>(p.rows_per_req) * p.nchunks <= kFuseDrawMaxRecords ? 1 : 0;
  return static_cast<int>(dt == SV_BF16 ? launch_verify_t<SV_BF16>(p, sampled, s)
                                        : launch_verify_t<SV_F32>(p, sampled, s));
}

}  // namespace sv
