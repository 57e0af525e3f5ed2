// D-cut verification-depth scheduling kernel of libsv (one CTA).
//
// AngelSpec explainer, section "D-cut: verification depth is a shared resource", Figure 3
// panels 2-3 and eq. K_rho; AngelSpec abstract (expected utility with a profiled cost):
//   s_{i,0} = 1, s_{i,k} = s_{i,k-1} * alpha_{i,k}               (float32, left to right)
//   every request keeps its slot 0; the other slots of the whole batch are ranked by
//   (s desc, request asc, position asc) and a global top-K is kept
//   K in { clip(max(B, ceil(rho N)), B, cap) : rho in ratios },  N = sum_i (D_i + 1)
//   U(K) = sum of round(s * 2^48) over the kept slots (exact int64, order independent)
//   pick the K maximising U / c(K) (or U - c(K)), c(K) = a + b K; ties -> smaller K
// The ranking is a bitonic sort of 64-bit keys (~bits(s) : request : position) in shared
// memory, or (up to 8192 slots) a merge of the per-request runs, which are already in order;
// with s >= 0 the float bits order like unsigned integers.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kSchedThreads = 1024;
constexpr double kTwoM48 = 3.552713678800500929355621337890625e-15;  // 2^-48

// round(s * 2^48), ties to even, for a float 0 <= s <= 1 given by its bits, in integer arithmetic
// (s = mant * 2^(exp - 150); the shift by exp - 102 is exact when non-negative).
__device__ __forceinline__ int64_t q48_of_bits(uint32_t bits) {
  const int exp = static_cast<int>((bits >> 23) & 0xFF);
  if (exp == 0) return 0;  // zero or subnormal: below 2^-126, rounds to 0
  const uint64_t mant = (bits & 0x7FFFFFu) | 0x800000u;
  const int sh = exp - 102;
  if (sh >= 0) return static_cast<int64_t>(mant << sh);
  if (sh <= -25) return 0;  // below 2^-49 even at the top of the mantissa: rounds to 0
  const int r = -sh;
  const uint64_t q = mant >> r, rem = mant & ((1ull << r) - 1), half = 1ull << (r - 1);
  return static_cast<int64_t>(q + ((rem > half || (rem == half && (q & 1))) ? 1 : 0));
}
__device__ __forceinline__ int64_t q48_of_key(unsigned long long key) {
  return q48_of_bits(~static_cast<uint32_t>(key >> 32));
}

// Block-wide exclusive scan of one int per thread (kSchedThreads threads); returns the total.
__device__ int block_exclusive_scan(int v, int* excl, int* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) warp_tot[32] = wi;
  }
  __syncthreads();
  *excl = warp_tot[warp] + incl - v;
  const int total = warp_tot[32];
  __syncthreads();
  return total;
}

// Bitonic merge step for one element: keep the smaller key when this element is the lower index
// of its pair and the pair sorts ascending (or the higher index of a descending pair).
__device__ __forceinline__ unsigned long long bitonic_keep(unsigned long long mine, unsigned long long other,
                                                           bool is_lo, bool up) {
  const unsigned long long lo = mine < other ? mine : other, hi = mine < other ? other : mine;
  return (is_lo == up) ? lo : hi;
}

// Bitonic sort of P = E * 1024 keys in shared memory, ascending.  Element index e * 1024 + tid
// lives in register r[e] of thread tid: partners 1024 or more apart are in the same thread,
// partners 32..512 apart go through shared memory, closer partners are in the same warp.
template <int E>
__device__ void bitonic_sort(unsigned long long* keys, int P) {
  const int tid = threadIdx.x, lane = tid & 31;
  unsigned long long r[E];
#pragma unroll
  for (int e = 0; e < E; ++e) r[e] = keys[e * kSchedThreads + tid];
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= kSchedThreads) {
#pragma unroll
        for (int sh = 0; sh < 4; ++sh) {
          const int jj = 1 << sh;
          if (jj < E && j == jj * kSchedThreads) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
              if ((e & jj) == 0 && (e | jj) < E) {
                const bool up = ((e * kSchedThreads + tid) & k) == 0;
                const unsigned long long a = r[e], b = r[e | jj];
                const bool swap = (a > b) == up;
                r[e] = swap ? b : a;
                r[e | jj] = swap ? a : b;
              }
            }
          }
        }
      } else if (j >= 32) {
#pragma unroll
        for (int e = 0; e < E; ++e) keys[e * kSchedThreads + tid] = r[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int idx = e * kSchedThreads + tid, partner = idx ^ j;
          r[e] = bitonic_keep(r[e], keys[partner], idx < partner, (idx & k) == 0);
        }
        __syncthreads();
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, r[e], j);
          r[e] = bitonic_keep(r[e], other, (lane & j) == 0, ((e * kSchedThreads + tid) & k) == 0);
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) keys[e * kSchedThreads + tid] = r[e];
  __syncthreads();
}

struct SchedSmem {
  long long usum[8];
  double obj[8];
  int cand[8];
  int ncand;
  int warp_tot[33];
  unsigned int bad;
};

// ceil(r * N) for a float 0 < r <= 1 and 0 <= N < 2^31, exactly, in integer arithmetic
// (r = mant * 2^-sh with sh >= 23; mant * N < 2^56).
__device__ __forceinline__ int ceil_ratio_times(float r, int N) {
  const uint32_t b = __float_as_uint(r);
  const int ex = static_cast<int>((b >> 23) & 0xFF);
  const uint64_t mant = (b & 0x7FFFFFu) | (ex ? 0x800000u : 0u);
  const int sh = 150 - (ex ? ex : 1);
  const uint64_t prod = mant * static_cast<uint64_t>(N);
  if (prod == 0) return 0;
  if (sh >= 64) return 1;
  return static_cast<int>((prod + ((1ull << sh) - 1)) >> sh);
}

// Candidate budgets (eq. K_rho) clipped to [B, cap], ascending, duplicates dropped, computed by
// warp 0: lane r takes ratio r, the lanes sort the values with a bitonic network over shuffles,
// and lane 0 writes the distinct ones.
__device__ void candidates(const ScheduleParams& p, int N, int B, SchedSmem& sm) {
  const int lane = threadIdx.x & 31;
  const int cap = p.budget > 0 ? min(p.budget, N) : N;
  int K = INT_MAX;
  if (lane < p.n_ratios) K = max(min(max(ceil_ratio_times(p.ratios[lane], N), B), cap), B);
#pragma unroll
  for (int k = 2; k <= 8; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const int other = __shfl_xor_sync(0xFFFFFFFFu, K, j);
      const bool up = (lane & k) == 0, lower = (lane & j) == 0;
      K = lower == up ? min(K, other) : max(K, other);
    }
  const int prev = __shfl_up_sync(0xFFFFFFFFu, K, 1);
  const bool keep = lane < 8 && K != INT_MAX && (lane == 0 || K != prev);
  const unsigned mask = __ballot_sync(0xFFFFFFFFu, keep);
  if (keep) sm.cand[__popc(mask & ((1u << lane) - 1u))] = K;
  if (lane == 0) sm.ncand = __popc(mask);
}

// Merge sort of the B runs of Dmax keys (request q's keys, ascending along its positions) in
// ceil(log2 B) levels.  At level 0 run q's key t sits at a[t * B + q] (position-major); later
// levels hold runs contiguously.  A key of the left run of a pair lands at its index plus the
// number of partner keys below it, a key of the right run at its index plus the number of
// partner keys at or below it: a stable merge, so equal keys (the padding) stay valid.
// Returns the buffer holding the sorted keys.
__device__ unsigned long long* merge_runs(unsigned long long* a, unsigned long long* b, int B, int Dmax) {
  const int tid = threadIdx.x;
  const int n = B * Dmax;
  if (B <= 1) return a;  // one run: position-major is already contiguous
  // level 0: pairs of single requests; threads walk the position-major order
  for (int jj = tid; jj < n; jj += kSchedThreads) {
    const int t = jj / B, q = jj - t * B;
    const unsigned long long x = a[jj];
    const int pq = q ^ 1;
    int cnt = 0;
    if (pq < B) {
      const bool left = q < pq;
      int lo = 0, len = Dmax;
      while (len > 0) {
        const int half = len >> 1;
        const unsigned long long v = a[(lo + half) * B + pq];
        if (left ? v < x : v <= x) {
          lo += half + 1;
          len -= half + 1;
        } else {
          len = half;
        }
      }
      cnt = lo;
    }
    b[(pq < B ? min(q, pq) : q) * Dmax + t + cnt] = x;
  }
  __syncthreads();
  unsigned long long* src = b;
  unsigned long long* dst = a;
  // this thread's slots (at most kMergeMaxSlots / kSchedThreads) and their runs, for every level
  constexpr int kPer = (kMergeMaxSlots + kSchedThreads - 1) / kSchedThreads;
  int qs[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) qs[e] = Dmax > 0 ? (tid + e * kSchedThreads) / Dmax : 0;
  for (int lvl = 1; (1 << lvl) < B; ++lvl) {
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int j = tid + e * kSchedThreads;
      if (j >= n) break;
      const int q = qs[e];
      const int r = q >> lvl, pr = r ^ 1;
      const int rq = r << lvl, pq = pr << lvl;
      const unsigned long long x = src[j];
      if (pq >= B) {  // no partner run at this level
        dst[j] = x;
        continue;
      }
      const bool left = r < pr;
      const int pbase = pq * Dmax;
      int lo = 0, len = (min(pq + (1 << lvl), B) - pq) * Dmax;
      while (len > 0) {
        const int half = len >> 1;
        const unsigned long long v = src[pbase + lo + half];
        if (left ? v < x : v <= x) {
          lo += half + 1;
          len -= half + 1;
        } else {
          len = half;
        }
      }
      dst[min(rq, pq) * Dmax + (j - rq * Dmax) + lo] = x;
    }
    __syncthreads();
    unsigned long long* t = src;
    src = dst;
    dst = t;
  }
  return src;
}

// Cost of verifying K tokens (float64, explicit rounding): the linear model, or the
// latency table interpolated linearly between knots (slope form) with its end values held
// outside them.  The segment is found by an unrolled count, so the knot loads are
// independent of each other.
__device__ double cost_of(const ScheduleParams& p, int K) {
  if (p.n_cost == 0) return __dadd_rn(p.cost_a, __dmul_rn(p.cost_b, static_cast<double>(K)));
  const int n = p.n_cost;
  if (K <= p.cost_K[0]) return p.cost_c[0];
  if (K >= p.cost_K[n - 1]) return p.cost_c[n - 1];
  int j = 0;  // cost_K[0] < K < cost_K[n - 1]: the last j <= n - 2 with cost_K[j] <= K
#pragma unroll
  for (int i = 1; i < SV_MAX_COST_KNOTS - 1; ++i) j += (i < n - 1 && p.cost_K[i] <= K) ? 1 : 0;
  return __dadd_rn(p.cost_c[j], __dmul_rn(p.cost_s[j], static_cast<double>(K - p.cost_K[j])));
}

// U(K) of every candidate (exact integer sums over the first K - B sorted keys), the
// objective, and the chosen K (same in every thread).
__device__ void choose(const ScheduleParams& p, const unsigned long long* sorted, int n, int B, SchedSmem& sm,
                       int* Kb, long long* Ub) {
  const int tid = threadIdx.x;
  const int nc = sm.ncand;
  int lim[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) lim[c] = c < nc ? sm.cand[c] - B : 0;
  long long part[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const int jmax = min(sm.cand[nc - 1] - B, n);  // the largest candidate's slots
  for (int j = tid; j < jmax; j += kSchedThreads) {
    const long long q = q48_of_key(sorted[j]);
#pragma unroll
    for (int c = 0; c < 8; ++c)
      if (j < lim[c]) part[c] += q;
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    if (c >= nc) break;
    long long v = part[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if ((tid & 31) == 0 && v != 0)
      atomicAdd(reinterpret_cast<unsigned long long*>(&sm.usum[c]), static_cast<unsigned long long>(v));
  }
  __syncthreads();

  // objective (float64 with explicit rounding: no contraction), one thread per candidate
  if (tid < nc) {
    const long long U = sm.usum[tid] + static_cast<long long>(B) * (1ll << 48);
    const double util = __dmul_rn(__ll2double_rn(U), kTwoM48);
    const double cost = cost_of(p, sm.cand[tid]);
    sm.obj[tid] = p.objective == SV_OBJ_NET ? __dsub_rn(util, cost) : __ddiv_rn(util, cost);
    sm.usum[tid] = U;
  }
  __syncthreads();
  int bc = 0;  // ties -> the smaller K (candidates are ascending)
  for (int c = 1; c < nc; ++c)
    if (sm.obj[c] > sm.obj[bc]) bc = c;
  *Kb = sm.cand[bc];
  *Ub = sm.usum[bc];
}

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const ScheduleParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int B = p.B, Dmax = p.Dmax, n = B * Dmax;
  // merge mode: keys [n] (position-major) + second buffer [n]; bitonic mode: keys [P]; then one
  // kept flag per slot, position-major: request i's position k at (k - 1) * B + i
  const int P = p.sort_size;
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);
  unsigned long long* keys2 = keys + n;
  uint8_t* kept = smem + static_cast<size_t>(p.merge ? 2 * n : P) * 8;
  __shared__ SchedSmem sm;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) sm.bad = 0;
  if (tid < 8) sm.usum[tid] = 0;
  __syncthreads();

  // 0. each thread owns a contiguous block of requests: their lengths and confidences (all Dmax
  //    confidences of a request are requested together; entries past D_i are not used), the
  //    prefix products (float32, left to right) and the sort keys (~bits(s) : request :
  //    position) of their non-root slots, stored position-major so that neighbouring threads
  //    write neighbouring words.  Slots past D_i get the largest key (sorted last, never kept).
  const int per = (B + kSchedThreads - 1) / kSchedThreads;
  const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
  int local = 0;
  for (int i = r0; i < r1; ++i) {
    const int D = p.draft_len ? __ldg(p.draft_len + i) : Dmax;
    if (D < 0 || D > Dmax) atomicOr(&sm.bad, SV_DEV_BAD_DRAFT_LEN);
    const int Dc = min(max(D, 0), Dmax);
    const float* a_row = p.alpha + static_cast<int64_t>(i) * p.alpha_stride;
    float s = 1.0f;
    for (int k0 = 0; k0 < Dmax; k0 += 16) {  // 16 confidences per round trip
      float a[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) a[u] = k0 + u < Dmax ? __ldg(a_row + k0 + u) : 0.0f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int k = k0 + u + 1;
        if (k > Dmax) break;
        unsigned long long key = ~0ull;
        if (k <= Dc) {
          if (!(a[u] >= 0.0f && a[u] <= 1.0f)) atomicOr(&sm.bad, SV_DEV_BAD_ALPHA);
          s = __fmul_rn(s, a[u]);
          const uint32_t bits = __float_as_uint(s > 0.0f ? s : 0.0f);  // -0 sorts as +0
          key = (static_cast<unsigned long long>(~bits) << 32) | (static_cast<unsigned long long>(i) << 10) |
                static_cast<unsigned long long>(k);
        }
        keys[static_cast<int64_t>(k - 1) * B + i] = key;
        kept[static_cast<int64_t>(k - 1) * B + i] = 0;
      }
    }
    local += Dc;
  }
  if (!p.merge)
    for (int j = n + tid; j < P; j += kSchedThreads) keys[j] = ~0ull;
  int wsum = local;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xFFFFFFFFu, wsum, o);
  if (lane == 0) sm.warp_tot[warp] = wsum;
  __syncthreads();
  int M = 0;  // non-root slots of the batch
#pragma unroll
  for (int w = 0; w < kSchedThreads / 32; ++w) M += sm.warp_tot[w];

  if (sm.bad) {
    if (tid == 0) {
      atomicOr(p.status, sm.bad);
      *p.out_total_K = -1;
      if (p.out_utility_q48) *p.out_utility_q48 = -1;
    }
    for (int i = tid; i < B; i += kSchedThreads) p.out_keep_len[i] = 0;
    if (p.out_row_offsets)
      for (int i = tid; i <= B; i += kSchedThreads) p.out_row_offsets[i] = i;
    return;
  }

  // 1. candidate budgets: warp 0 computes them before it joins the ranking (whose barriers
  //    publish them)
  if (warp == 0) candidates(p, M + B, B, sm);

  // 2-5. rank the non-root slots (s desc, request asc, position asc == ascending key), then
  //      utilities, objective, chosen K
  const unsigned long long* sorted;
  if (p.merge) {
    sorted = merge_runs(keys, keys2, B, Dmax);
    if (B <= 1) __syncthreads();  // no merge level ran: publish the candidates
  } else {
    switch (P / kSchedThreads) {
      case 1: bitonic_sort<1>(keys, P); break;
      case 2: bitonic_sort<2>(keys, P); break;
      case 4: bitonic_sort<4>(keys, P); break;
      case 8: bitonic_sort<8>(keys, P); break;
      default: bitonic_sort<16>(keys, P); break;
    }
    sorted = keys;
  }
  int Kb;
  long long Ub;
  choose(p, sorted, p.merge ? n : P, B, sm, &Kb, &Ub);

  // 6. kept slots: the first Kb - B sorted keys, marked at their (position, request) place; a
  //    request's kept slots are a prefix of its positions, so its depth is their count
  for (int j = tid; j < Kb - B; j += kSchedThreads) {
    const unsigned long long key = sorted[j];
    const int i = static_cast<int>((key >> 10) & 0x3FFFFFull), k = static_cast<int>(key & 0x3FFull);
    kept[static_cast<int64_t>(k - 1) * B + i] = 1;
  }
  __syncthreads();

  // 7. per-request kept depth and packed row offsets
  int loc = 0;
  for (int i = r0; i < r1; ++i) {
    int cnt = 0;
    for (int k = 0; k < Dmax; ++k) cnt += kept[static_cast<int64_t>(k) * B + i];
    p.out_keep_len[i] = cnt;
    loc += cnt + 1;
  }
  int rexcl;
  const int rtot = block_exclusive_scan(loc, &rexcl, sm.warp_tot);
  if (p.out_row_offsets) {
    for (int i = r0, o = rexcl; i < r1; ++i) {
      p.out_row_offsets[i] = o;
      o += p.out_keep_len[i] + 1;
    }
    if (tid == 0) p.out_row_offsets[B] = rtot;
  }
  if (tid == 0) {
    *p.out_total_K = Kb;
    if (p.out_utility_q48) *p.out_utility_q48 = Ub;
  }
}

// the kernel's shared-memory attribute, set once per device under a lock
constexpr int kMaxDevices = 64;
bool g_sched_attr_set[kMaxDevices] = {};
std::mutex g_sched_mu;

}  // namespace

int launch_schedule(const ScheduleParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // sort keys (two buffers when merging), then one kept flag per slot
  const size_t n = static_cast<size_t>(p.B) * p.Dmax;
  const size_t dyn = (p.merge ? 2 * n : static_cast<size_t>(p.sort_size)) * 8 + n;
  cudaError_t e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return static_cast<int>(e);
  if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(cudaErrorInvalidDevice);
  {
    std::lock_guard<std::mutex> lk(g_sched_mu);
    if (!g_sched_attr_set[dev]) {
      const int max_dyn = SV_MAX_SCHEDULE_SLOTS * 8 + SV_MAX_SCHEDULE_SLOTS;
      if ((e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn)) !=
          cudaSuccess)
        return static_cast<int>(e);
      g_sched_attr_set[dev] = true;
    }
  }
  prof_before(SV_KERNEL_SCHEDULE, stream);
  schedule_kernel<<<1, kSchedThreads, dyn, s>>>(p);
  prof_after(SV_KERNEL_SCHEDULE, stream);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace sv
