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
// memory; with s >= 0 the float bits order like unsigned integers.  U(K) for every candidate
// comes from one integer prefix scan of the sorted order.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

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

// Inclusive scan, across the CTA, of E 64-bit values per thread: thread t's value e belongs to
// row e at column t (element e * kSchedThreads + t of the sorted order).  On return v[e] holds
// the inclusive prefix within its row and row_tot[e] row e's total.
template <int E>
__device__ void block_row_scan64(long long (&v)[E], long long* wtot, long long* row_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int e = 0; e < E; ++e) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xFFFFFFFFu, v[e], o);
      if (lane >= o) v[e] += y;
    }
    if (lane == 31) wtot[e * 32 + warp] = v[e];
  }
  __syncthreads();
  if (warp == 0) {
    for (int e = 0; e < E; ++e) {
      const long long w = wtot[e * 32 + lane];
      long long wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
        if (lane >= o) wi += y;
      }
      wtot[e * 32 + lane] = wi - w;  // exclusive prefix of the warp totals
      if (lane == 31) row_tot[e] = wi;
    }
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] += wtot[e * 32 + warp];
}

struct SchedSmem {
  long long wtot[16 * 32];
  long long row_tot[16];
  long long ucand[8];
  double obj[8];
  int cand[8];
  int ncand;
  int warp_tot[33];
  unsigned int bad;
};

// Sort, then U(K) of every candidate, the objective, and the chosen K (same in every thread).
template <int E>
__device__ void sort_and_choose(const ScheduleParams& p, unsigned long long* keys, int P, int B, SchedSmem& sm,
                                int* Kb, long long* Ub) {
  const int tid = threadIdx.x;
  // ascending key == (s desc, request asc, position asc)
  bitonic_sort<E>(keys, P);
  const int nc = sm.ncand;  // written by thread 0 before the sort's barriers

  // U(K) = sum of round(s * 2^48) over the first K - B sorted slots: one scan of the sorted
  // order, read at each candidate (exact integer sums)
  long long v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = q48_of_key(keys[e * kSchedThreads + tid]);  // padding gives 0
  block_row_scan64<E>(v, sm.wtot, sm.row_tot);
  for (int c = 0; c < nc; ++c) {
    const int L = sm.cand[c] - B;  // slots beyond the always-kept roots
    if (L == 0) {
      if (tid == 0) sm.ucand[c] = 0;
    } else if (((L - 1) & (kSchedThreads - 1)) == tid) {
      const int er = (L - 1) / kSchedThreads;
      long long u = 0;
      for (int e = 0; e < er; ++e) u += sm.row_tot[e];
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (e == er) u += v[e];
      sm.ucand[c] = u;
    }
  }
  __syncthreads();

  // objective (float64 with explicit rounding: no contraction), one thread per candidate
  if (tid < nc) {
    const long long U = sm.ucand[tid] + static_cast<long long>(B) * (1ll << 48);
    const double util = __dmul_rn(__ll2double_rn(U), kTwoM48);
    const double cost = __dadd_rn(p.cost_a, __dmul_rn(p.cost_b, static_cast<double>(sm.cand[tid])));
    sm.obj[tid] = p.objective == SV_OBJ_NET ? __dsub_rn(util, cost) : __ddiv_rn(util, cost);
    sm.ucand[tid] = U;
  }
  __syncthreads();
  int bc = 0;  // ties -> the smaller K (candidates are ascending)
  for (int c = 1; c < nc; ++c)
    if (sm.obj[c] > sm.obj[bc]) bc = c;
  *Kb = sm.cand[bc];
  *Ub = sm.ucand[bc];
}

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const ScheduleParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int B = p.B, Dmax = p.Dmax, P = p.sort_size;
  // keys [P]; kept flags [Dmax][B], position-major: request i's position k at (k - 1) * B + i
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);
  uint8_t* kept = smem + static_cast<size_t>(P) * 8;
  __shared__ SchedSmem sm;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) sm.bad = 0;
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
    for (int k0 = 0; k0 < Dmax; k0 += 8) {
      float a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = k0 + u < Dmax ? __ldg(a_row + k0 + u) : 0.0f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
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
  for (int j = B * Dmax + tid; j < P; j += kSchedThreads) keys[j] = ~0ull;
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

  // 1. candidate budgets (eq. K_rho) clipped to [B, cap], ascending, duplicates dropped.  Thread
  //    0 computes them while the other threads start the sort; the sort's barriers publish them.
  const int N = M + B;
  if (tid == 0) {
    const int cap = p.budget > 0 ? min(p.budget, N) : N;
    int nc = 0;
    for (int r = 0; r < p.n_ratios; ++r) {
      int K = static_cast<int>(ceil(static_cast<double>(p.ratios[r]) * static_cast<double>(N)));
      K = max(K, B);
      K = min(K, cap);
      K = max(K, B);
      bool dup = false;
      for (int c = 0; c < nc; ++c) dup |= sm.cand[c] == K;
      if (dup) continue;
      int pos = nc++;
      while (pos > 0 && sm.cand[pos - 1] > K) {
        sm.cand[pos] = sm.cand[pos - 1];
        --pos;
      }
      sm.cand[pos] = K;
    }
    sm.ncand = nc;
  }

  // 2-5. sort, utilities, objective, chosen K
  int Kb = B;
  long long Ub = 0;
  switch (P / kSchedThreads) {
    case 1: sort_and_choose<1>(p, keys, P, B, sm, &Kb, &Ub); break;
    case 2: sort_and_choose<2>(p, keys, P, B, sm, &Kb, &Ub); break;
    case 4: sort_and_choose<4>(p, keys, P, B, sm, &Kb, &Ub); break;
    case 8: sort_and_choose<8>(p, keys, P, B, sm, &Kb, &Ub); break;
    default: sort_and_choose<16>(p, keys, P, B, sm, &Kb, &Ub); break;
  }

  // 6. kept slots: the first Kb - B sorted keys, marked at their (position, request) place; a
  //    request's kept slots are a prefix of its positions, so its depth is their count
  for (int j = tid; j < Kb - B; j += kSchedThreads) {
    const unsigned long long key = keys[j];
    const int i = static_cast<int>((key >> 10) & 0x3FFFFFull), k = static_cast<int>(key & 0x3FFull);
    kept[static_cast<int64_t>(k - 1) * B + i] = 1;
  }
  __syncthreads();

  // 7. per-request kept depth and packed row offsets
  int loc = 0;
  for (int i = r0; i < r1; ++i) {
    int n = 0;
    for (int k = 0; k < Dmax; ++k) n += kept[static_cast<int64_t>(k) * B + i];
    p.out_keep_len[i] = n;
    loc += n + 1;
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

bool g_sched_attr_set = false;

}  // namespace

int launch_schedule(const ScheduleParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // sort keys, then one kept flag per slot
  const size_t dyn = static_cast<size_t>(p.sort_size) * 8 + static_cast<size_t>(p.B) * p.Dmax;
  cudaError_t e;
  if (!g_sched_attr_set) {
    const int max_dyn = SV_MAX_SCHEDULE_SLOTS * 8 + SV_MAX_SCHEDULE_SLOTS;
    if ((e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn)) !=
        cudaSuccess)
      return static_cast<int>(e);
    g_sched_attr_set = true;
  }
  prof_before(SV_KERNEL_SCHEDULE, stream);
  schedule_kernel<<<1, kSchedThreads, dyn, s>>>(p);
  prof_after(SV_KERNEL_SCHEDULE, stream);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace sv
