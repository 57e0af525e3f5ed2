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
// memory; with s >= 0 the float bits order like unsigned integers.
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

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
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

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const ScheduleParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int B = p.B, Dmax = p.Dmax, P = p.sort_size;
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);                  // [P]
  float* alpha_s = reinterpret_cast<float*>(smem + static_cast<size_t>(P) * 8);             // [B * Dmax]
  int* cnt = reinterpret_cast<int*>(smem + static_cast<size_t>(P) * 8 +
                                    ((static_cast<size_t>(B) * Dmax * 4 + 15) & ~size_t(15)));  // [B]
  __shared__ int warp_tot[33];
  __shared__ unsigned int bad;
  __shared__ long long usum[8];
  __shared__ int cand[8];
  __shared__ int ncand;
  __shared__ int bestK;
  __shared__ long long bestU;

  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  if (tid < 8) usum[tid] = 0;

  // 0. one round of asynchronous copies: every confidence and every draft length
  for (int j = tid; j < B * Dmax; j += kSchedThreads) {
    const int i = j / Dmax, k = j - (j / Dmax) * Dmax;
    cp_async4(alpha_s + j, p.alpha + static_cast<int64_t>(i) * p.alpha_stride + k);
  }
  if (p.draft_len)
    for (int i = tid; i < B; i += kSchedThreads) cp_async4(cnt + i, p.draft_len + i);
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // 1. per-request lengths and their exclusive scan (each thread owns a contiguous block)
  const int per = (B + kSchedThreads - 1) / kSchedThreads;
  const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
  int local = 0;
  for (int i = r0; i < r1; ++i) {
    const int D = p.draft_len ? cnt[i] : Dmax;
    if (D < 0 || D > Dmax) atomicOr(&bad, SV_DEV_BAD_DRAFT_LEN);
    const int Dc = min(max(D, 0), Dmax);
    cnt[i] = Dc;
    local += Dc;
  }
  int excl;
  const int M = block_exclusive_scan(local, &excl, warp_tot);

  // 2. prefix-confidence products and sort keys of the non-root slots
  for (int i = r0, start = excl; i < r1; ++i) {
    const int D = cnt[i];
    float s = 1.0f;
    for (int k = 1; k <= D; ++k) {
      const float a = alpha_s[i * Dmax + (k - 1)];
      if (!(a >= 0.0f && a <= 1.0f)) atomicOr(&bad, SV_DEV_BAD_ALPHA);
      s = __fmul_rn(s, a);
      const uint32_t bits = __float_as_uint(s > 0.0f ? s : 0.0f);  // -0 sorts as +0
      keys[start + k - 1] = (static_cast<unsigned long long>(~bits) << 32) |
                            (static_cast<unsigned long long>(i) << 10) | static_cast<unsigned long long>(k);
    }
    start += D;
  }
  for (int j = M + tid; j < P; j += kSchedThreads) keys[j] = ~0ull;
  __syncthreads();

  if (bad) {
    if (tid == 0) {
      atomicOr(p.status, bad);
      *p.out_total_K = -1;
      if (p.out_utility_q48) *p.out_utility_q48 = -1;
    }
    for (int i = tid; i < B; i += kSchedThreads) p.out_keep_len[i] = 0;
    if (p.out_row_offsets)
      for (int i = tid; i <= B; i += kSchedThreads) p.out_row_offsets[i] = i;
    return;
  }

  // 3. bitonic sort, ascending key == (s desc, request asc, position asc)
  switch (P / kSchedThreads) {
    case 1: bitonic_sort<1>(keys, P); break;
    case 2: bitonic_sort<2>(keys, P); break;
    case 4: bitonic_sort<4>(keys, P); break;
    case 8: bitonic_sort<8>(keys, P); break;
    default: bitonic_sort<16>(keys, P); break;
  }

  // 4. candidate budgets (eq. K_rho), clipped to [B, cap]: one thread per ratio
  const int N = M + B;
  if (tid < 8) {
    int K = -1;
    if (tid < p.n_ratios) {
      const int cap = p.budget > 0 ? min(p.budget, N) : N;
      K = static_cast<int>(ceil(static_cast<double>(p.ratios[tid]) * static_cast<double>(N)));
      K = max(B, K);
      K = min(K, cap);
      K = max(K, B);
    }
    cand[tid] = K;
  }
  __syncthreads();
  if (tid == 0) {  // sort ascending, drop duplicates and unused slots
    int nc = 0;
    for (int a = 0; a < 8; ++a) {
      const int K = cand[a];
      if (K < 0) continue;
      bool dup = false;
      for (int c = 0; c < nc; ++c) dup |= cand[c] == K;
      if (dup) continue;
      int pos = nc++;
      while (pos > 0 && cand[pos - 1] > K) {
        cand[pos] = cand[pos - 1];
        --pos;
      }
      cand[pos] = K;
    }
    ncand = nc;
  }
  __syncthreads();

  // 5. U(K) for every candidate: exact integer sums over the sorted prefix
  long long part[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const int nc = ncand;
  int lim[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) lim[c] = c < nc ? cand[c] - B : 0;
  for (int j = tid; j < M; j += kSchedThreads) {
    const long long q = q48_of_key(keys[j]);
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
    if ((tid & 31) == 0 && v != 0) atomicAdd(reinterpret_cast<unsigned long long*>(&usum[c]),
                                             static_cast<unsigned long long>(v));
  }
  __syncthreads();

  // 6. objective (float64 with explicit rounding: no contraction), one thread per candidate;
  //    ties -> smaller K
  __shared__ double obj_s[8];
  if (tid < nc) {
    const long long U = usum[tid] + static_cast<long long>(B) * (1ll << 48);
    const double util = __dmul_rn(__ll2double_rn(U), kTwoM48);
    const double cost = __dadd_rn(p.cost_a, __dmul_rn(p.cost_b, static_cast<double>(cand[tid])));
    obj_s[tid] = p.objective == SV_OBJ_NET ? __dsub_rn(util, cost) : __ddiv_rn(util, cost);
    usum[tid] = U;
  }
  __syncthreads();
  if (tid == 0) {
    int bc = 0;
    for (int c = 1; c < nc; ++c)
      if (obj_s[c] > obj_s[bc]) bc = c;
    bestK = cand[bc];
    bestU = usum[bc];
  }
  for (int i = tid; i < B; i += kSchedThreads) cnt[i] = 0;
  __syncthreads();

  // 7. per-request kept depth and packed row offsets
  const int Kb = bestK;
  for (int j = tid; j < Kb - B; j += kSchedThreads) atomicAdd(&cnt[(keys[j] >> 10) & 0x3FFFFFull], 1);
  __syncthreads();
  int loc = 0;
  for (int i = r0; i < r1; ++i) {
    p.out_keep_len[i] = cnt[i];
    loc += cnt[i] + 1;
  }
  int rexcl;
  const int rtot = block_exclusive_scan(loc, &rexcl, warp_tot);
  if (p.out_row_offsets) {
    for (int i = r0, o = rexcl; i < r1; ++i) {
      p.out_row_offsets[i] = o;
      o += cnt[i] + 1;
    }
    if (tid == 0) p.out_row_offsets[B] = rtot;
  }
  if (tid == 0) {
    *p.out_total_K = Kb;
    if (p.out_utility_q48) *p.out_utility_q48 = bestU;
  }
}

bool g_sched_attr_set = false;

}  // namespace

int launch_schedule(const ScheduleParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t dyn = static_cast<size_t>(p.sort_size) * 8 +
                     ((static_cast<size_t>(p.B) * p.Dmax * 4 + 15) & ~size_t(15)) + static_cast<size_t>(p.B) * 4;
  cudaError_t e;
  if (!g_sched_attr_set) {
    const int max_dyn = SV_MAX_SCHEDULE_SLOTS * 8 + SV_MAX_SCHEDULE_SLOTS * 4 + SV_MAX_BATCH * 4;
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
