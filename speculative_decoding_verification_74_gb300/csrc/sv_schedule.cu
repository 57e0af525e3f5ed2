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

__device__ __forceinline__ int64_t q48_of_key(unsigned long long key) {
  const uint32_t bits = ~static_cast<uint32_t>(key >> 32);
  const double s = static_cast<double>(__uint_as_float(bits));
  return __double2ll_rn(s * 281474976710656.0);  // exact scaling by 2^48, then round-half-even
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

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const ScheduleParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);
  int* cnt = reinterpret_cast<int*>(smem + static_cast<size_t>(p.sort_size) * 8);
  __shared__ int warp_tot[33];
  __shared__ unsigned int bad;
  __shared__ long long usum[8];
  __shared__ int cand[8];
  __shared__ int ncand;
  __shared__ int bestK;
  __shared__ long long bestU;

  const int tid = threadIdx.x;
  const int B = p.B, Dmax = p.Dmax, P = p.sort_size;
  if (tid == 0) bad = 0;
  if (tid < 8) usum[tid] = 0;
  __syncthreads();

  // 1. per-request lengths and their exclusive scan (each thread owns a contiguous block)
  const int per = (B + kSchedThreads - 1) / kSchedThreads;
  const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
  int local = 0;
  for (int i = r0; i < r1; ++i) {
    const int D = p.draft_len ? __ldg(p.draft_len + i) : Dmax;
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
      const float a = __ldg(p.alpha + static_cast<int64_t>(i) * p.alpha_stride + (k - 1));
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
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int t = tid; t < (P >> 1); t += kSchedThreads) {
        const int lo = (t / j) * 2 * j + (t % j);
        const int hi = lo + j;
        const bool up = (lo & k) == 0;
        const unsigned long long a = keys[lo], b = keys[hi];
        if ((a > b) == up) {
          keys[lo] = b;
          keys[hi] = a;
        }
      }
      __syncthreads();
    }
  }

  // 4. candidate budgets (eq. K_rho), clipped to [B, cap]
  const int N = M + B;
  if (tid == 0) {
    const int cap = p.budget > 0 ? min(p.budget, N) : N;
    int nc = 0;
    for (int r = 0; r < p.n_ratios; ++r) {
      int K = static_cast<int>(ceil(static_cast<double>(p.ratios[r]) * static_cast<double>(N)));
      K = max(B, K);
      K = min(K, cap);
      K = max(K, B);
      bool dup = false;
      for (int c = 0; c < nc; ++c) dup |= cand[c] == K;
      if (!dup) cand[nc++] = K;
    }
    // ascending order so that "ties -> smaller K" is a strict-greater scan
    for (int a = 1; a < nc; ++a)
      for (int b = a; b > 0 && cand[b - 1] > cand[b]; --b) {
        const int t = cand[b];
        cand[b] = cand[b - 1];
        cand[b - 1] = t;
      }
    ncand = nc;
  }
  __syncthreads();

  // 5. U(K) for every candidate: exact integer sums over the sorted prefix
  long long part[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const int nc = ncand;
  for (int j = tid; j < M; j += kSchedThreads) {
    const long long q = q48_of_key(keys[j]);
    for (int c = 0; c < nc; ++c)
      if (j < cand[c] - B) part[c] += q;
  }
  for (int c = 0; c < nc; ++c) {
    long long v = part[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if ((tid & 31) == 0 && v != 0) atomicAdd(reinterpret_cast<unsigned long long*>(&usum[c]),
                                             static_cast<unsigned long long>(v));
  }
  __syncthreads();

  // 6. objective (float64 with explicit rounding: no contraction), ties -> smaller K
  if (tid == 0) {
    double best = 0.0;
    int bk = -1;
    long long bu = 0;
    for (int c = 0; c < nc; ++c) {
      const long long U = usum[c] + static_cast<long long>(B) * (1ll << 48);
      const double util = __dmul_rn(__ll2double_rn(U), kTwoM48);
      const double cost = __dadd_rn(p.cost_a, __dmul_rn(p.cost_b, static_cast<double>(cand[c])));
      const double obj = p.objective == SV_OBJ_NET ? __dsub_rn(util, cost) : __ddiv_rn(util, cost);
      if (bk < 0 || obj > best) {
        best = obj;
        bk = cand[c];
        bu = U;
      }
    }
    bestK = bk;
    bestU = bu;
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
  const size_t dyn = static_cast<size_t>(p.sort_size) * 8 + static_cast<size_t>(p.B) * 4;
  cudaError_t e;
  if (!g_sched_attr_set) {
    const int max_dyn = SV_MAX_SCHEDULE_SLOTS * 8 + SV_MAX_BATCH * 4;
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
