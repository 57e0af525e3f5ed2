// Device helpers shared by the libsv kernels: Philox4x32-10, mbarrier and
// bulk-copy wrappers (inline PTX, sm_90+ forms used on sm_103a), bf16 unpacking,
// bounded waits.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "sv_internal.h"

namespace sv {

// ---------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of the 4x32 S-box; each round
// multiplies counter words 0 and 2 by fixed odd constants, and the key advances by the two Weyl
// increments between rounds.  Counter = (position, request, purpose, round), key = seed.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint64_t seed) {
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return c0;
}

// u in [0, 1): the 24 high bits of word 0 times 2^-24 (exact in float and double).
__device__ __forceinline__ double philox_uniform(uint64_t seed, uint32_t position, uint32_t request,
                                                 uint32_t purpose, uint32_t round) {
  return static_cast<double>(philox_word0(position, request, purpose, round, seed) >> 8) *
         (1.0 / 16777216.0);
}

// ---------------------------------------------------------------------------------------------
// small math
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Pairs of floats in one 64-bit register for the packed f32x2 arithmetic of sm_100 and later:
// one instruction performs two independently rounded float operations.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// (2^(x.lo k - c), 2^(x.hi k - c)) with k2 = (k, k) and nc2 = (-c, -c).
__device__ __forceinline__ f32x2 f2_exp2_offset(f32x2 x, f32x2 k2, f32x2 nc2) {
  float d0, d1;
  f2_unpack(f2_fma(x, k2, nc2), d0, d1);
  return f2_pack(ex2_approx(d0), ex2_approx(d1));
}

template <int DT>
__device__ __forceinline__ float load_logit(const void* row, int64_t v) {
  if constexpr (DT == SV_BF16) {
    const uint16_t b = __ldg(reinterpret_cast<const uint16_t*>(row) + v);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  } else {
    return __ldg(reinterpret_cast<const float*>(row) + v);
  }
}

// Exponent offset of a sampled row piece whose largest logit is m: c(m) = rint(m k), an
// integer-valued float.  A piece stores (m, s) with s = sum of 2^(x k - c(m)) over its logits:
// each term is one fused multiply-add and one ex2, every term is at most 2^0.5, and two pieces'
// sums rescale to a common offset by exact powers of two.
__device__ __forceinline__ float exp_offset(float m, float k) { return rintf(__fmul_rn(m, k)); }

// 2^d for an integer-valued d <= 0 (0 below the normal float range).
__device__ __forceinline__ float pow2_nonpos(float d) {
  const int e = static_cast<int>(fmaxf(d, -127.0f));
  return e <= -127 ? 0.0f : __int_as_float((e + 127) << 23);
}

// Merge two (max, sum of 2^(x k - c(max))) pairs.  A max of -inf means an empty sum.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float k) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  const float M = fmaxf(m, m2);
  const float C = exp_offset(M, k);
  s = s * pow2_nonpos(exp_offset(m, k) - C) + s2 * pow2_nonpos(exp_offset(m2, k) - C);
  m = M;
}

// (value, index) argmax merge: larger value wins, ties go to the lower index.
// An index of -1 means "no element seen"; -inf is an ordinary value here (an all -inf row
// yields its first index, like a first-occurrence argmax).
__device__ __forceinline__ void merge_argmax(float& m, int& idx, float m2, int idx2) {
  if (idx2 < 0) return;
  if (idx < 0 || m2 > m || (m2 == m && idx2 < idx)) {
    m = m2;
    idx = idx2;
  }
}

// ---------------------------------------------------------------------------------------------
// mbarrier / bulk copy (inline PTX)
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// try_wait with a suspend-time hint: a waiting thread sleeps until the phase completes (or the
// hint, in ns, runs out) instead of spinning and taking issue slots from working warps.
constexpr uint32_t kSuspendHintNs = 100000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
// Non-blocking test of a phase (no suspend).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: gives up after limit_ns (~2 s by default; or 2^24 polls), records
// SV_DEV_TIMEOUT and returns false.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitMaxPolls = 1u << 24;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  // a few quick polls, then back off with nanosleep so a waiting warp takes few issue slots;
  // the timer is read only once a wait runs long
  for (uint32_t it = 0; it < 4; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 4; it < kWaitMaxPolls; ++it) {
    __nanosleep(it < 64 ? 32 : 256);
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0 && globaltimer_ns() - t0 > limit_ns) break;
  }
  atomicOr(status, SV_DEV_TIMEOUT);
  return false;
}
// Bounded wait by polling (test_wait with a short sleep): for a wait whose copies were issued
// just before, where try_wait's suspension can oversleep the phase by microseconds.  Gives up
// after limit_ns, records SV_DEV_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait_poll(uint64_t* bar, uint32_t parity, uint32_t* status,
                                               uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1; it < kWaitMaxPolls; ++it) {
    __nanosleep(20);
    if (mbar_test_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) break;
  }
  atomicOr(status, SV_DEV_TIMEOUT);
  return false;
}
// Philox uniform as float (exact: 24 significant bits).
__device__ __forceinline__ float philox_uniform_f(uint64_t seed, uint32_t position, uint32_t request,
                                                  uint32_t purpose, uint32_t round) {
  return static_cast<float>(philox_word0(position, request, purpose, round, seed) >> 8) * (1.0f / 16777216.0f);
}
// 1-D bulk copy global -> shared, completion signalled on `bar` with `bytes` transaction bytes.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// The same with an L2 cache-eviction policy for the copied lines (createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Barrier of every thread of the thread-block cluster; orders the memory accesses before it
// (release) before those after it (acquire) across the cluster's CTAs.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Named barrier over `nthreads` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}
// Programmatic dependent launch controls.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace sv
