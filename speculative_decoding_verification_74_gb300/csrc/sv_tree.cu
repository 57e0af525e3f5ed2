// Tree (multi-candidate) verification of libsv: multi-step speculative sampling (Miao et al.,
// "SpecInfer: Accelerating Large Language Model Serving with Tree-based Speculative Inference and
// Verification", ASPLOS 2024, section 4.2) over a token tree per request.
//
// The streaming kernel first reduces every node row of the call (target rows of all nodes, draft
// rows of the sampled requests' nodes) into chunk records, as it does for a chain.  The walk
// kernel then walks each request from the root (on a cluster of CTAs, below):
//   * every node row's statistics (max, sum of 2^(x k - c), argmax) are merged from its chunk
//     records up front, one row per warp across the cluster, and shared through distributed
//     shared memory;
//   * the accept test of a child needs p and q at the child's token only: two logits;
//   * after j rejections at a node, the renormalised residual p' = norm(max(0, p' - q)) is
//     max(0, p - a_j q) / N_j with a_0 = 0, N_0 = 1, a_{j+1} = a_j + N_j and
//     N_{j+1} = sum_v max(0, p_v - a_{j+1} q_v) (induction on j: max(0, max(0, p - a q) / N - q)
//     = max(0, p - (a + N) q) / N).  So a rejection costs one pass over the node's target and draft
//     rows, which sums the weights in 8 ranges per vocabulary chunk; the pass after the last
//     rejection also serves the draw: the crossing range among the range sums, then a scan of it.
// A request's walk runs on a cluster of 7 CTAs: every CTA takes the same decisions (same records,
// same logits, same Philox uniforms), and each pass is split across them by vocabulary chunk, each
// CTA streaming its chunks of the two rows through a 2-stage ring of 1-D bulk copies
// (cp.async.bulk) and summing them with 16-byte shared-memory loads and packed f32x2 arithmetic;
// the range sums meet in the workspace behind cluster barriers, and every CTA adds them up in the
// same order.
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
constexpr int kWalkThreads = 256;
constexpr int kWalkWarps = kWalkThreads / 32;
constexpr int kWalkStages = 2;  // ring of (target chunk, draft chunk) pairs
// CTAs per request (a thread-block cluster).  Seven lets a GPC of 19 SMs x 3 CTAs hold 8 clusters,
// so 64 requests walk in one wave (measured: 76.9 us per step against 82.5 with 8 and 85.9 with 6).
constexpr int kCluster = 7;
static_assert(kWalkWarps == kDrawRanges, "one draw range of a chunk per warp");

__device__ __forceinline__ float kscale_of(float T) { return __fdiv_rn(kLog2eF, T); }

template <int DT>
__device__ __forceinline__ const char* node_row(const void* base, int64_t row, int64_t stride) {
  constexpr int kElt = DT == SV_BF16 ? 2 : 4;
  return reinterpret_cast<const char*>(base) + row * stride * kElt;
}

// A range [c0, c0 + len) of a row as a head of plain loads, a 16-byte aligned interior of nvec
// vectors (the part a bulk copy can move) and a tail.
struct Split {
  int head, nvec, tail;
};
template <int kElt>
__device__ __forceinline__ Split split_range(const char* row, int c0, int len) {
  const uintptr_t s = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(c0) * kElt;
  const uintptr_t e = s + static_cast<uintptr_t>(len) * kElt;
  const uintptr_t a = (s + 15u) & ~uintptr_t(15), z = e & ~uintptr_t(15);
  if (z <= a) return Split{len, 0, 0};
  return Split{static_cast<int>((a - s) / kElt), static_cast<int>((z - a) / 16), static_cast<int>((e - z) / kElt)};
}

// Element e (chunk-relative) of a staged chunk: from the stage inside the copied interior, else
// from the row.
template <int DT>
__device__ __forceinline__ float staged(const unsigned char* sb, const char* row, int c0, int e, const Split& sp) {
  constexpr int kVec = DT == SV_BF16 ? 8 : 4;
  if (e >= sp.head && e < sp.head + sp.nvec * kVec) {
    if constexpr (DT == SV_BF16)
      return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(sb)[e - sp.head]) << 16);
    else
      return reinterpret_cast<const float*>(sb)[e - sp.head];
  }
  return load_logit<DT>(row, c0 + e);
}

__device__ __forceinline__ void range_of(int len, int r, int* lo, int* hi) {
  const int seg = (len + kDrawRanges - 1) / kDrawRanges;
  *lo = min(len, r * seg);
  *hi = min(len, *lo + seg);
}

__device__ __forceinline__ ChunkRecord ld_rec(const ChunkRecord* r) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(r));
  return ChunkRecord{v.x, v.y, __float_as_int(v.z), v.w};
}

__device__ __forceinline__ void two_sum_add(float& hi, float& lo, float x) {
  const float s = __fadd_rn(hi, x);
  const float bb = __fsub_rn(s, hi);
  lo = __fadd_rn(lo, __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(x, bb)));
  hi = s;
}

// Row statistics from a row's chunk records, by one warp: max and (sampled) the sum of
// 2^(x k - c(max)), or (greedy) the first argmax.
__device__ void merge_row(const ChunkRecord* rr, int NC, bool sampled, float kscale, float* m_out, float* s_out,
                          int* g_out) {
  const int lane = threadIdx.x & 31;
  // the first 64 records stay in registers (one round trip); longer rows read the rest twice
  const ChunkRecord none{-INFINITY, 0.0f, -1, NAN};
  const ChunkRecord r0 = lane < NC ? ld_rec(rr + lane) : none;
  const ChunkRecord r1 = lane + 32 < NC ? ld_rec(rr + lane + 32) : none;
  float m = -INFINITY;
  int g = -1;
  if (sampled) {
    m = fmaxf(r0.m, r1.m);
  } else {
    merge_argmax(m, g, r0.m, r0.g);
    merge_argmax(m, g, r1.m, r1.g);
  }
  for (int c = lane + 64; c < NC; c += 32) {
    const ChunkRecord rc = ld_rec(rr + c);
    if (sampled) m = fmaxf(m, rc.m);
    else merge_argmax(m, g, rc.m, rc.g);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    if (sampled) {
      m = fmaxf(m, m2);
    } else {
      const int g2 = __shfl_xor_sync(0xFFFFFFFFu, g, o);
      merge_argmax(m, g, m2, g2);
    }
  }
  float S = 0.0f;
  if (sampled && m != -INFINITY) {
    const float C = exp_offset(m, kscale);
    float hi = 0.0f, lo = 0.0f;
    if (r0.m != -INFINITY) two_sum_add(hi, lo, r0.s * pow2_nonpos(exp_offset(r0.m, kscale) - C));
    if (r1.m != -INFINITY) two_sum_add(hi, lo, r1.s * pow2_nonpos(exp_offset(r1.m, kscale) - C));
    for (int c = lane + 64; c < NC; c += 32) {
      const ChunkRecord rc = ld_rec(rr + c);
      if (rc.m != -INFINITY) two_sum_add(hi, lo, rc.s * pow2_nonpos(exp_offset(rc.m, kscale) - C));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float h2 = __shfl_xor_sync(0xFFFFFFFFu, hi, o), l2 = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
      two_sum_add(hi, lo, h2);
      lo += l2;
    }
    S = hi + lo;
  }
  *m_out = m;
  *s_out = S;
  *g_out = g;
}

// The draw weights of a node: bonus  w_v = 2^(t_v k - ct)  (p up to a factor),
//                             residual w_v = max(0, 2^(t_v k - ct) / St - a 2^(d_v k - cd) / Sd).
struct Weights {
  bool residual;
  float kscale, ct, cd, inv_st, qs;  // qs = a / Sd
};
__device__ __forceinline__ float weight(float tx, float dx, const Weights& w) {
  const float pv = ex2_approx(__fmaf_rn(tx, w.kscale, -w.ct));
  if (!w.residual) return pv;
  return fmaxf(0.0f, __fmaf_rn(pv, w.inv_st, -ex2_approx(__fmaf_rn(dx, w.kscale, -w.cd)) * w.qs));
}

// Packed float pairs beyond the streaming kernel's set: a product, and the distributed shared
// memory of a cluster (the address of a variable in another CTA of the cluster, and a 16-byte load
// from there).
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// The weights of staged vectors [v_lo, v_hi) of a chunk (16 bytes each, target in ts, draft in
// ds), lanes striding by 32, summed per lane: the same weight() per element, computed two at a
// time in packed f32x2 registers (fma, mul and add round each half like the scalar operation).
template <int DT>
__device__ __forceinline__ float weight_sum_vec(const unsigned char* ts, const unsigned char* ds, int v_lo, int v_hi,
                                                int lane, const Weights& w) {
  const f32x2 k2 = f2_pack(w.kscale, w.kscale), nct2 = f2_pack(-w.ct, -w.ct), ncd2 = f2_pack(-w.cd, -w.cd);
  const f32x2 ist2 = f2_pack(w.inv_st, w.inv_st), nqs2 = f2_pack(-w.qs, -w.qs);
  f32x2 acc[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
  auto add_pair = [&](int slot, f32x2 t2, f32x2 d2) {
    const f32x2 pt = f2_exp2_offset(t2, k2, nct2);
    if (!w.residual) {
      acc[slot] = f2_add(acc[slot], pt);
      return;
    }
    float r0, r1;
    f2_unpack(f2_fma(pt, ist2, f2_mul(f2_exp2_offset(d2, k2, ncd2), nqs2)), r0, r1);
    acc[slot] = f2_add(acc[slot], f2_pack(fmaxf(0.0f, r0), fmaxf(0.0f, r1)));
  };
  for (int v = v_lo + lane; v < v_hi; v += 32) {
    const uint4 tv = lds128(ts + static_cast<size_t>(v) * 16);
    const uint4 dv = w.residual ? lds128(ds + static_cast<size_t>(v) * 16) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t tw[4] = {tv.x, tv.y, tv.z, tv.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
    if constexpr (DT == SV_BF16) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        add_pair(e & 1, f2_pack(bf16_lo(tw[e]), bf16_hi(tw[e])), f2_pack(bf16_lo(dw[e]), bf16_hi(dw[e])));
    } else {
#pragma unroll
      for (int e = 0; e < 2; ++e)
        add_pair(e, f2_pack(__uint_as_float(tw[2 * e]), __uint_as_float(tw[2 * e + 1])),
                 f2_pack(__uint_as_float(dw[2 * e]), __uint_as_float(dw[2 * e + 1])));
    }
  }
  float a0, a1, a2, a3;
  f2_unpack(acc[0], a0, a1);
  f2_unpack(acc[1], a2, a3);
  return (a0 + a1) + (a2 + a3);
}

struct WalkSmem {
  int accept;            // the current child's test
  float Z;               // the last pass's total weight
  int y;                 // the drawn / emitted token
  int nkids;             // children of the current node
  int estar;             // pick: the crossing range
  float before;          // pick: the weight before it
  float ssub[kWalkWarps];  // pick: the crossing range's weight in sub-ranges, one per warp
  int slast[kWalkWarps];   // pick: the last entry with weight > 0 in each sub-range (-1: none)
  uint32_t flags, bad;
  int aborted;
};

template <int DT>
__global__ void __launch_bounds__(kWalkThreads) tree_walk_kernel(const VerifyParams p) {
  constexpr int kElt = DT == SV_BF16 ? 2 : 4;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;  // [kWalkStages][2][kStageBytes]
  const int Nmax = p.Kmax + 1;
  int* par = reinterpret_cast<int*>(smem + static_cast<size_t>(kWalkStages) * 2 * kStageBytes);  // [Nmax]
  int* tokn = par + Nmax;   // [Nmax]
  int* first = tokn + Nmax; // [Nmax] first child (-1 none)
  int* next = first + Nmax; // [Nmax] next sibling (-1 none)
  int* path = next + Nmax;  // [Nmax]
  int* kid = path + Nmax;   // [Nmax] children of the current node, in order
  float* kp = reinterpret_cast<float*>(kid + Nmax);  // [Nmax] p at each child's token
  float* kq = kp + Nmax;                             // [Nmax] q at each child's token
  // [2 Nmax] row statistics (max, sum, argmax) of every node row: target row of node n at n,
  // draft row at Nmax + n
  float4* rst = reinterpret_cast<float4*>(kq + Nmax);
  __shared__ __align__(8) uint64_t full_bar[kWalkStages];
  __shared__ WalkSmem ws;
  pdl_wait();  // the streaming kernel's records are complete

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blockIdx.x / kCluster;                       // request
  const int crank = static_cast<int>(cluster_rank());        // rank in its cluster
  const int NC = p.nchunks, R = 2 * p.Kmax + 1;
  int32_t* out_path = p.out_path + static_cast<int64_t>(i) * Nmax;
  int32_t* out_tok = p.out_tokens + static_cast<int64_t>(i) * Nmax;

  // ---- the request: validity, nodes, parents, tokens, child lists ----
  const int o = __ldg(p.t_off + i);
  const int N = __ldg(p.t_off + i + 1) - o;
  const float T = p.temperature ? __ldg(p.temperature + i) : 0.0f;
  uint32_t bad = 0;
  if (N < 1 || N > Nmax) bad |= SV_DEV_BAD_KEEP_LEN;
  if (!(T >= 0.0f) || isinf(T)) bad |= SV_DEV_BAD_TEMPERATURE;
  const bool sampled = T > 0.0f;
  if (!bad && (o < 0 || static_cast<int64_t>(o) + N > p.t_rows)) bad |= SV_DEV_BAD_OFFSETS;
  if (!bad && sampled && N > 1 && p.draft == nullptr) bad |= SV_DEV_NO_DRAFT_ROWS;
  if (tid == 0) {
    ws.bad = 0;
    ws.flags = 0;
    ws.aborted = 0;
    for (int s = 0; s < kWalkStages; ++s) mbar_init(&full_bar[s], 1);
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (!bad) {
    for (int c = tid; c < N; c += kWalkThreads) {
      const int pc = c == 0 ? -1 : __ldg(p.tree_parent + o + c);
      const int tc = c == 0 ? -1 : __ldg(p.tree_tokens + o + c);
      if (c > 0 && (pc < 0 || pc >= c)) atomicOr(&ws.bad, SV_DEV_BAD_PARENT);
      if (c > 0 && (tc < 0 || tc >= p.V)) atomicOr(&ws.bad, SV_DEV_BAD_TOKEN);
      par[c] = pc;
      tokn[c] = tc;
      first[c] = -1;
    }
  }
  __syncthreads();
  bad |= ws.bad;
  if (bad) {  // the same in every CTA of the cluster: the first one reports it
    if (crank == 0) {
      for (int j = tid; j < Nmax; j += kWalkThreads) {
        out_path[j] = -1;
        out_tok[j] = -1;
      }
      if (tid == 0) {
        atomicOr(p.status, bad);
        p.out_accept_len[i] = -1;
        if (p.out_flags) p.out_flags[i] = SV_FLAG_INVALID;
      }
    }
    return;
  }
  if (tid == 0) {  // children in increasing node order: insert from the last node down
    for (int c = N - 1; c >= 1; --c) {
      next[c] = first[par[c]];
      first[par[c]] = c;
    }
  }
  const float kscale = sampled ? kscale_of(T) : 0.0f;
  const int rid = p.request_ids ? __ldg(p.request_ids + i) : i;
  const ChunkRecord* recs = p.rec + static_cast<int64_t>(i) * R * NC;
  // Row statistics of every node row, merged from the chunk records up front, one row per warp
  // across the cluster (row j: target row of node j for j < N, else draft row of node j - N; a
  // sampled tree's draft rows are those of nodes 0..N-2), so no node visit waits on records.
  // Row j belongs to CTA (j / warps) mod kCluster; the others fetch it after the barrier below.
  const int nrows = sampled ? 2 * N - 1 : N;
  for (int j = crank * kWalkWarps + warp; j < nrows; j += kCluster * kWalkWarps) {
    const bool drow = j >= N;
    const int node = drow ? j - N : j;
    float m, sum;
    int g;
    merge_row(recs + static_cast<int64_t>(drow ? p.Kmax + 1 + node : node) * NC, NC, sampled, kscale, &m, &sum, &g);
    if (lane == 0) rst[(drow ? Nmax : 0) + node] = make_float4(m, sum, __int_as_float(g), 0.0f);
  }
  // range sums, double-buffered across passes: a pass writes one buffer while no CTA can still be
  // reading it (every CTA read the other pass's sums before the barrier that ended that pass)
  float* const mass0 = p.mass + static_cast<int64_t>(i) * NC * kDrawRanges;
  float* const mass1 = p.mass_p + static_cast<int64_t>(i) * NC * kDrawRanges;
  float* mass = mass0;  // the last pass's sums
  int npass = 0;
  // a wait that ran out in any CTA of the cluster (set before a cluster barrier, read after it);
  // cleared before the first barrier
  uint32_t* abort_word = reinterpret_cast<uint32_t*>(p.req + i);
  if (crank == 0 && tid == 0) *abort_word = 0;
  __syncthreads();
  cluster_sync();  // the word is clear before any CTA may set it; every CTA's rows are merged
  for (int j = tid; j < nrows; j += kWalkThreads) {  // the other CTAs' rows, from their shared memory
    const int owner = (j / kWalkWarps) % kCluster;
    if (owner == crank) continue;
    const int idx = j >= N ? Nmax + (j - N) : j;
    rst[idx] = ld_cluster_f4(cluster_addr(rst + idx, static_cast<uint32_t>(owner)));
  }
  __syncthreads();

  uint32_t it = 0;  // ring stages consumed so far (every thread keeps the same count)
  // One pass over a node's rows with weights w: the range sums (mass) and their total (ws.Z).
  auto pass = [&](const char* trow, const char* drow, const Weights& w) {
    auto issue = [&](int c, uint32_t k) {  // chunk c into ring slot k % kWalkStages (thread 0)
      const int stage = k % kWalkStages;
      unsigned char* sb = ring + static_cast<size_t>(stage) * 2 * kStageBytes;
      const int c0 = c * p.chunk_len, len = min(p.chunk_len, p.V - c0);
      const Split st = split_range<kElt>(trow, c0, len);
      const Split sd = w.residual ? split_range<kElt>(drow, c0, len) : Split{0, 0, 0};
      const uint32_t bytes = static_cast<uint32_t>(st.nvec + sd.nvec) * 16u;
      if (bytes == 0) {
        mbar_arrive(&full_bar[stage]);
        return;
      }
      mbar_arrive_expect_tx(&full_bar[stage], bytes);
      if (st.nvec) bulk_g2s(sb, trow + static_cast<int64_t>(c0 + st.head) * kElt, st.nvec * 16u, &full_bar[stage]);
      if (sd.nvec)
        bulk_g2s(sb + kStageBytes, drow + static_cast<int64_t>(c0 + sd.head) * kElt, sd.nvec * 16u, &full_bar[stage]);
    };
    mass = (npass & 1) ? mass1 : mass0;
    ++npass;
    // this CTA's chunks: crank, crank + kCluster, ...
    const int nloc = crank < NC ? (NC - 1 - crank) / kCluster + 1 : 0;
    if (tid == 0)
      for (int k = 0; k < kWalkStages && k < nloc; ++k) issue(crank + k * kCluster, it + k);
    for (int k = 0; k < nloc; ++k, ++it) {
      const int c = crank + k * kCluster;
      const int stage = it % kWalkStages;
      if (tid == 0 && !ws.aborted && !mbar_wait(&full_bar[stage], (it / kWalkStages) & 1u, p.status, p.wait_limit_ns))
        ws.aborted = 1;
      __syncthreads();
      const unsigned char* sb = ring + static_cast<size_t>(stage) * 2 * kStageBytes;
      const int c0 = c * p.chunk_len, len = min(p.chunk_len, p.V - c0);
      const Split st = split_range<kElt>(trow, c0, len);
      const Split sd = w.residual ? split_range<kElt>(drow, c0, len) : Split{0, 0, 0};
      int lo, hi;
      range_of(len, warp, &lo, &hi);
      float sum = 0.0f;
      // a chunk staged whole (both rows) with this warp's range on vector boundaries: 16-byte
      // loads and packed arithmetic; otherwise element by element
      constexpr int kVec = 16 / kElt;
      const bool whole = st.head == 0 && st.nvec * kVec == len &&
                         (!w.residual || (sd.head == 0 && sd.nvec * kVec == len)) && lo % kVec == 0 && hi % kVec == 0;
      if (whole) {
        sum = weight_sum_vec<DT>(sb, sb + kStageBytes, lo / kVec, hi / kVec, lane, w);
      } else {
        for (int e = lo + lane; e < hi; e += 32) {
          const float tx = staged<DT>(sb, trow, c0, e, st);
          const float dx = w.residual ? staged<DT>(sb + kStageBytes, drow, c0, e, sd) : 0.0f;
          sum += weight(tx, dx, w);
        }
      }
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o2);
      if (lane == 0) mass[c * kDrawRanges + warp] = sum;
      __syncthreads();  // the stage is read: it may be refilled
      if (tid == 0 && !ws.aborted && k + kWalkStages < nloc)
        issue(crank + (k + kWalkStages) * kCluster, it + kWalkStages);
    }
    if (tid == 0 && ws.aborted) atomicOr(abort_word, 1u);
    __syncthreads();
    cluster_sync();  // every CTA's range sums (and any wait that ran out) are written
    if (tid == 0) ws.aborted = __ldcg(abort_word) != 0u ? 1 : 0;  // the same in every CTA
    if (warp == 0) {  // the total, in a fixed order (the same in every CTA)
      float z = 0.0f;
      for (int e = lane; e < NC * kDrawRanges; e += 32) z += __ldcg(mass + e);
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o2);
      if (lane == 0) ws.Z = z;
    }
    __syncthreads();
  };

  // Inverse-CDF pick over the weights of the last pass (total ws.Z) with uniform u, in one CTA of
  // the cluster (rank 0; every thread of every CTA calls it): the range sums and then the crossing
  // range's weights are brought into shared memory in one round trip each (the ring is idle now),
  // and warp 0 scans them.  Sets ws.y.
  auto pick = [&](const char* trow, const char* drow, const Weights& w, float u) {
    constexpr int kMaxStagedSums = 4096;                            // 16 KB of the ring
    float* ssum = reinterpret_cast<float*>(ring);                    // [NE] range sums
    float* swt = reinterpret_cast<float*>(ring + 4 * kMaxStagedSums);  // [range] weights
    const int NE = NC * kDrawRanges;
    const bool staged_sums = NE <= kMaxStagedSums;
    const float thr = u * ws.Z;
    if (crank == 0 && staged_sums)
      for (int j = tid; j < NE; j += kWalkThreads) ssum[j] = __ldcg(mass + j);
    __syncthreads();
    if (warp == 0 && crank == 0) {
      // first range whose running sum exceeds thr (or the last with weight > 0)
      float before = 0.0f, run = 0.0f, before_last = 0.0f;
      int estar = -1, last_pos = -1;
      for (int j0 = 0; j0 < NE && estar < 0; j0 += 32) {
        const int j = j0 + lane;
        const float wj = j < NE ? (staged_sums ? ssum[j] : __ldcg(mass + j)) : 0.0f;
        float incl = wj;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
          const float yv = __shfl_up_sync(0xFFFFFFFFu, incl, o2);
          if (lane >= o2) incl += yv;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, j < NE && wj > 0.0f && run + incl > thr);
        const unsigned pos = __ballot_sync(0xFFFFFFFFu, j < NE && wj > 0.0f);
        if (hit) {
          const int src = __ffs(hit) - 1;
          estar = j0 + src;
          before = run + __shfl_sync(0xFFFFFFFFu, incl - wj, src);
        } else if (pos) {
          const int src = 31 - __clz(pos);
          last_pos = j0 + src;
          before_last = run + __shfl_sync(0xFFFFFFFFu, incl - wj, src);
        }
        run += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (estar < 0) {
        estar = last_pos >= 0 ? last_pos : 0;
        before = before_last;
      }
      if (lane == 0) {
        ws.estar = estar;
        ws.before = before;
      }
    }
    __syncthreads();
    // the crossing range's weights, every load issued at once
    const int estar = ws.estar, c = estar / kDrawRanges, r = estar - c * kDrawRanges;
    const int c0 = c * p.chunk_len, len = min(p.chunk_len, p.V - c0);
    int lo, hi;
    range_of(len, r, &lo, &hi);
    if (crank == 0)
      for (int e = lo + tid; e < hi; e += kWalkThreads)
        swt[e - lo] = weight(load_logit<DT>(trow, c0 + e), w.residual ? load_logit<DT>(drow, c0 + e) : 0.0f, w);
    __syncthreads();
    // The range in one sub-range per warp: each warp sums its own; warp 0 then finds the sub-range
    // where the running sum passes thr and scans only that one.
    const int n = hi - lo, sub = (n + kWalkWarps - 1) / kWalkWarps;
    if (crank == 0) {
      const int s_lo = min(n, warp * sub), s_hi = min(n, s_lo + sub);
      float acc = 0.0f;
      int lastp = -1;
      for (int e = s_lo + lane; e < s_hi; e += 32) {
        const float wv = swt[e];
        acc += wv;
        if (wv > 0.0f) lastp = e;
      }
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) {
        acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o2);
        lastp = max(lastp, __shfl_xor_sync(0xFFFFFFFFu, lastp, o2));
      }
      if (lane == 0) {
        ws.ssub[warp] = acc;
        ws.slast[warp] = lastp;
      }
    }
    __syncthreads();
    if (warp == 0 && crank == 0) {  // the entry inside the range
      const float sv = lane < kWalkWarps ? ws.ssub[lane] : 0.0f;
      float incl = sv;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const float yv = __shfl_up_sync(0xFFFFFFFFu, incl, o2);
        if (lane >= o2) incl += yv;
      }
      const float excl_up = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
      const float excl = lane == 0 ? 0.0f : excl_up;
      const unsigned cross = __ballot_sync(0xFFFFFFFFu, lane < kWalkWarps && sv > 0.0f && ws.before + incl > thr);
      int y = -1;
      if (cross) {
        const int sidx = __ffs(cross) - 1;
        float run2 = ws.before + __shfl_sync(0xFFFFFFFFu, excl, sidx);
        const int s_lo = min(n, sidx * sub), s_hi = min(n, s_lo + sub);
        for (int e0 = s_lo; e0 < s_hi && y < 0; e0 += 32) {
          const int e = e0 + lane;
          const float wv = e < s_hi ? swt[e] : 0.0f;
          float run = wv;
#pragma unroll
          for (int o2 = 1; o2 < 32; o2 <<= 1) {
            const float yv = __shfl_up_sync(0xFFFFFFFFu, run, o2);
            if (lane >= o2) run += yv;
          }
          const unsigned hit = __ballot_sync(0xFFFFFFFFu, e < s_hi && wv > 0.0f && run2 + run > thr);
          if (hit) y = c0 + lo + e0 + __ffs(hit) - 1;
          run2 += __shfl_sync(0xFFFFFFFFu, run, 31);
        }
        if (y < 0) y = c0 + lo + ws.slast[sidx];  // rounding: the sum passed thr at the sub-range's end
      } else {  // rounding: the range ends at or below thr; its last entry with weight > 0
        int lp = lane < kWalkWarps ? ws.slast[lane] : -1;
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) lp = max(lp, __shfl_xor_sync(0xFFFFFFFFu, lp, o2));
        y = c0 + lo + (lp >= 0 ? lp : 0);
      }
      if (lane == 0) ws.y = y;
    }
    __syncthreads();
  };

  // ---- the walk ----
  int node = 0, L = 0;
  for (int step = 0; step < N; ++step) {
    const bool kids = first[node] >= 0;
    const float4 tstat = rst[node];                                            // target row
    const float4 dstat = sampled && kids ? rst[Nmax + node] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);  // draft row
    if (!sampled) {  // greedy: the first child holding the target argmax
      const int g = __float_as_int(tstat.z);
      int acc = -1;
      for (int c = first[node]; c >= 0; c = next[c])
        if (tokn[c] == g) {
          acc = c;
          break;
        }
      if (acc < 0) {
        if (tid == 0) ws.y = g;
        break;
      }
      if (tid == 0) path[L] = acc;
      ++L;
      node = acc;
      __syncthreads();
      continue;
    }
    const char* trow = node_row<DT>(p.target, static_cast<int64_t>(o) + node, p.t_row_stride);
    const char* drow = kids ? node_row<DT>(p.draft, static_cast<int64_t>(o) + node, p.d_row_stride) : trow;
    Weights w;
    w.kscale = kscale;
    w.ct = exp_offset(tstat.x, kscale);
    w.inv_st = __frcp_rn(tstat.y);
    w.cd = kids ? exp_offset(dstat.x, kscale) : 0.0f;
    const float inv_sd = kids ? __frcp_rn(dstat.y) : 0.0f;
    const float u_draw = philox_uniform_f(p.seed, static_cast<uint32_t>(node), static_cast<uint32_t>(rid), 1u, p.round);
    if (!kids) {  // a leaf: y ~ p
      w.residual = false;
      w.qs = 0.0f;
      pass(trow, trow, w);
      if (ws.aborted) break;
      pick(trow, trow, w, u_draw);
      break;
    }
    // p and q at every child's token, all loaded at once
    if (tid == 0) {
      int nk = 0;
      for (int c = first[node]; c >= 0; c = next[c]) kid[nk++] = c;
      ws.nkids = nk;
    }
    __syncthreads();
    const int nk = ws.nkids;
    for (int j = tid; j < nk; j += kWalkThreads) {
      const int x = tokn[kid[j]];
      const float tx = load_logit<DT>(trow, x), dx = load_logit<DT>(drow, x);
      kp[j] = __fmul_rn(ex2_approx(__fmaf_rn(tx, kscale, -w.ct)), w.inv_st);
      kq[j] = __fmul_rn(ex2_approx(__fmaf_rn(dx, kscale, -w.cd)), inv_sd);
    }
    __syncthreads();
    // the children in order; after each rejection the residual's normaliser (one pass)
    float a = 0.0f, Nr = 1.0f, a_pass = -1.0f;  // a_pass: the a of the weights the last pass summed
    int acc = -1;
    for (int j = 0; j < nk; ++j) {
      const int c = kid[j];
      if (tid == 0) {
        const float pv = kp[j], qv = kq[j];
        const float prv = __fdiv_rn(fmaxf(0.0f, __fmaf_rn(-a, qv, pv)), Nr);
        const float u = philox_uniform_f(p.seed, static_cast<uint32_t>(c - 1), static_cast<uint32_t>(rid), 0u, p.round);
        if (qv == 0.0f) ws.flags |= SV_FLAG_Q_ZERO;
        ws.accept = u * qv < prv ? 1 : 0;
      }
      __syncthreads();
      if (ws.accept) {
        acc = c;
        break;
      }
      const float a_next = a + Nr;
      w.residual = true;
      w.qs = __fmul_rn(a_next, inv_sd);
      pass(trow, drow, w);
      if (ws.aborted) break;
      if (ws.Z > 0.0f) {
        a = a_next;
        Nr = ws.Z;
        a_pass = a;
      } else {  // residual mass 0 (not reachable in exact arithmetic): p' stays
        if (tid == 0) ws.flags |= SV_FLAG_Z_ZERO;
        a_pass = -1.0f;
      }
      __syncthreads();
    }
    if (ws.aborted) break;
    if (acc >= 0) {
      if (tid == 0) path[L] = acc;
      ++L;
      node = acc;
      __syncthreads();
      continue;
    }
    // every child rejected: y ~ max(0, p - a q), from the last pass's range sums when they are of a
    w.residual = a > 0.0f;
    w.qs = __fmul_rn(a, inv_sd);
    if (a_pass != a) {
      pass(trow, drow, w);
      if (ws.aborted) break;
    }
    pick(trow, drow, w, u_draw);
    break;
  }
  __syncthreads();
  cluster_sync();          // no CTA leaves while another may still read its row statistics
  if (crank != 0) return;  // one CTA of the cluster writes the outputs
  // ---- outputs ----
  for (int j = tid; j < Nmax; j += kWalkThreads) {
    int pj = -1, tj = -1;
    if (j < L) {
      pj = path[j];
      tj = tokn[pj];
    } else if (j == L) {
      tj = ws.aborted ? -1 : ws.y;
    }
    out_path[j] = pj;
    out_tok[j] = tj;
  }
  if (tid == 0) {
    p.out_accept_len[i] = L;
    if (p.out_flags) p.out_flags[i] = static_cast<uint8_t>(ws.flags);
  }
}

size_t walk_smem_bytes(int Nmax) {  // the ring, six int and two float arrays of Nmax, 2 Nmax float4
  return static_cast<size_t>(kWalkStages) * 2 * kStageBytes + (8 * sizeof(int) + 2 * sizeof(float4)) * static_cast<size_t>(Nmax);
}

std::mutex g_tree_mu;
bool g_tree_ready[64][2] = {};

template <int DT>
cudaError_t launch_walk_t(const VerifyParams& p, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(g_tree_mu);
    if (!g_tree_ready[dev][DT == SV_BF16 ? 0 : 1]) {
      if ((e = cudaFuncSetAttribute(tree_walk_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(walk_smem_bytes(SV_MAX_DRAFT + 1)))) != cudaSuccess)
        return e;
      g_tree_ready[dev][DT == SV_BF16 ? 0 : 1] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.B * kCluster, 1, 1);
  cfg.blockDim = dim3(kWalkThreads, 1, 1);
  cfg.dynamicSmemBytes = walk_smem_bytes(p.Kmax + 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = prof_enabled() ? 1 : 2;
  prof_before(SV_KERNEL_TREE_WALK, stream);
  e = cudaLaunchKernelEx(&cfg, tree_walk_kernel<DT>, p);
  prof_after(SV_KERNEL_TREE_WALK, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int launch_tree(const VerifyParams& p, sv_dtype dt, void* stream) {
  const int e = launch_stats(p, dt, stream);
  if (e != 0) return e;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return static_cast<int>(dt == SV_BF16 ? launch_walk_t<SV_BF16>(p, s) : launch_walk_t<SV_F32>(p, s));
}

}  // namespace sv
