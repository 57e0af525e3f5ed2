// Internal declarations shared by libsv's translation units (host and device).
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/sv.h"

namespace sv {

// ---- row_stats kernel geometry ---------------------------------------------------------------
constexpr int kStageBytes = 16384;     // one vocabulary chunk per pipeline stage
// Bulk-copy ring depth and resident CTAs per SM of the streaming kernel, per logit type: fp32
// chunks (4096 logits) leave the consumers idle between copies, so 3 CTAs of 4 stages keep HBM
// busy; bf16 chunks (8192 logits) are bound by instruction issue, so 4 CTAs of 3 stages (the same
// bytes in flight per SM) add warps.
template <int DT>
struct StreamShape {
  static constexpr int kStages = DT == SV_BF16 ? 3 : 4;
  static constexpr int kCtasPerSm = DT == SV_BF16 ? 4 : 3;
};
constexpr int kConsumerWarps = 4;      // warps that reduce a chunk (8 vectors per thread: the
                                       // per-chunk bookkeeping is spread over 64 logits)
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kStatsThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kVecPerThread = kStageBytes / 16 / kConsumerThreads;  // 16-byte vectors per thread
static_assert(kVecPerThread * 16 * kConsumerThreads == kStageBytes, "stage split");


// Each vocabulary chunk's draw weights are summed in kDrawRanges contiguous ranges (one per
// warp); a pick finds the crossing range and scans only that range.
constexpr int kDrawRanges = 8;

// Per-(row, chunk) statistics written by row_stats.
struct alignas(16) ChunkRecord {
  float m;     // max logit in the chunk
  float s;     // sum of 2^(x k - rint(m k)) over the chunk, k = log2(e) / T (0 for greedy rows)
  int32_t g;   // first argmax in the chunk (vocabulary index), greedy rows only
  float xval;  // logit at the row's drafted token, when that token lies in the chunk
};

// What the draw at the accepted length needs (written by the combine kernel, read by the mass and
// pick kernels).
enum : int32_t { kModeNone = 0, kModeBonus = 1, kModeResidual = 2 };
struct alignas(16) ReqState {
  int32_t mode;
  int32_t a;          // accepted length == position of the draw
  int64_t row_t;      // absolute target row index of row a
  int64_t row_d;      // absolute draft row index of row a (residual mode)
  float kscale;       // log2(e) / T, rounded to float
  float ct, cd;       // exponent offsets exp_offset(row max, kscale) of the two rows
  float inv_st, inv_sd;  // 1 / row sums (float)
  float st;           // target row a's sum
  float u;            // u' for the draw
  int32_t flags;
};

struct VerifyParams {
  const void* target;
  int64_t t_row_stride;     // elements
  const int32_t* t_off;     // [B+1] or null => i * (Kmax + 1)
  const void* draft;
  int64_t d_row_stride;
  const int32_t* d_off;     // [B+1] or null => i * Kmax
  const int32_t* tokens;    // [B, tok_stride] or null => draft argmax (greedy only)
  int32_t tok_stride;
  const int32_t* keep_len;  // [B] or null => Kmax
  const float* temperature; // [B] or null => greedy
  const int32_t* request_ids;
  int64_t t_rows, d_rows;   // rows the packed arrays hold (ragged calls; < 0 = not checked)
  uint64_t seed;
  uint32_t round;
  int32_t B, Kmax, V;
  int32_t chunk_len, nchunks;  // vocabulary tiling
  int32_t rows_per_req;        // 2 * Kmax + 1 record rows per request
  // outputs
  int32_t* out_tokens;      // [B, Kmax+1]
  int32_t* out_accept_len;  // [B]
  float* out_p;             // [B, Kmax] nullable
  float* out_q;
  uint8_t* out_flags;       // [B] nullable
  // workspace
  uint32_t* status;
  ReqState* req;            // [B] draw state per request
  ChunkRecord* rec;         // [B * rows_per_req * nchunks]
  float* mass;              // [B * nchunks * 8] residual mass per draw range (8 per chunk)
  float* mass_p;            // [B * nchunks * 8] target-row weight per draw range (bonus / fallback)
  // tree verification: the stream runs on every node row (n_i = N_i - 1 from t_off, no tokens)
  int32_t tree;
  const int32_t* tree_parent;  // [sum N_i] parent node per node
  const int32_t* tree_tokens;  // [sum N_i] drafted token per node
  int32_t* out_path;           // [B, Kmax + 1] accepted nodes
  // vocabulary shard (a range of chunks; the whole row by default): the stream and the draw read
  // chunks [c_begin, c_end), whose columns start at v_begin in the logit arrays given
  int32_t c_begin, c_end;
  int64_t v_begin;
  uint64_t wait_limit_ns;   // bound of every wait in the stream kernel
  int32_t stall_cta;        // test hook: > 0 makes CTA stall_cta - 1 of the stream issue no copy
  int32_t uniform_rows;     // > 0: every request has this many record rows (no per-request plan)
  int32_t fuse_draw;        // 1: the combine kernel's CTAs also sum the draw weights per chunk
};

// Largest B * Dmax ranked by merging the per-request runs (two key buffers in shared memory);
// larger batches use the bitonic sort, which is faster there on one CTA.
constexpr int kMergeMaxSlots = 2048;

struct ScheduleParams {
  const float* alpha;
  int32_t alpha_stride;
  const int32_t* draft_len;
  int32_t B, Dmax;
  double cost_a, cost_b;
  // n_cost == 0: c(K) = cost_a + cost_b * K; else the latency table (cost_K, cost_c) with
  // the slope cost_s[j] of segment j (j <= n_cost - 2), computed on the host
  int32_t n_cost;
  int32_t cost_K[SV_MAX_COST_KNOTS];
  double cost_c[SV_MAX_COST_KNOTS];
  double cost_s[SV_MAX_COST_KNOTS];
  int32_t budget;
  int32_t n_ratios;
  float ratios[8];
  int32_t objective;
  int32_t sort_size;  // bitonic mode: power of two >= B * Dmax, at least 1024
  int32_t merge;      // 1: merge the per-request runs (B * Dmax <= kMergeMaxSlots), 0: bitonic sort
  int32_t* out_keep_len;
  int32_t* out_row_offsets;
  int32_t* out_total_K;
  int64_t* out_utility_q48;
  uint32_t* status;
};

// Workspace layout for SV_OP_VERIFY.
struct VerifyLayout {
  size_t status, req, rec, mass, mass_p, total;
};
VerifyLayout verify_layout(int B, int Kmax, int nchunks);
void vocab_tiling(int V, sv_dtype dt, int* chunk_len, int* nchunks);

// Launchers (return cudaError_t as int to keep CUDA headers out of this file).
int launch_verify(const VerifyParams& p, sv_dtype dt, bool sampled, void* stream);
// One step of a sampled verification over a vocabulary shard (SV_PHASE_*).
int launch_phase(const VerifyParams& p, sv_dtype dt, int phase, void* stream);
// The streaming kernel alone (its records feed the tree walk).
int launch_stats(const VerifyParams& p, sv_dtype dt, void* stream);
// Tree verification: the streaming kernel, then the walk kernel behind it.
int launch_tree(const VerifyParams& p, sv_dtype dt, void* stream);
int launch_schedule(const ScheduleParams& p, void* stream);

// Host-side argument checks of sv_verify_sample (sv_api.cu); touch no GPU.
sv_status validate_sample(const void* target, int64_t t_row_stride, const void* draft, int64_t d_row_stride,
                          const int32_t* draft_tokens, const float* temperature, sv_dtype dt, int B, int K, int V,
                          const int32_t* out_tokens, const int32_t* out_accept_len);

// Records the message returned by sv_last_error_string and returns s (sv_api.cu).
sv_status set_error(sv_status s, const char* fmt, ...);

// Instrumentation hooks implemented in sv_api.cu.
bool prof_enabled();
void prof_before(int kernel_id, void* stream);
void prof_after(int kernel_id, void* stream);

}  // namespace sv
