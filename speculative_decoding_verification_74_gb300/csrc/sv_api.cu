// C ABI of libsv: argument checks, workspace layout, launches, status and instrumentation.
// Every check here runs on the host before any CUDA call, so an invalid call touches no GPU.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "sv_internal.h"

namespace {

thread_local char g_err[512] = "";

sv_status fail(sv_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

sv_status cuda_fail(int e, const char* what) {
  return fail(SV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(static_cast<cudaError_t>(e)));
}

int elt_size(sv_dtype dt) { return dt == SV_BF16 ? 2 : 4; }

sv_status check_rows(const char* name, const void* base, int64_t stride, int V, sv_dtype dt) {
  if ((reinterpret_cast<uintptr_t>(base) % elt_size(dt)) != 0)
    return fail(SV_ERR_INVALID_ARG, "%s is not aligned to its element size", name);
  if (stride < V) return fail(SV_ERR_INVALID_ARG, "%s row stride %lld < V %d", name, (long long)stride, V);
  return SV_OK;
}

sv_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr) return fail(SV_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(SV_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if (ws_bytes < need) return fail(SV_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return SV_OK;
}

// ---- instrumentation ------------------------------------------------------------------------
struct ProfRec {
  int id;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;
cudaEvent_t g_pending_start[SV_NUM_KERNELS];
std::atomic<int64_t> g_launches{0};

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Test hook (sv_test_stall_next_verify): wait limit in ms for the next verification call, 0 = none.
std::atomic<int> g_stall_ms{0};

// ---- shared verify entry ----------------------------------------------------------------------
sv_status verify_common(sv::VerifyParams& p, sv_dtype dt, bool sampled, void* ws, size_t ws_bytes,
                        void* stream, int phase = -1) {
  if (p.B == 0) return SV_OK;  // nothing to verify: no workspace needed, nothing enqueued
  int cl, nc;
  sv::vocab_tiling(p.V, dt, &cl, &nc);
  const sv::VerifyLayout L = sv::verify_layout(p.B, p.Kmax, nc);
  sv_status s = check_ws(ws, ws_bytes, L.total);
  if (s != SV_OK) return s;
  unsigned char* w = static_cast<unsigned char*>(ws);
  p.chunk_len = cl;
  p.nchunks = nc;
  if (phase < 0) {  // a whole call: every chunk of every row
    p.c_begin = 0;
    p.c_end = nc;
    p.v_begin = 0;
  } else {
    if (p.c_begin < 0 || p.c_end > nc || p.c_begin >= p.c_end)
      return fail(SV_ERR_INVALID_ARG, "chunk range [%d, %d) outside [0, %d)", p.c_begin, p.c_end, nc);
    p.v_begin = static_cast<int64_t>(p.c_begin) * cl;
  }
  p.rows_per_req = 2 * p.Kmax + 1;
  // Greedy fixed-K calls need no per-request plan: every request has the same rows.  Sampling
  // calls take the per-request plan, which leaves out the draft rows of T == 0 requests.
  if (p.keep_len == nullptr && p.t_off == nullptr && p.d_off == nullptr && p.temperature == nullptr)
    p.uniform_rows = p.tokens == nullptr ? 2 * p.Kmax + 1 : p.Kmax + 1;
  p.status = reinterpret_cast<uint32_t*>(w + L.status);
  const int stall_ms = g_stall_ms.exchange(0);
  p.wait_limit_ns = stall_ms > 0 ? static_cast<uint64_t>(stall_ms) * 1000000ull : 2000000000ull;
  p.stall_cta = stall_ms > 0 ? 1 : 0;
  p.req = reinterpret_cast<sv::ReqState*>(w + L.req);
  p.rec = reinterpret_cast<sv::ChunkRecord*>(w + L.rec);
  p.mass = reinterpret_cast<float*>(w + L.mass);
  p.mass_p = reinterpret_cast<float*>(w + L.mass_p);
  const int e = phase >= 0 ? sv::launch_phase(p, dt, phase, stream)
                 : p.tree ? sv::launch_tree(p, dt, stream) : sv::launch_verify(p, dt, sampled, stream);
  if (e != 0) return cuda_fail(e, "verify launch");
  return SV_OK;
}

sv_status check_common(const void* target, int64_t t_row_stride, const void* draft, int64_t d_row_stride,
                       sv_dtype dt, int B, int K, int V, const int32_t* out_tokens, const int32_t* out_accept_len) {
  if (dt != SV_BF16 && dt != SV_F32) return fail(SV_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (B < 0 || B > SV_MAX_BATCH) return fail(SV_ERR_INVALID_ARG, "B=%d outside [0, %d]", B, SV_MAX_BATCH);
  if (K < 0 || K > SV_MAX_DRAFT) return fail(SV_ERR_INVALID_ARG, "K=%d outside [0, %d]", K, SV_MAX_DRAFT);
  if (V < 1 || V > (1 << 30)) return fail(SV_ERR_INVALID_ARG, "V=%d outside [1, 2^30]", V);
  if (B == 0) return SV_OK;
  if (target == nullptr) return fail(SV_ERR_INVALID_ARG, "target is NULL");
  sv_status s = check_rows("target", target, t_row_stride, V, dt);
  if (s != SV_OK) return s;
  if (draft != nullptr && (s = check_rows("draft", draft, d_row_stride, V, dt)) != SV_OK) return s;
  if (out_tokens == nullptr || out_accept_len == nullptr)
    return fail(SV_ERR_INVALID_ARG, "out_tokens / out_accept_len is NULL");
  return SV_OK;
}

}  // namespace

// =============================================================================================
// sv:: hooks used by the kernels' launchers
// =============================================================================================
namespace {
// Inside a stream capture the bracket must become an event-record node of the graph (external
// record) so that every replay re-records it and its elapsed time can be read.
void record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}
}  // namespace

namespace sv {
sv_status validate_sample(const void* target, int64_t t_row_stride, const void* draft, int64_t d_row_stride,
                          const int32_t* draft_tokens, const float* temperature, sv_dtype dt, int B, int K, int V,
                          const int32_t* out_tokens, const int32_t* out_accept_len) {
  sv_status s = check_common(target, t_row_stride, draft, d_row_stride, dt, B, K, V, out_tokens, out_accept_len);
  if (s != SV_OK) return s;
  if (B > 0 && (temperature == nullptr || (K > 0 && draft_tokens == nullptr)))
    return fail(SV_ERR_INVALID_ARG, "sampled verification needs temperature and draft_tokens");
  return SV_OK;
}
sv_status set_error(sv_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}
bool prof_enabled() { return g_prof_on; }
void prof_before(int id, void* stream) {
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t a = take_event();
  record(a, static_cast<cudaStream_t>(stream));
  g_pending_start[id] = a;
}
void prof_after(int id, void* stream) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t b = take_event();
  record(b, static_cast<cudaStream_t>(stream));
  g_prof.push_back({id, g_pending_start[id], b});
}
}  // namespace sv

// =============================================================================================
// C ABI
// =============================================================================================
extern "C" {

int sv_abi_version(void) { return 2; }

void sv_test_stall_next_verify(int wait_limit_ms) { g_stall_ms.store(wait_limit_ms > 0 ? wait_limit_ms : 0); }

size_t sv_workspace_size(int op, int B, int Kmax, int V, sv_dtype dt) {
  if (op == SV_OP_SCHEDULE) return 256;
  if (op == SV_OP_TREE) {  // Kmax is Nmax here: a tree of N nodes has the rows of a chain of N - 1
    if (Kmax < 1) return 0;
    --Kmax;
  } else if (op != SV_OP_VERIFY) {
    return 0;
  }
  if (B < 0 || B > SV_MAX_BATCH || Kmax < 0 || Kmax > SV_MAX_DRAFT || V < 1 || V > (1 << 30)) return 0;
  if (dt != SV_BF16 && dt != SV_F32) return 0;
  int cl, nc;
  sv::vocab_tiling(V, dt, &cl, &nc);
  return sv::verify_layout(B, Kmax, nc).total;
}

sv_status sv_verify_greedy(const void* target, int64_t t_row_stride, const void* draft, int64_t d_row_stride,
                           const int32_t* draft_tokens, sv_dtype dt, int B, int K, int V, int32_t* out_tokens,
                           int32_t* out_accept_len, void* ws, size_t ws_bytes, void* stream) {
  sv_status s = check_common(target, t_row_stride, draft, d_row_stride, dt, B, K, V, out_tokens, out_accept_len);
  if (s != SV_OK) return s;
  if (B > 0 && K > 0 && draft == nullptr && draft_tokens == nullptr)
    return fail(SV_ERR_INVALID_ARG, "greedy verification needs draft logits or draft tokens");
  sv::VerifyParams p = {};
  p.target = target;
  p.t_row_stride = t_row_stride;
  p.draft = draft_tokens ? nullptr : draft;  // with tokens given the draft rows are never read
  p.d_row_stride = d_row_stride;
  p.tokens = draft_tokens;
  p.tok_stride = K;
  p.B = B;
  p.Kmax = K;
  p.V = V;
  p.t_rows = p.d_rows = -1;
  p.out_tokens = out_tokens;
  p.out_accept_len = out_accept_len;
  return verify_common(p, dt, false, ws, ws_bytes, stream);
}

static sv::VerifyParams sample_params(const void* target, int64_t t_row_stride, const void* draft,
                                      int64_t d_row_stride, const int32_t* draft_tokens, const float* temperature,
                                      uint64_t seed, uint32_t round, const int32_t* request_ids, int B, int K, int V,
                                      int32_t* out_tokens, int32_t* out_accept_len, float* out_p, float* out_q,
                                      uint8_t* out_flags) {
  sv::VerifyParams p = {};
  p.target = target;
  p.t_row_stride = t_row_stride;
  p.draft = draft;
  p.d_row_stride = d_row_stride;
  p.tokens = draft_tokens;
  p.tok_stride = K;
  p.temperature = temperature;
  p.request_ids = request_ids;
  p.seed = seed;
  p.round = round;
  p.B = B;
  p.Kmax = K;
  p.V = V;
  p.out_tokens = out_tokens;
  p.out_accept_len = out_accept_len;
  p.out_p = out_p;
  p.out_q = out_q;
  p.out_flags = out_flags;
  p.t_rows = p.d_rows = -1;
  return p;
}

sv_status sv_verify_sample(const void* target, int64_t t_row_stride, const void* draft, int64_t d_row_stride,
                           const int32_t* draft_tokens, const float* temperature, uint64_t seed, uint32_t round,
                           const int32_t* request_ids, sv_dtype dt, int B, int K, int V, int32_t* out_tokens,
                           int32_t* out_accept_len, float* out_p, float* out_q, uint8_t* out_flags, void* ws,
                           size_t ws_bytes, void* stream) {
  sv_status s = sv::validate_sample(target, t_row_stride, draft, d_row_stride, draft_tokens, temperature, dt, B, K,
                                    V, out_tokens, out_accept_len);
  if (s != SV_OK) return s;
  sv::VerifyParams p = sample_params(target, t_row_stride, draft, d_row_stride, draft_tokens, temperature, seed, round,
                                     request_ids, B, K, V, out_tokens, out_accept_len, out_p, out_q, out_flags);
  return verify_common(p, dt, true, ws, ws_bytes, stream);
}

sv_status sv_vocab_chunks(int V, sv_dtype dt, int* chunk_len, int* nchunks) {
  if (V < 1 || V > (1 << 30) || (dt != SV_BF16 && dt != SV_F32) || chunk_len == nullptr || nchunks == nullptr)
    return fail(SV_ERR_INVALID_ARG, "sv_vocab_chunks: V=%d dt=%d", V, (int)dt);
  sv::vocab_tiling(V, dt, chunk_len, nchunks);
  return SV_OK;
}

sv_status sv_verify_regions(int B, int K, int V, sv_dtype dt, size_t* rec_offset, size_t* rec_bytes,
                            size_t* mass_offset, size_t* mass_p_offset, size_t* mass_bytes) {
  if (B < 1 || B > SV_MAX_BATCH || K < 0 || K > SV_MAX_DRAFT || V < 1 || V > (1 << 30) ||
      (dt != SV_BF16 && dt != SV_F32))
    return fail(SV_ERR_INVALID_ARG, "sv_verify_regions: B=%d K=%d V=%d dt=%d", B, K, V, (int)dt);
  int cl, nc;
  sv::vocab_tiling(V, dt, &cl, &nc);
  const sv::VerifyLayout L = sv::verify_layout(B, K, nc);
  if (rec_offset) *rec_offset = L.rec;
  if (rec_bytes) *rec_bytes = sizeof(sv::ChunkRecord) * static_cast<size_t>(B) * (2 * static_cast<size_t>(K) + 1) * nc;
  if (mass_offset) *mass_offset = L.mass;
  if (mass_p_offset) *mass_p_offset = L.mass_p;
  if (mass_bytes) *mass_bytes = sizeof(float) * static_cast<size_t>(B) * nc * sv::kDrawRanges;
  return SV_OK;
}

sv_status sv_verify_sample_phase(const void* target, int64_t t_row_stride, const void* draft, int64_t d_row_stride,
                                 const int32_t* draft_tokens, const float* temperature, uint64_t seed,
                                 uint32_t round, const int32_t* request_ids, sv_dtype dt, int B, int K, int V,
                                 int c_begin, int c_end, int phase, int32_t* out_tokens, int32_t* out_accept_len,
                                 float* out_p, float* out_q, uint8_t* out_flags, void* ws, size_t ws_bytes,
                                 void* stream) {
  if (phase < SV_PHASE_STATS || phase > SV_PHASE_PICK) return fail(SV_ERR_INVALID_ARG, "unknown phase %d", phase);
  if (V < 1 || V > (1 << 30) || (dt != SV_BF16 && dt != SV_F32)) return fail(SV_ERR_INVALID_ARG, "V=%d dt=%d", V, (int)dt);
  int cl, nc;
  sv::vocab_tiling(V, dt, &cl, &nc);
  if (c_begin < 0 || c_end > nc || c_begin >= c_end)
    return fail(SV_ERR_INVALID_ARG, "chunk range [%d, %d) outside [0, %d)", c_begin, c_end, nc);
  // the arrays hold this range's columns: rows need at least that many entries
  const int V_local = static_cast<int>(std::min<int64_t>(V, static_cast<int64_t>(c_end) * cl) -
                                       static_cast<int64_t>(c_begin) * cl);
  sv_status s = sv::validate_sample(target, t_row_stride, draft, d_row_stride, draft_tokens, temperature, dt, B, K,
                                    V_local, out_tokens, out_accept_len);
  if (s != SV_OK) return s;
  sv::VerifyParams p = sample_params(target, t_row_stride, draft, d_row_stride, draft_tokens, temperature, seed, round,
                                     request_ids, B, K, V, out_tokens, out_accept_len, out_p, out_q, out_flags);
  p.c_begin = c_begin;
  p.c_end = c_end;
  return verify_common(p, dt, true, ws, ws_bytes, stream, phase);
}

sv_status sv_verify_ragged(const void* target, int64_t t_row_stride, const int32_t* t_row_offsets, int64_t t_rows,
                           const void* draft, int64_t d_row_stride, const int32_t* d_row_offsets, int64_t d_rows,
                           const int32_t* draft_tokens, int tok_stride, const int32_t* keep_len,
                           const float* temperature, uint64_t seed, uint32_t round, const int32_t* request_ids,
                           sv_dtype dt, int B, int Kmax, int V, int32_t* out_tokens, int32_t* out_accept_len,
                           float* out_p, float* out_q, uint8_t* out_flags, void* ws, size_t ws_bytes,
                           void* stream) {
  sv_status s = check_common(target, t_row_stride, draft, d_row_stride, dt, B, Kmax, V, out_tokens, out_accept_len);
  if (s != SV_OK) return s;
  if (B > 0) {
    if (t_row_offsets == nullptr || keep_len == nullptr || temperature == nullptr)
      return fail(SV_ERR_INVALID_ARG, "t_row_offsets, keep_len and temperature are required");
    if (draft != nullptr && d_row_offsets == nullptr)
      return fail(SV_ERR_INVALID_ARG, "d_row_offsets is required with draft rows");
    if (draft_tokens != nullptr && tok_stride < Kmax)
      return fail(SV_ERR_INVALID_ARG, "tok_stride %d < Kmax %d", tok_stride, Kmax);
    if (draft_tokens == nullptr && draft == nullptr && Kmax > 0)
      return fail(SV_ERR_INVALID_ARG, "need draft logits or draft tokens");
    if (t_rows < 0 || (draft != nullptr && d_rows < 0))
      return fail(SV_ERR_INVALID_ARG, "t_rows / d_rows must be >= 0");
  }
  sv::VerifyParams p = {};
  p.target = target;
  p.t_row_stride = t_row_stride;
  p.t_off = t_row_offsets;
  p.t_rows = t_rows;
  p.draft = draft;
  p.d_row_stride = d_row_stride;
  p.d_off = d_row_offsets;
  p.d_rows = draft != nullptr ? d_rows : 0;
  p.tokens = draft_tokens;
  p.tok_stride = tok_stride;
  p.keep_len = keep_len;
  p.temperature = temperature;
  p.request_ids = request_ids;
  p.seed = seed;
  p.round = round;
  p.B = B;
  p.Kmax = Kmax;
  p.V = V;
  p.out_tokens = out_tokens;
  p.out_accept_len = out_accept_len;
  p.out_p = out_p;
  p.out_q = out_q;
  p.out_flags = out_flags;
  return verify_common(p, dt, true, ws, ws_bytes, stream);
}

sv_status sv_verify_tree(const void* target, int64_t t_row_stride, const void* draft, int64_t d_row_stride,
                         const int32_t* node_offsets, int64_t n_rows, const int32_t* parent, const int32_t* tokens,
                         const float* temperature, uint64_t seed, uint32_t round, const int32_t* request_ids,
                         sv_dtype dt, int B, int Nmax, int V, int32_t* out_path, int32_t* out_tokens,
                         int32_t* out_accept_len, uint8_t* out_flags, void* ws, size_t ws_bytes, void* stream) {
  if (Nmax < 1 || Nmax > SV_MAX_DRAFT + 1)
    return fail(SV_ERR_INVALID_ARG, "Nmax=%d outside [1, %d]", Nmax, SV_MAX_DRAFT + 1);
  sv_status s = check_common(target, t_row_stride, draft, d_row_stride, dt, B, Nmax - 1, V, out_tokens,
                             out_accept_len);
  if (s != SV_OK) return s;
  if (B > 0) {
    if (node_offsets == nullptr || parent == nullptr || tokens == nullptr || out_path == nullptr)
      return fail(SV_ERR_INVALID_ARG, "node_offsets, parent, tokens and out_path are required");
    if (n_rows < 0) return fail(SV_ERR_INVALID_ARG, "n_rows must be >= 0");
  }
  sv::VerifyParams p = {};
  p.tree = 1;
  p.target = target;
  p.t_row_stride = t_row_stride;
  p.t_off = node_offsets;
  p.t_rows = n_rows;
  p.draft = draft;
  p.d_row_stride = d_row_stride;
  p.d_off = node_offsets;
  p.d_rows = draft != nullptr ? n_rows : 0;
  p.tree_parent = parent;
  p.tree_tokens = tokens;
  p.temperature = temperature;
  p.request_ids = request_ids;
  p.seed = seed;
  p.round = round;
  p.B = B;
  p.Kmax = Nmax - 1;
  p.V = V;
  p.out_tokens = out_tokens;
  p.out_path = out_path;
  p.out_accept_len = out_accept_len;
  p.out_flags = out_flags;
  return verify_common(p, dt, true, ws, ws_bytes, stream);
}

// Checks and launch shared by both scheduling entry points; p arrives with its cost
// fields (cost_a, cost_b or the latency table) already set and checked.
static sv_status schedule_common(sv::ScheduleParams& p, const float* alpha, int alpha_stride,
                                 const int32_t* draft_len, int B, int Dmax, int budget, const float* ratios,
                                 int n_ratios, int objective, int32_t* out_keep_len, int32_t* out_row_offsets,
                                 int32_t* out_total_K, int64_t* out_utility_q48, void* ws, size_t ws_bytes,
                                 void* stream) {
  if (B < 1 || B > SV_MAX_BATCH) return fail(SV_ERR_INVALID_ARG, "B=%d outside [1, %d]", B, SV_MAX_BATCH);
  if (Dmax < 0 || Dmax > SV_MAX_DRAFT) return fail(SV_ERR_INVALID_ARG, "Dmax=%d outside [0, %d]", Dmax, SV_MAX_DRAFT);
  if (static_cast<int64_t>(B) * Dmax > SV_MAX_SCHEDULE_SLOTS)
    return fail(SV_ERR_INVALID_ARG, "B*Dmax=%lld exceeds %d", (long long)B * Dmax, SV_MAX_SCHEDULE_SLOTS);
  if (Dmax > 0 && (alpha == nullptr || alpha_stride < Dmax))
    return fail(SV_ERR_INVALID_ARG, "alpha is NULL or alpha_stride < Dmax");
  if (out_keep_len == nullptr || out_total_K == nullptr) return fail(SV_ERR_INVALID_ARG, "outputs are NULL");
  if (budget > 0 && budget < B) return fail(SV_ERR_INVALID_ARG, "budget %d below one slot per request (%d)", budget, B);
  if (objective != SV_OBJ_THROUGHPUT && objective != SV_OBJ_NET)
    return fail(SV_ERR_INVALID_ARG, "unknown objective %d", objective);
  if (ratios == nullptr) {
    const float def[4] = {0.25f, 0.5f, 0.75f, 1.0f};
    p.n_ratios = 4;
    for (int r = 0; r < 4; ++r) p.ratios[r] = def[r];
  } else {
    if (n_ratios < 1 || n_ratios > 8) return fail(SV_ERR_INVALID_ARG, "n_ratios=%d outside [1, 8]", n_ratios);
    for (int r = 0; r < n_ratios; ++r) {
      if (!(ratios[r] > 0.0f && ratios[r] <= 1.0f)) return fail(SV_ERR_INVALID_ARG, "ratio %d outside (0, 1]", r);
      p.ratios[r] = ratios[r];
    }
    p.n_ratios = n_ratios;
  }
  sv_status s = check_ws(ws, ws_bytes, 256);
  if (s != SV_OK) return s;
  int P = 1024;  // the sort holds at least one key per thread
  while (P < B * Dmax) P <<= 1;
  p.alpha = alpha;
  p.alpha_stride = alpha_stride;
  p.draft_len = draft_len;
  p.B = B;
  p.Dmax = Dmax;
  p.budget = budget;
  p.objective = objective;
  p.sort_size = P;
  p.merge = static_cast<int64_t>(B) * Dmax <= sv::kMergeMaxSlots ? 1 : 0;
  p.out_keep_len = out_keep_len;
  p.out_row_offsets = out_row_offsets;
  p.out_total_K = out_total_K;
  p.out_utility_q48 = out_utility_q48;
  p.status = static_cast<uint32_t*>(ws);
  const int e = sv::launch_schedule(p, stream);
  if (e != 0) return cuda_fail(e, "schedule launch");
  return SV_OK;
}

sv_status sv_schedule_depth(const float* alpha, int alpha_stride, const int32_t* draft_len, int B, int Dmax,
                            float cost_a, float cost_b, int budget, const float* ratios, int n_ratios, int objective,
                            int32_t* out_keep_len, int32_t* out_row_offsets, int32_t* out_total_K,
                            int64_t* out_utility_q48, void* ws, size_t ws_bytes, void* stream) {
  if (!(cost_a >= 0.0f) || !(cost_b >= 0.0f) || !(cost_a + cost_b > 0.0f) || std::isinf(cost_a) || std::isinf(cost_b))
    return fail(SV_ERR_INVALID_ARG, "cost model needs a >= 0, b >= 0, a + b > 0, finite");
  sv::ScheduleParams p = {};
  p.cost_a = static_cast<double>(cost_a);
  p.cost_b = static_cast<double>(cost_b);
  p.n_cost = 0;
  return schedule_common(p, alpha, alpha_stride, draft_len, B, Dmax, budget, ratios, n_ratios, objective,
                         out_keep_len, out_row_offsets, out_total_K, out_utility_q48, ws, ws_bytes, stream);
}

sv_status sv_schedule_depth_table(const float* alpha, int alpha_stride, const int32_t* draft_len, int B, int Dmax,
                                  const int32_t* cost_K, const double* cost_c, int n_cost, int budget,
                                  const float* ratios, int n_ratios, int objective, int32_t* out_keep_len,
                                  int32_t* out_row_offsets, int32_t* out_total_K, int64_t* out_utility_q48,
                                  void* ws, size_t ws_bytes, void* stream) {
  if (cost_K == nullptr || cost_c == nullptr) return fail(SV_ERR_INVALID_ARG, "cost table is NULL");
  if (n_cost < 1 || n_cost > SV_MAX_COST_KNOTS)
    return fail(SV_ERR_INVALID_ARG, "n_cost=%d outside [1, %d]", n_cost, SV_MAX_COST_KNOTS);
  sv::ScheduleParams p = {};
  for (int j = 0; j < n_cost; ++j) {
    if (cost_K[j] < 1 || (j > 0 && cost_K[j] <= cost_K[j - 1]))
      return fail(SV_ERR_INVALID_ARG, "cost_K[%d]=%d: token counts must be >= 1 and strictly increasing", j, cost_K[j]);
    if (!(cost_c[j] > 0.0) || std::isinf(cost_c[j]))
      return fail(SV_ERR_INVALID_ARG, "cost_c[%d] must be finite and positive", j);
    p.cost_K[j] = cost_K[j];
    p.cost_c[j] = cost_c[j];
  }
  for (int j = 0; j + 1 < n_cost; ++j)  // segment slopes, each rounded once after one rounded difference
    p.cost_s[j] = (p.cost_c[j + 1] - p.cost_c[j]) / static_cast<double>(p.cost_K[j + 1] - p.cost_K[j]);
  p.n_cost = n_cost;
  return schedule_common(p, alpha, alpha_stride, draft_len, B, Dmax, budget, ratios, n_ratios, objective,
                         out_keep_len, out_row_offsets, out_total_K, out_utility_q48, ws, ws_bytes, stream);
}

sv_status sv_query_status(void* ws, void* stream, uint32_t* device_status) {
  if (ws == nullptr || device_status == nullptr) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v != 0) {
    e = cudaMemsetAsync(ws, 0, sizeof(v), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *device_status = v;
  if (v == 0) return SV_OK;
  return (v & SV_DEV_TIMEOUT) ? SV_ERR_TIMEOUT : SV_ERR_DEVICE_INPUT;
}

const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARG: return "invalid argument";
    case SV_ERR_WORKSPACE: return "workspace too small or misaligned";
    case SV_ERR_CUDA: return "CUDA error";
    case SV_ERR_DEVICE_INPUT: return "device detected invalid input";
    case SV_ERR_TIMEOUT: return "a bounded device wait ran out";
  }
  return "unknown status";
}

const char* sv_last_error_string(void) { return g_err; }

void sv_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
}

sv_status sv_profile_collect(double* total_ms, int64_t* launches) {
  if (total_ms == nullptr || launches == nullptr) return fail(SV_ERR_INVALID_ARG, "NULL argument");
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "profile sync");
  for (const ProfRec& r : g_prof) {
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      total_ms[r.id] += ms;
      launches[r.id] += 1;
    }
  }
  return SV_OK;
}

void sv_profile_reset(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (const ProfRec& r : g_prof) {
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof.clear();
}

int64_t sv_launch_count(void) { return g_launches.load(); }

}  // extern "C"
