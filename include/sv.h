/*
 * sv.h -- C ABI of libsv: speculative-decoding draft verification and D-cut
 * verification-depth scheduling on one NVIDIA GB300 (sm_103a).
 *
 * Sources (web pages describing AngelSpec, Liu et al., Tencent):
 *   [explainer]  "AngelSpec: specialize the drafter, share the verification
 *                budget" (ai.thesatyajit.com/articles/angelspec)
 *   [release]    tradepoint.io article on the open-source AngelSpec release
 *   [abstract]   abstract of "AngelSpec: Towards Real-World High Performance
 *                Inference with Speculative Decoding"
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory    All array arguments are DEVICE pointers owned by the caller,
 *           except `ratios` of sv_schedule_depth (host).  The library never
 *           allocates device memory.  Scratch comes from a caller workspace
 *           of at least sv_workspace_size(...) bytes, 256-byte aligned, that
 *           must be zero-filled once before its first use; the library leaves
 *           it reusable (the status word stays zero unless a kernel flags an
 *           error, and every other region is written before it is read in
 *           each call).  One workspace must not be used by two calls that may
 *           run at the same time (different streams).
 * Streams   `stream` is a cudaStream_t passed as void* (NULL = legacy
 *           default stream).  All work is enqueued asynchronously; no call
 *           synchronizes, except sv_query_status and sv_profile_collect.
 *           Every call may be captured into a CUDA graph.
 * Errors    Every call returns an sv_status.  Host-side checks (NULL
 *           pointers, sizes, alignment, workspace size) return before any
 *           work is enqueued.  Values that only the device sees (token ids,
 *           temperatures, kept lengths, row offsets, confidences) are checked
 *           by the kernels: a bad request gets accept_len = -1 and all tokens
 *           -1, a bad schedule gets total_K = -1, and a bit is OR-ed into the
 *           workspace status word, read (and cleared) by sv_query_status.
 *           The kernels never trap; every wait in them is bounded.
 * Logits    Rows of V logits, contiguous, bf16 (SV_BF16) or float32
 *           (SV_F32), finite or -inf (a masked token).  NaN and +inf are not
 *           valid logits (results unspecified).  The row stride (elements) is
 *           at least V; rows may start at any element (the 16-byte aligned
 *           interior of each row is bulk-copied, the few elements outside it
 *           are loaded one by one), so no byte outside a row is read.
 * Randomness  The accept test and the resampling draw use Philox4x32-10
 *           (Salmon et al., SC'11) with key = (seed low, seed high word) and
 *           counter = (position, request id, purpose, round); purpose 0 is the
 *           accept test at drafted position k, purpose 1 the draw at position
 *           a.  u = (word0 >> 8) * 2^-24.
 */
#ifndef SV_H_
#define SV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,  /* NULL pointer, bad size, stride or alignment   */
  SV_ERR_WORKSPACE = 2,    /* workspace NULL, misaligned or too small        */
  SV_ERR_CUDA = 3,         /* a CUDA runtime call failed; see sv_last_error_string */
  SV_ERR_DEVICE_INPUT = 4, /* sv_query_status: a kernel flagged bad input    */
  SV_ERR_TIMEOUT = 5       /* sv_query_status: a bounded wait ran out        */
} sv_status;

typedef enum { SV_BF16 = 0, SV_F32 = 1 } sv_dtype;

/* operation ids for sv_workspace_size */
enum { SV_OP_VERIFY = 0, SV_OP_SCHEDULE = 1, SV_OP_TREE = 2 };

/* objective of sv_schedule_depth */
enum {
  SV_OBJ_THROUGHPUT = 0, /* maximise U(K) / c(K): projected throughput ([explainer] "D-cut") */
  SV_OBJ_NET = 1         /* maximise U(K) - c(K): expected utility minus cost ([abstract])    */
};

/* bits of the device status word */
enum {
  SV_DEV_BAD_TOKEN = 1u << 0,       /* drafted token outside [0, V)                  */
  SV_DEV_BAD_TEMPERATURE = 1u << 1, /* temperature < 0 or NaN                        */
  SV_DEV_BAD_KEEP_LEN = 1u << 2,    /* keep_len outside [0, Kmax]                    */
  SV_DEV_BAD_OFFSETS = 1u << 3,     /* row offsets leave fewer rows than needed      */
  SV_DEV_NO_DRAFT_ROWS = 1u << 4,   /* T > 0 (or greedy without tokens) but draft NULL */
  SV_DEV_BAD_ALPHA = 1u << 5,       /* confidence outside [0, 1] or NaN              */
  SV_DEV_BAD_DRAFT_LEN = 1u << 6,   /* draft_len outside [0, Dmax]                   */
  SV_DEV_TIMEOUT = 1u << 7,         /* a bounded wait inside a kernel ran out        */
  SV_DEV_BAD_PARENT = 1u << 8       /* tree node whose parent is not an earlier node */
};

/* per-request bits of out_flags */
enum {
  SV_FLAG_Q_ZERO = 1u << 0, /* q(x) == 0 at some accept test: accepted iff p(x) > 0 */
  SV_FLAG_Z_ZERO = 1u << 1, /* residual mass 0 at the rejection: drew from p_a       */
  SV_FLAG_INVALID = 1u << 2 /* the request's input was invalid (outputs are -1)      */
};

/* Limits (checked on the host). */
#define SV_MAX_BATCH 4096
#define SV_MAX_DRAFT 1023
#define SV_MAX_SCHEDULE_SLOTS 16384 /* sum_i draft_len_i for sv_schedule_depth */

/* ABI version; bumped on any signature change. */
int sv_abi_version(void);

/* Bytes of workspace that `op` needs for the given sizes (Kmax = largest number
 * of drafted positions per request; V = vocabulary size; dt = logit dtype).
 * Returns 0 for invalid sizes. */
size_t sv_workspace_size(int op, int B, int Kmax, int V, sv_dtype dt);

/*
 * sv_verify_greedy -- T = 0 verification ([release] "The MTP path": greedy
 * acceptance; [explainer] "MTP: fix position 2 and 3": one rejection voids
 * every later position).
 *
 * For each request i (0 <= i < B) with K drafted positions:
 *   g_k = first argmax of target row k (k = 0..K; row K is the bonus row)
 *   x_k = draft_tokens[i*K + k], or, when draft_tokens is NULL, the first
 *         argmax of draft row k
 *   a   = first k with x_k != g_k, else K
 *   out_tokens[i*(K+1) + j] = x_j for j < a, g_a at j = a, -1 after
 *   out_accept_len[i] = a
 * Layout: target row k of request i starts at target + (i*(K+1) + k) *
 * t_row_stride elements; draft row k at draft + (i*K + k) * d_row_stride.
 * draft may be NULL when draft_tokens is given (the draft rows are not read).
 * Exactly one of draft / draft_tokens may be NULL.  B >= 0, 0 <= K <= SV_MAX_DRAFT,
 * V >= 1.  B == 0 is a no-op.
 */
sv_status sv_verify_greedy(const void* target, int64_t t_row_stride, const void* draft,
                           int64_t d_row_stride, const int32_t* draft_tokens, sv_dtype dt, int B,
                           int K, int V, int32_t* out_tokens, int32_t* out_accept_len, void* ws,
                           size_t ws_bytes, void* stream);

/*
 * sv_verify_sample -- lossless rejection-sampling verification in one pass
 * over the logits ([release] "Why one universal drafter underperforms":
 * drafted tokens are verified together in one target pass by rejection
 * sampling; [explainer] "D-cut": verification stays exact).
 *
 * Per request i with temperature T = temperature[i] (device, float32):
 *   T == 0: exactly sv_verify_greedy with the given tokens (its draft rows are
 *           not read);
 *           out_p = 1 if x_k is the target argmax else 0, out_q = 1.
 *   T  > 0: p_k = softmax(target_k / T), q_k = softmax(draft_k / T)
 *           accept k  <=>  u_k * q_k(x_k) < p_k(x_k),  u_k = Philox(purpose 0, k)
 *           a = first rejected position, else K
 *           y ~ norm(max(0, p_a - q_a)) when a < K, else y ~ p_K (bonus row),
 *           drawn by inverse CDF in vocabulary order with u' = Philox(purpose 1, a)
 *           out_tokens: x_0..x_{a-1}, y, then -1; out_accept_len[i] = a
 *           out_p / out_q [B*K] (nullable): p_k(x_k), q_k(x_k) for every k < K
 *           out_flags [B] (nullable): SV_FLAG_* bits
 * request_ids (nullable => i) names the request in the Philox counter; `round`
 * is the counter's last word.  Layouts as in sv_verify_greedy; draft_tokens
 * is required; draft may be NULL only if every temperature is 0.
 */
sv_status sv_verify_sample(const void* target, int64_t t_row_stride, const void* draft,
                           int64_t d_row_stride, const int32_t* draft_tokens,
                           const float* temperature, uint64_t seed, uint32_t round,
                           const int32_t* request_ids, sv_dtype dt, int B, int K, int V,
                           int32_t* out_tokens, int32_t* out_accept_len, float* out_p,
                           float* out_q, uint8_t* out_flags, void* ws, size_t ws_bytes,
                           void* stream);

/*
 * sv_verify_ragged -- verification of per-request kept prefixes
 * ([explainer] "D-cut", Figure 3 panel 4: the target verifies only the
 * surviving tokens of each request).
 *
 * As sv_verify_sample, with n_i = keep_len[i] (device, 0 <= n_i <= Kmax)
 * positions per request and packed rows:
 *   target row k (0 <= k <= n_i) of request i: target + (t_row_offsets[i] + k) * t_row_stride
 *   draft  row k (0 <= k <  n_i) of request i: draft  + (d_row_offsets[i] + k) * d_row_stride
 *   drafted token k: draft_tokens[i * tok_stride + k]
 * t_row_offsets / d_row_offsets are device int32 [B+1]; t_rows / d_rows are the
 * numbers of rows the target / draft arrays hold.  The kernels check, per request,
 * t_row_offsets[i] >= 0, t_row_offsets[i+1] - t_row_offsets[i] >= n_i + 1 and
 * t_row_offsets[i] + n_i + 1 <= t_rows, and the same with n_i draft rows for the
 * requests that read them; a request that fails gets SV_DEV_BAD_OFFSETS and
 * reads no row.  d_row_offsets may be NULL when draft is NULL.  Outputs are
 * [B, Kmax+1] tokens and [B, Kmax] p/q (entries k >= n_i are NaN).  draft_tokens
 * may be NULL only if every temperature is 0 and draft is given (x_k = first
 * argmax of draft row k).  t_rows >= 0, d_rows >= 0 (d_rows is ignored when draft
 * is NULL).
 */
sv_status sv_verify_ragged(const void* target, int64_t t_row_stride, const int32_t* t_row_offsets,
                           int64_t t_rows, const void* draft, int64_t d_row_stride,
                           const int32_t* d_row_offsets, int64_t d_rows, const int32_t* draft_tokens,
                           int tok_stride, const int32_t* keep_len, const float* temperature,
                           uint64_t seed, uint32_t round, const int32_t* request_ids, sv_dtype dt,
                           int B, int Kmax, int V, int32_t* out_tokens, int32_t* out_accept_len,
                           float* out_p, float* out_q, uint8_t* out_flags, void* ws,
                           size_t ws_bytes, void* stream);

/*
 * Vocabulary-parallel verification (the LM head split across GPUs by vocabulary
 * columns, as in the pages' TP = 8 serving: [explainer] "The numbers", [release]
 * "Key Takeaways").  sv_verify_sample is four steps, and every step but the
 * accept chain is a sum or a search over the vocabulary in fixed chunks
 * (sv_vocab_chunks).  With the chunks split into contiguous ranges, one per
 * GPU, each GPU runs:
 *   SV_PHASE_STATS    its chunks of every row  -> chunk records (workspace)
 *   (all-gather of the records region: every GPU then holds every chunk's record)
 *   SV_PHASE_ACCEPT   the accept chain from all records: identical p, q, accepted
 *                     prefixes and draw state on every GPU
 *   SV_PHASE_WEIGHTS  its chunks' draw-weight range sums (workspace)
 *   (all-gather of the two range-sum regions)
 *   SV_PHASE_PICK     the crossing range from all range sums; only the GPU whose
 *                     chunks hold it writes the drawn token (out_tokens[i][a]) and
 *                     the Z_ZERO flag; the others leave them (initialise the token
 *                     to -1 and take the maximum across GPUs)
 * Results match sv_verify_sample's: the same chunk arithmetic, with the sums
 * grouped at the shard boundaries (a chunk record merges the chunks one CTA
 * streams in a row), so p and q agree to float32 rounding and the decisions
 * agree outside the near-boundary band.  sv_verify_regions gives the regions' workspace offsets: records are
 * [B][2K+1][nchunks] ChunkRecords of 16 bytes (a GPU's chunks are a contiguous
 * run of every (request, row)), range sums [B][nchunks][8] floats in two arrays.
 */
enum { SV_PHASE_STATS = 0, SV_PHASE_ACCEPT = 1, SV_PHASE_WEIGHTS = 2, SV_PHASE_PICK = 3 };

/* The vocabulary tiling of the verification kernels: nchunks chunks of chunk_len
 * entries (the last may be shorter). */
sv_status sv_vocab_chunks(int V, sv_dtype dt, int* chunk_len, int* nchunks);

/* Workspace offsets and sizes (bytes) of the chunk records and of the two
 * range-sum arrays of a verification workspace for (B, K, V, dt). */
sv_status sv_verify_regions(int B, int K, int V, sv_dtype dt, size_t* rec_offset, size_t* rec_bytes,
                            size_t* mass_offset, size_t* mass_p_offset, size_t* mass_bytes);

/* One step of sv_verify_sample over the vocabulary chunks [c_begin, c_end)
 * (0 <= c_begin < c_end <= nchunks).  Arguments as sv_verify_sample, except
 * that target / draft address the GPU's own columns: entry v of a row (v in
 * [c_begin, c_end) chunks) is at row + (v - c_begin * chunk_len).  STATS and
 * WEIGHTS read logits; ACCEPT and PICK read the workspace (PICK also reads the
 * crossing range's logits on the GPU that holds them). */
sv_status sv_verify_sample_phase(const void* target, int64_t t_row_stride, const void* draft, int64_t d_row_stride,
                                 const int32_t* draft_tokens, const float* temperature, uint64_t seed,
                                 uint32_t round, const int32_t* request_ids, sv_dtype dt, int B, int K, int V,
                                 int c_begin, int c_end, int phase, int32_t* out_tokens, int32_t* out_accept_len,
                                 float* out_p, float* out_q, uint8_t* out_flags, void* ws, size_t ws_bytes,
                                 void* stream);

/*
 * sv_verify_tree -- multi-candidate (token tree) verification by multi-step
 * speculative sampling (Miao et al., "SpecInfer", ASPLOS 2024, section 4.2);
 * a chain-shaped tree is exactly sv_verify_ragged ([explainer] "DFly": the
 * draft block is one causal chain; "D-cut": verification stays lossless).
 *
 * Request i has N_i = node_offsets[i+1] - node_offsets[i] nodes, 1 <= N_i <=
 * Nmax, in an order where each parent precedes its children; node 0 is the
 * root (the verified context).  With o = node_offsets[i] (device int32 [B+1]):
 *   parent[o + c]  (1 <= c < N_i): the parent node of node c, 0 <= parent < c
 *   tokens[o + c]  (1 <= c < N_i): node c's drafted token, in [0, V)
 *   target + (o + c) * t_row_stride: target logits of the token after node c's path
 *   draft  + (o + c) * d_row_stride: the draft logits node c's children were drafted from
 * (entries c = 0 of parent / tokens and the draft rows of leaves are not read).
 * n_rows is the number of rows both arrays hold; every request's rows must lie
 * below it (else SV_DEV_BAD_OFFSETS).
 *
 * Per request with T = temperature[i], walking from the root: at a node with
 * children x_1..x_m (in node order), p = softmax(target/T), q = softmax(draft/T):
 *   p' = p; for j = 1..m: accept x_j iff u_j * q(x_j) < p'(x_j), u_j =
 *   Philox(purpose 0, position = node index of x_j minus 1); on a rejection
 *   p' = norm(max(0, p' - q)).  An accepted child is emitted and the walk goes
 *   on from it; if all are rejected, y ~ p' is drawn by inverse CDF in vocabulary
 *   order (u' = Philox(purpose 1, position = the node's index)) and the walk
 *   stops.  At a node without children y ~ p (the bonus draw).  T == 0: the
 *   first child equal to the target argmax (lowest index on ties) is accepted;
 *   otherwise the argmax is emitted and the walk stops.  Draft rows are read only
 *   for T > 0 (draft may be NULL when every T is 0).
 * Outputs (device): out_path [B, Nmax] int32: the accepted nodes (root
 * excluded) then -1; out_tokens [B, Nmax] int32: their tokens, then y, then -1;
 * out_accept_len [B]: accepted nodes; out_flags [B] (nullable): SV_FLAG_* bits.
 * Workspace: sv_workspace_size(SV_OP_TREE, B, Nmax, V, dt).  Invalid requests
 * get -1 outputs, SV_FLAG_INVALID and a SV_DEV_* bit (bad parents:
 * SV_DEV_BAD_PARENT, bad tokens: SV_DEV_BAD_TOKEN, N_i outside [1, Nmax]:
 * SV_DEV_BAD_KEEP_LEN).
 */
sv_status sv_verify_tree(const void* target, int64_t t_row_stride, const void* draft, int64_t d_row_stride,
                         const int32_t* node_offsets, int64_t n_rows, const int32_t* parent,
                         const int32_t* tokens, const float* temperature, uint64_t seed, uint32_t round,
                         const int32_t* request_ids, sv_dtype dt, int B, int Nmax, int V,
                         int32_t* out_path, int32_t* out_tokens, int32_t* out_accept_len,
                         uint8_t* out_flags, void* ws, size_t ws_bytes, void* stream);

/*
 * sv_schedule_depth -- D-cut batch-shared verification-depth allocation
 * ([explainer] "D-cut: verification depth is a shared resource", Figure 3
 * panels 2-3 and eq. K_rho; [abstract]: expected utility with a profiled
 * cost model).
 *
 * alpha [B, alpha_stride] float32 (device): alpha[i*alpha_stride + k-1] is the
 * drafter's confidence in drafted position k (1 <= k <= D_i), in [0, 1].
 * draft_len [B] (device, nullable => Dmax) gives D_i.
 *   s_{i,0} = 1, s_{i,k} = s_{i,k-1} * alpha_{i,k}  (float32, left to right)
 *   slot 0 of every request is always kept; the other N - B slots
 *   (N = sum_i (D_i + 1)) are ranked by (s desc, request asc, position asc)
 *   candidates K = clip(max(B, ceil(rho * N)), B, cap) for rho in ratios
 *   (host array, NULL => {0.25, 0.5, 0.75, 1.0}, n_ratios <= 8), cap =
 *   min(budget, N) (budget <= 0 => N); duplicates collapse
 *   U(K) = sum of round(s * 2^48) over the top K slots (exact int64)
 *   cost c(K) = cost_a + cost_b * K (float64); objective SV_OBJ_THROUGHPUT
 *   (U / 2^48 / c) or SV_OBJ_NET (U / 2^48 - c); ties pick the smaller K
 * Outputs (device): out_keep_len [B] = n_i (kept drafted positions),
 * out_row_offsets [B+1] (nullable) = packed target-row offsets with n_i + 1
 * rows per request, out_total_K [1], out_utility_q48 [1] (nullable) = U(K).
 * Limits: 1 <= B <= SV_MAX_BATCH, 0 <= Dmax <= SV_MAX_DRAFT,
 * B * Dmax <= SV_MAX_SCHEDULE_SLOTS, budget <= 0 or budget >= B,
 * cost_a >= 0, cost_b >= 0, cost_a + cost_b > 0.
 */
sv_status sv_schedule_depth(const float* alpha, int alpha_stride, const int32_t* draft_len, int B,
                            int Dmax, float cost_a, float cost_b, int budget, const float* ratios,
                            int n_ratios, int objective, int32_t* out_keep_len,
                            int32_t* out_row_offsets, int32_t* out_total_K,
                            int64_t* out_utility_q48, void* ws, size_t ws_bytes, void* stream);

/*
 * sv_schedule_depth_table -- sv_schedule_depth with the profiled runtime latency
 * table in place of the linear cost ([explainer] D-cut section, Figure 3 panel 2:
 * a cost table profiled at startup across batch sizes and keep ratios picks the
 * ratio of largest projected throughput).  Batch size and keep ratio together set
 * the number of verified tokens K, so the table is latency against K:
 *   cost_K [n_cost] (host): token counts, K_0 >= 1, strictly increasing
 *   cost_c [n_cost] (host): the latency of verifying cost_K[j] tokens, finite, > 0
 *   1 <= n_cost <= SV_MAX_COST_KNOTS; both arrays are copied at the call.
 * c(K) = cost_c[0] for K <= cost_K[0], cost_c[n-1] for K >= cost_K[n-1], else
 * with cost_K[j] <= K < cost_K[j+1], in slope form: s_j = (c_{j+1} - c_j) /
 * (K_{j+1} - K_j) (computed on the host at the call), c = c_j + s_j * (K - K_j),
 * float64, each operation rounded once in that order.  Everything else (scores, ranking, candidates, U(K), both objectives,
 * outputs, limits other than the cost, workspace) is as in sv_schedule_depth.
 * A bad table returns SV_ERR_INVALID_ARG and enqueues nothing.
 */
#define SV_MAX_COST_KNOTS 32
sv_status sv_schedule_depth_table(const float* alpha, int alpha_stride, const int32_t* draft_len,
                                  int B, int Dmax, const int32_t* cost_K, const double* cost_c,
                                  int n_cost, int budget, const float* ratios, int n_ratios,
                                  int objective, int32_t* out_keep_len, int32_t* out_row_offsets,
                                  int32_t* out_total_K, int64_t* out_utility_q48, void* ws,
                                  size_t ws_bytes, void* stream);

/*
 * sv_verify_sample_noalloc -- sv_verify_sample without a caller workspace.  The AngelSpec
 * pages have no counterpart to this call; it exists for callers that cannot call cudaMalloc:
 * code that runs while its stream is being captured into a CUDA graph (an allocation there
 * would break the capture), plugins inside a host framework whose device memory belongs to
 * that framework's own allocator, and serving loops that allow no allocation on the hot path
 * (cudaMalloc can synchronize the whole device).
 *
 * Arguments and results are those of sv_verify_sample, without ws / ws_bytes; the caller
 * still passes every input and output.  The scratch is an array of SV_NOALLOC_SCRATCH_BYTES
 * (4 MiB) inside the library, held on every GPU that loads the library until the process
 * exits.  A call whose sv_workspace_size(SV_OP_VERIFY, B, K, V, dt) exceeds it returns
 * SV_ERR_WORKSPACE (message in sv_last_error_string) and enqueues nothing.  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) and caches it; make
 * that first call before any stream capture.  Each call clears only the array's status word, with
 * cudaMemsetAsync on `stream`; every other region of the array is written before it is read.
 * All calls share the one
 * array: calls that may overlap on the GPU (different streams of one device) race.  Nothing
 * is allocated: no cudaMalloc, cudaFree or allocating library routine.  Input errors that
 * only the kernels see are reported through out_accept_len = -1 and out_flags
 * (SV_FLAG_INVALID); there is no status word to query.
 */
#define SV_NOALLOC_SCRATCH_BYTES (4u << 20)
sv_status sv_verify_sample_noalloc(const void* target, int64_t t_row_stride, const void* draft,
                                   int64_t d_row_stride, const int32_t* draft_tokens,
                                   const float* temperature, uint64_t seed, uint32_t round,
                                   const int32_t* request_ids, sv_dtype dt, int B, int K, int V,
                                   int32_t* out_tokens, int32_t* out_accept_len, float* out_p,
                                   float* out_q, uint8_t* out_flags, void* stream);

/* Testing hook for the bounded waits.  The next verification call (any entry
 * point, on any thread) runs with every wait of its streaming kernel limited to
 * wait_limit_ms (instead of about 2 s), and the producer of that kernel's first
 * CTA issues no copy: the CTA's consumers wait for a stage nothing fills, give
 * up after the limit, record SV_DEV_TIMEOUT and finish the launch on what they
 * hold (that call's outputs are meaningless).  No GPU fault is involved and no
 * copy is in flight when the CTA exits; sv_query_status then returns
 * SV_ERR_TIMEOUT and the workspace stays usable.  wait_limit_ms <= 0 cancels a
 * pending request. */
void sv_test_stall_next_verify(int wait_limit_ms);

/* Synchronizes `stream`, returns the workspace's device status word in
 * *device_status (SV_DEV_* bits) and clears it.  Returns SV_OK if the word was
 * zero, SV_ERR_TIMEOUT if SV_DEV_TIMEOUT is set, else SV_ERR_DEVICE_INPUT. */
sv_status sv_query_status(void* ws, void* stream, uint32_t* device_status);

const char* sv_status_string(sv_status s);

/* Text of the last SV_ERR_CUDA / SV_ERR_INVALID_ARG on this host thread. */
const char* sv_last_error_string(void);

/* Instrumentation.  While enabled, every library kernel launch is bracketed by
 * CUDA events on its stream (recorded into the graph when the stream is being
 * captured, so a graph replay re-records them).  sv_profile_collect
 * synchronizes the device and adds, for every bracket recorded since the last
 * sv_profile_reset, its elapsed time to total_ms[kernel id] and 1 to
 * launches[kernel id] (arrays of SV_NUM_KERNELS).  sv_profile_reset forgets the
 * brackets.  sv_launch_count returns the number of library kernel launches (or
 * captured launch nodes) since the library was loaded. */
enum {
  SV_KERNEL_ROW_STATS = 0, /* streaming pass over the logit rows                          */
  SV_KERNEL_COMBINE = 1,   /* accept chain (+ per-chunk draw weights for short requests)  */
  SV_KERNEL_SCHEDULE = 2,  /* D-cut depth allocation                                      */
  SV_KERNEL_MASS = 3,      /* per-chunk draw weights for long requests                    */
  SV_KERNEL_PICK = 4,      /* inverse-CDF draw                                            */
  SV_KERNEL_TREE_WALK = 5, /* tree verification: the walk from the root                   */
  SV_NUM_KERNELS = 6
};
void sv_profile_enable(int on);
sv_status sv_profile_collect(double* total_ms, int64_t* launches);
void sv_profile_reset(void);
int64_t sv_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* SV_H_ */
