// sv_verify_sample_noalloc: sampled verification for callers that cannot allocate device
// memory.  The scratch that sv_verify_sample takes from a caller workspace lives here in a
// file-scope device array instead; the caller still passes its inputs and outputs.
#include <cuda_runtime.h>

#include <mutex>

#include "sv_internal.h"

namespace {

constexpr size_t kScratchBytes = SV_NOALLOC_SCRATCH_BYTES;

// Loaded with the library on every GPU that uses it and kept until the process exits.  In host
// code this name is only a stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" sv_status sv_verify_sample_noalloc(const void* target, int64_t t_row_stride, const void* draft,
                                              int64_t d_row_stride, const int32_t* draft_tokens,
                                              const float* temperature, uint64_t seed, uint32_t round,
                                              const int32_t* request_ids, sv_dtype dt, int B, int K, int V,
                                              int32_t* out_tokens, int32_t* out_accept_len, float* out_p,
                                              float* out_q, uint8_t* out_flags, void* stream) {
  sv_status s = sv::validate_sample(target, t_row_stride, draft, d_row_stride, draft_tokens, temperature, dt, B, K,
                                    V, out_tokens, out_accept_len);
  if (s != SV_OK || B == 0) return s;
  const size_t need = sv_workspace_size(SV_OP_VERIFY, B, K, V, dt);
  if (need == 0) {
    return sv::set_error(SV_ERR_INVALID_ARG, "invalid sizes B=%d K=%d V=%d", B, K, V);
  }
  if (need > kScratchBytes) {
    return sv::set_error(SV_ERR_WORKSPACE,
                         "B=%d K=%d V=%d needs %zu bytes of scratch; the built-in scratch holds %zu bytes "
                         "(use sv_verify_sample with a caller workspace)",
                         B, K, V, need, kScratchBytes);
  }
  void* ws = nullptr;
  cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess) {
    return sv::set_error(SV_ERR_CUDA, "scratch address: %s", cudaGetErrorString(e));
  }
  // The array keeps the previous call's contents: the status word must start at zero
  // (everything else is written before it is read).
  int cl, nc;
  sv::vocab_tiling(V, dt, &cl, &nc);
  const sv::VerifyLayout L = sv::verify_layout(B, K, nc);
  e = cudaMemsetAsync(ws, 0, L.req, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    return sv::set_error(SV_ERR_CUDA, "scratch clear: %s", cudaGetErrorString(e));
  }
  return sv_verify_sample(target, t_row_stride, draft, d_row_stride, draft_tokens, temperature, seed, round,
                          request_ids, dt, B, K, V, out_tokens, out_accept_len, out_p, out_q, out_flags, ws,
                          kScratchBytes, stream);
}
