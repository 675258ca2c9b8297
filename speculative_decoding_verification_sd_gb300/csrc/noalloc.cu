// noalloc.cu -- sd_verify_noalloc: sd_verify on a workspace that lives in a
// file-scope device array, so a call allocates nothing.
//
// The scratch is SD_NOALLOC_SCRATCH_BYTES of static device memory, loaded
// with the library.  Its address is looked up once per device with
// cudaGetSymbolAddress and kept; later calls only read the cached address.
// Each call clears, on the caller's stream, the part of the workspace that
// must start at zero (the residual sums and the counters) and then runs
// sd_verify on it.  Two calls that overlap in time on one device share the
// scratch and race.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "sd_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[SD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// The scratch's device address on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" sd_status sd_verify_noalloc(const void* target_logits, const void* draft_logits,
                                       sd_dtype dt, int V, const int* draft_ids,
                                       const float* uniforms, const float* temps,
                                       const int* cu_seqlens, int bs, int k_max,
                                       int* accepted_len, int* out_tokens, float* probs_out,
                                       int* err_flag, void* stream) {
  if (bs < 1 || k_max < 0) return SD_ERR_INVALID_ARG;
  if (k_max > SD_MAX_K || bs > SD_MAX_VERIFY_BS) return SD_ERR_UNSUPPORTED;
  const size_t need = sd_verify_workspace_bytes(bs, k_max);
  if (need > static_cast<size_t>(SD_NOALLOC_SCRATCH_BYTES)) {
    char msg[160];
    snprintf(msg, sizeof msg,
             "sd_verify_noalloc: bs=%d, k_max=%d needs %zu bytes of workspace; the static "
             "scratch holds %zu",
             bs, k_max, need, static_cast<size_t>(SD_NOALLOC_SCRATCH_BYTES));
    sdk::set_last_error(msg);
    return SD_ERR_UNSUPPORTED;
  }
  void* ws = nullptr;
  cudaError_t e = scratch_address(&ws);
  if (e == cudaSuccess) {
    const size_t zero = sdk::verify_ws_zero_offset(bs, k_max);
    e = cudaMemsetAsync(static_cast<char*>(ws) + zero, 0, need - zero,
                        static_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) {
    char msg[160];
    snprintf(msg, sizeof msg, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    sdk::set_last_error(msg);
    return SD_ERR_CUDA;
  }
  return sd_verify(target_logits, draft_logits, dt, V, draft_ids, uniforms, temps, cu_seqlens, bs,
                   k_max, accepted_len, out_tokens, probs_out, err_flag, ws, need, stream);
}
