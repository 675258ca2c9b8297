// noalloc.cu -- sd_verify_noalloc: the sampling stage on a workspace that
// lives in a file-scope device array, so a call allocates nothing.  It serves
// callers that cannot call cudaMalloc around the step (a serving loop that
// reserved the device's memory up front, or a process whose allocator belongs
// to another framework).
//
// The scratch is SD_NOALLOC_SCRATCH_BYTES of static device memory, loaded
// with the library and held by every device that loads it until the process
// exits.  In host code `g_scratch` names a host-side stand-in, not a device
// address, so its device address is looked up with cudaGetSymbolAddress, with
// the device current: on the first call on a device, and again on every call
// that is not being captured into a graph (so a call after a device reset, or
// from another context on the device, gets the address valid there).  Under
// capture the address cached by the last call outside capture is used.
//
// Each call checks its arguments first, then clears on the caller's stream
// the part of the workspace that must start at zero (the counters), then
// launches the sampling kernel on it.  Two calls that overlap in time on one
// device share the scratch and race.
#include <cuda_runtime.h>

#include <mutex>

#include "sd_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[SD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// The scratch's device address on the current device.
cudaError_t scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cs);
  if (e == cudaErrorStreamCaptureImplicit) {  // legacy stream while another stream captures
    (void)cudaGetLastError();
    cs = cudaStreamCaptureStatusActive;
  } else if (e != cudaSuccess) {
    return e;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (cs == cudaStreamCaptureStatusNone || g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

sd_status cuda_failure(cudaError_t e) {
  return sdk::refuse(SD_ERR_CUDA, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
}

}  // namespace

extern "C" sd_status sd_verify_noalloc(const void* target_logits, const void* draft_logits,
                                       sd_dtype dt, int V, const int* draft_ids,
                                       const float* uniforms, const float* temps,
                                       const int* cu_seqlens, int bs, int k_max,
                                       int* accepted_len, int* out_tokens, float* probs_out,
                                       int* err_flag, void* stream) {
  sdk::clear_last_error();
  sdk::VerifyCall call;
  const sd_status st = sdk::verify_setup(target_logits, draft_logits, dt, V, draft_ids, uniforms,
                                         temps, cu_seqlens, bs, k_max, accepted_len, out_tokens,
                                         probs_out, err_flag, nullptr, &call);
  if (st != SD_OK) return st;
  if (call.ws_need > static_cast<size_t>(SD_NOALLOC_SCRATCH_BYTES))
    return sdk::refuse(SD_ERR_UNSUPPORTED,
                       "sd_verify_noalloc: bs=%d, k_max=%d, V=%d needs %zu bytes of workspace; "
                       "the static scratch holds %zu",
                       bs, k_max, V, call.ws_need, static_cast<size_t>(SD_NOALLOC_SCRATCH_BYTES));
  const sd_status sh = sdk::verify_shape(&call);
  if (sh != SD_OK) return sh;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  cudaError_t e = scratch_address(s, &ws);
  if (e != cudaSuccess) return cuda_failure(e);
  e = cudaMemsetAsync(static_cast<char*>(ws) + call.zero_off, 0, call.ws_need - call.zero_off, s);
  if (e != cudaSuccess) return cuda_failure(e);
  sdk::verify_bind(&call, ws);
  return sdk::verify_launch(call, stream);
}
