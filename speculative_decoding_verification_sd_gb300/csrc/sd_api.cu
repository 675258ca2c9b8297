// sd_api.cu -- host side of the C ABI declared in include/sd.h: argument
// validation, workspace carving, launch-shape selection and kernel launches.
// No entry point allocates device memory or synchronises the stream.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "sd_internal.h"

namespace {

thread_local char g_last_error[256] = "no error";

// Records a failing CUDA call for sd_last_error_string(); returns it unchanged.
cudaError_t note(cudaError_t e) {
  if (e != cudaSuccess) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(e),
             cudaGetErrorString(e));
  }
  return e;
}

int pow2ceil(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

size_t align16(size_t v) { return (v + 15) & ~static_cast<size_t>(15); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct VerifyWs {
  uint8_t* accept;
  int* cand;
  int* status;
};

size_t verify_ws_bytes(int bs, int k_max) {
  const size_t rows = static_cast<size_t>(bs) * (k_max + 1);
  return align16(rows) + align16(rows * 4) + 16;
}

VerifyWs carve(void* ws, int bs, int k_max) {
  const size_t rows = static_cast<size_t>(bs) * (k_max + 1);
  char* b = static_cast<char*>(ws);
  VerifyWs w;
  w.accept = reinterpret_cast<uint8_t*>(b);
  w.cand = reinterpret_cast<int*>(b + align16(rows));
  w.status = reinterpret_cast<int*>(b + align16(rows) + align16(rows * 4));
  return w;
}

// Per-device cache of the co-resident cluster count for a launch shape.
struct ClusterCache {
  std::mutex mu;
  struct Entry {
    int dev, elem, C, S, SL, threads, bulk;
    size_t smem;
    int n;
  } e[64];
  int used = 0;
};
ClusterCache g_clusters;

cudaError_t resident_clusters(int elem, const sdk::VerifyShape& s, int* n) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lk(g_clusters.mu);
    for (int k = 0; k < g_clusters.used; ++k) {
      const auto& c = g_clusters.e[k];
      if (c.dev == dev && c.elem == elem && c.C == s.C && c.S == s.S && c.SL == s.SL &&
          c.threads == s.threads && c.bulk == static_cast<int>(s.bulk) && c.smem == s.smem) {
        *n = c.n;
        return cudaSuccess;
      }
    }
  }
  int m = 0;
  err = sdk::max_active_clusters(elem, s, &m);
  if (err != cudaSuccess) return err;
  if (m < 1) return cudaErrorInvalidConfiguration;
  std::lock_guard<std::mutex> lk(g_clusters.mu);
  if (g_clusters.used < 64)
    g_clusters.e[g_clusters.used++] = {dev, elem, s.C, s.S, s.SL, s.threads,
                                      static_cast<int>(s.bulk), s.smem, m};
  *n = m;
  return cudaSuccess;
}

sd_status shape_for(int V, sd_dtype dt, int bs, const sd_launch_cfg* cfg, bool bulk,
                    sdk::VerifyShape* shape) {
  const int elem = dt == SD_F32 ? 4 : 2;
  bool fits = false;
  if (note(sdk::choose_verify_shape(V, elem, bs, cfg, bulk, shape, &fits)) != cudaSuccess)
    return SD_ERR_CUDA;
  if (!fits) return SD_ERR_UNSUPPORTED;
  int m = 0;
  if (note(resident_clusters(elem, *shape, &m)) != cudaSuccess) return SD_ERR_CUDA;
  if (shape->clusters <= 0 || shape->clusters > m) shape->clusters = m;
  return SD_OK;
}

}  // namespace

extern "C" {

int sd_abi_version(void) { return 1; }

const char* sd_last_error_string(void) { return g_last_error; }

const char* sd_status_string(sd_status s) {
  switch (s) {
    case SD_OK: return "ok";
    case SD_ERR_INVALID_ARG: return "invalid argument";
    case SD_ERR_SHAPE: return "inconsistent sizes";
    case SD_ERR_UNSUPPORTED: return "beyond this build's limits";
    case SD_ERR_CUDA: return "CUDA runtime or launch error";
    case SD_ERR_DEVICE_CHECK: return "device-side check failed";
  }
  return "unknown status";
}

size_t sd_plan_workspace_bytes(int bs, int k_max) {
  (void)bs;
  (void)k_max;
  return 0;
}

sd_status sd_plan(const float* conf_logits, const float* budget_conf, const int* budget_draft_lens,
                  int bs_budget, const int* draft_lens, int bs, int k_max, const float* cost_table,
                  int cost_len, int T, sd_mode mode, int* B_out, uint8_t* slot_mask,
                  int* num_verified, int* cu_seqlens, int* err_flag, void* workspace,
                  size_t ws_bytes, void* stream) {
  (void)workspace;
  (void)ws_bytes;
  if (bs < 1 || k_max < 0) return SD_ERR_INVALID_ARG;
  if (k_max > SD_MAX_K) return SD_ERR_UNSUPPORTED;
  if (mode != SD_MODE_ADAPTIVE && mode != SD_MODE_ALL_SLOTS) return SD_ERR_INVALID_ARG;
  if (!draft_lens || !B_out || !num_verified || !cu_seqlens || !err_flag) return SD_ERR_INVALID_ARG;
  if (k_max > 0 && !slot_mask) return SD_ERR_INVALID_ARG;
  const int P = pow2ceil(k_max < 1 ? 1 : k_max);
  if (static_cast<long long>(pow2ceil(bs)) * P > SD_MAX_PLAN_SLOTS) return SD_ERR_UNSUPPORTED;
  int NPb = 0;
  if (mode == SD_MODE_ADAPTIVE) {
    if (!conf_logits || !cost_table) return SD_ERR_INVALID_ARG;
    if (T < 1 || cost_len < 1) return SD_ERR_INVALID_ARG;
    if (T >= cost_len) return SD_ERR_SHAPE;
    if (budget_conf) {
      if (!budget_draft_lens || bs_budget < 1) return SD_ERR_INVALID_ARG;
      if (static_cast<long long>(pow2ceil(bs_budget)) * P > SD_MAX_PLAN_SLOTS)
        return SD_ERR_UNSUPPORTED;
      NPb = pow2ceil(bs_budget) * P;
    }
  }
  sdk::PlanParams p;
  p.conf = conf_logits;
  p.budget_conf = mode == SD_MODE_ADAPTIVE ? budget_conf : nullptr;
  p.budget_lens = budget_draft_lens;
  p.bs_budget = bs_budget;
  p.lens = draft_lens;
  p.bs = bs;
  p.k_max = k_max;
  p.cost = cost_table;
  p.cost_len = cost_len;
  p.T = T;
  p.mode = mode;
  p.P = P;
  p.NP = pow2ceil(bs) * P;
  p.NPb = p.budget_conf ? NPb : 0;
  p.B_out = B_out;
  p.mask = slot_mask;
  p.num_verified = num_verified;
  p.cu = cu_seqlens;
  p.err = err_flag;
  return note(sdk::launch_plan(p, static_cast<cudaStream_t>(stream))) == cudaSuccess ? SD_OK
                                                                                    : SD_ERR_CUDA;
}

size_t sd_verify_workspace_bytes(int bs, int k_max) {
  if (bs < 1 || k_max < 0) return 0;
  return verify_ws_bytes(bs, k_max);
}

static sd_status check_verify_common(int bs, int k_max, void* workspace, size_t ws_bytes) {
  if (bs < 1 || k_max < 0) return SD_ERR_INVALID_ARG;
  if (k_max > SD_MAX_K || bs > SD_MAX_VERIFY_BS) return SD_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace)) return SD_ERR_INVALID_ARG;
  if (ws_bytes < verify_ws_bytes(bs, k_max)) return SD_ERR_SHAPE;
  return SD_OK;
}

sd_status sd_verify_rows(const void* target_logits, const void* draft_logits, sd_dtype dt, int V,
                         const int* draft_ids, const float* uniforms, const float* temps,
                         const int* cu_seqlens, int bs, int k_max, float* probs_out,
                         int* err_flag, void* workspace, size_t ws_bytes,
                         const sd_launch_cfg* cfg, void* stream) {
  sd_status st = check_verify_common(bs, k_max, workspace, ws_bytes);
  if (st != SD_OK) return st;
  if (dt != SD_F32 && dt != SD_BF16) return SD_ERR_INVALID_ARG;
  if (V < 1) return SD_ERR_INVALID_ARG;
  if (V > SD_MAX_V) return SD_ERR_UNSUPPORTED;
  if (!target_logits || !uniforms || !temps || !cu_seqlens || !err_flag) return SD_ERR_INVALID_ARG;
  if (k_max > 0 && !draft_ids) return SD_ERR_INVALID_ARG;
  if (cfg && (cfg->cluster < 0 || cfg->stages < 0 || cfg->clusters < 0 || cfg->threads < 0))
    return SD_ERR_INVALID_ARG;
  const int elem = dt == SD_F32 ? 4 : 2;
  const bool bulk = (static_cast<size_t>(V) * elem) % 16 == 0 && aligned16(target_logits) &&
                    (draft_logits == nullptr || aligned16(draft_logits));
  sdk::VerifyShape shape;
  st = shape_for(V, dt, bs, cfg, bulk, &shape);
  if (st != SD_OK) return st;
  VerifyWs w = carve(workspace, bs, k_max);
  sdk::VerifyParams p;
  p.target = target_logits;
  p.draft = draft_logits;
  p.V = V;
  p.draft_ids = draft_ids;
  p.uniforms = uniforms;
  p.temps = temps;
  p.cu = cu_seqlens;
  p.bs = bs;
  p.k_max = k_max;
  p.probs_out = probs_out;
  p.err = err_flag;
  p.ws_accept = w.accept;
  p.ws_cand = w.cand;
  p.ws_status = w.status;
  p.C = shape.C;
  p.S = shape.S;
  p.SL = shape.SL;
  p.stage_bytes = static_cast<int>(2 * static_cast<size_t>(shape.SL) * elem);
  return note(sdk::launch_verify_rows(p, elem, shape, static_cast<cudaStream_t>(stream))) ==
                 cudaSuccess
             ? SD_OK
             : SD_ERR_CUDA;
}

sd_status sd_verify_finalize(const int* draft_ids, const int* cu_seqlens, int bs, int k_max,
                             int* accepted_len, int* out_tokens, int* err_flag,
                             const void* workspace, size_t ws_bytes, void* stream) {
  sd_status st = check_verify_common(bs, k_max, const_cast<void*>(workspace), ws_bytes);
  if (st != SD_OK) return st;
  if (!cu_seqlens || !accepted_len || !out_tokens || !err_flag) return SD_ERR_INVALID_ARG;
  if (k_max > 0 && !draft_ids) return SD_ERR_INVALID_ARG;
  VerifyWs w = carve(const_cast<void*>(workspace), bs, k_max);
  return note(sdk::launch_verify_finalize(draft_ids, cu_seqlens, bs, k_max, accepted_len,
                                          out_tokens, err_flag, w.accept, w.cand, w.status,
                                          static_cast<cudaStream_t>(stream))) == cudaSuccess
             ? SD_OK
             : SD_ERR_CUDA;
}

sd_status sd_verify(const void* target_logits, const void* draft_logits, sd_dtype dt, int V,
                    const int* draft_ids, const float* uniforms, const float* temps,
                    const int* cu_seqlens, int bs, int k_max, int* accepted_len, int* out_tokens,
                    float* probs_out, int* err_flag, void* workspace, size_t ws_bytes,
                    void* stream) {
  if (!accepted_len || !out_tokens) return SD_ERR_INVALID_ARG;
  sd_status st = sd_verify_rows(target_logits, draft_logits, dt, V, draft_ids, uniforms, temps,
                                cu_seqlens, bs, k_max, probs_out, err_flag, workspace, ws_bytes,
                                nullptr, stream);
  if (st != SD_OK) return st;
  return sd_verify_finalize(draft_ids, cu_seqlens, bs, k_max, accepted_len, out_tokens, err_flag,
                            workspace, ws_bytes, stream);
}

sd_status sd_verify_launch_info(int V, sd_dtype dt, const sd_launch_cfg* req,
                                sd_launch_cfg* chosen, int* threads, size_t* smem_bytes) {
  if (V < 1 || (dt != SD_F32 && dt != SD_BF16) || !chosen) return SD_ERR_INVALID_ARG;
  const int elem = dt == SD_F32 ? 4 : 2;
  const bool bulk = (static_cast<size_t>(V) * elem) % 16 == 0;
  sdk::VerifyShape shape;
  sd_status st = shape_for(V, dt, 1, req, bulk, &shape);
  if (st != SD_OK) return st;
  chosen->cluster = shape.C;
  chosen->stages = shape.S;
  chosen->clusters = shape.clusters;
  chosen->threads = shape.threads;
  if (threads) *threads = shape.threads;
  if (smem_bytes) *smem_bytes = shape.smem;
  return SD_OK;
}

}  // extern "C"
