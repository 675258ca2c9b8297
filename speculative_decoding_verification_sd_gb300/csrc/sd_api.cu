// sd_api.cu -- host side of the C ABI declared in include/sd.h: argument
// validation, workspace carving, launch-shape selection and kernel launches.
// No entry point allocates device memory or synchronises the stream.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <mutex>

#include "calib.h"
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
  sdk::RowStat* st_t;
  sdk::RowStat* st_d;
  float2* st_c;
  unsigned long long* rs;
  int* req_cnt;
  int* res_list;
  int* slice_cnt;
  int* ctrl;
};

// Workspace layout (each part 16-byte aligned):
// st_t | st_d | st_c | rs | req_cnt | res_list | slice_cnt | ctrl.
struct WsLayout {
  size_t st_t, st_d, st_c, rs, req_cnt, res_list, slice_cnt, ctrl, total;
};

WsLayout ws_layout(int bs, int k_max) {
  const size_t rows_t = static_cast<size_t>(bs) * (k_max + 1);
  const size_t rows_d = static_cast<size_t>(bs) * k_max;
  const size_t ib = align16(4 * static_cast<size_t>(bs));
  WsLayout L;
  L.st_t = 0;
  L.st_d = L.st_t + 16 * rows_t;
  L.st_c = L.st_d + 16 * rows_d;
  L.rs = L.st_c + 8 * sdk::kStatStride * rows_t;
  L.req_cnt = L.rs + 8 * sdk::kStatStride * static_cast<size_t>(bs);
  L.res_list = L.req_cnt + ib;
  L.slice_cnt = L.res_list + ib;
  L.ctrl = L.slice_cnt + ib;
  L.total = L.ctrl + 32;
  return L;
}

size_t verify_ws_bytes(int bs, int k_max) { return ws_layout(bs, k_max).total; }

VerifyWs carve(void* ws, int bs, int k_max) {
  const WsLayout L = ws_layout(bs, k_max);
  char* b = static_cast<char*>(ws);
  VerifyWs w;
  w.st_t = reinterpret_cast<sdk::RowStat*>(b + L.st_t);
  w.st_d = reinterpret_cast<sdk::RowStat*>(b + L.st_d);
  w.st_c = reinterpret_cast<float2*>(b + L.st_c);
  w.rs = reinterpret_cast<unsigned long long*>(b + L.rs);
  w.req_cnt = reinterpret_cast<int*>(b + L.req_cnt);
  w.res_list = reinterpret_cast<int*>(b + L.res_list);
  w.slice_cnt = reinterpret_cast<int*>(b + L.slice_cnt);
  w.ctrl = reinterpret_cast<int*>(b + L.ctrl);
  return w;
}

sd_status shape_for(int V, sd_dtype dt, int bs, const sd_launch_cfg* cfg, bool vec,
                    sdk::VerifyShape* shape) {
  const int elem = dt == SD_F32 ? 4 : 2;
  bool fits = false;
  if (note(sdk::choose_verify_shape(V, elem, bs, cfg, vec, shape, &fits)) != cudaSuccess)
    return SD_ERR_CUDA;
  return fits ? SD_OK : SD_ERR_UNSUPPORTED;
}

}  // namespace

namespace sdk {
size_t verify_ws_zero_offset(int bs, int k_max) { return ws_layout(bs, k_max).rs; }
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }
}  // namespace sdk

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
  if (mode != SD_MODE_ADAPTIVE && mode != SD_MODE_ALL_SLOTS && mode != SD_MODE_UNIFORM_K)
    return SD_ERR_INVALID_ARG;
  if (!draft_lens || !B_out || !num_verified || !cu_seqlens || !err_flag) return SD_ERR_INVALID_ARG;
  if (k_max > 0 && !slot_mask) return SD_ERR_INVALID_ARG;
  const int P = pow2ceil(k_max < 1 ? 1 : k_max);
  if (static_cast<long long>(pow2ceil(bs)) * P > SD_MAX_PLAN_SLOTS) return SD_ERR_UNSUPPORTED;
  int NPb = 0;
  if (mode != SD_MODE_ALL_SLOTS) {
    if (!conf_logits || !cost_table) return SD_ERR_INVALID_ARG;
    if (T < 1 || cost_len < 1) return SD_ERR_INVALID_ARG;
    if (T >= cost_len) return SD_ERR_SHAPE;
    if (mode == SD_MODE_ADAPTIVE && budget_conf) {
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

// Host checks shared by the two calibration calls; fills the shape fields.
static sd_status calib_shape(int bs, int k_max, sdk::CalibParams& p) {
  if (bs < 1 || k_max < 0) return SD_ERR_INVALID_ARG;
  if (k_max > SD_MAX_K) return SD_ERR_UNSUPPORTED;
  const int P = pow2ceil(k_max < 1 ? 1 : k_max);
  if (static_cast<long long>(pow2ceil(bs)) * P > SD_MAX_PLAN_SLOTS) return SD_ERR_UNSUPPORTED;
  p.bs = bs;
  p.k_max = k_max;
  p.P = P;
  p.NP = pow2ceil(bs) * P;
  return SD_OK;
}

sd_status sd_calibrate(const float* conf_logits, const int* draft_lens, const int* num_verified,
                       const int* accepted_len, int bs, int k_max, float lr, float* w, float* b,
                       int* err_flag, void* stream) {
  sdk::CalibParams p{};
  const sd_status st = calib_shape(bs, k_max, p);
  if (st != SD_OK) return st;
  if (!(std::isfinite(lr) && lr >= 0.0f)) return SD_ERR_INVALID_ARG;
  if (!draft_lens || !num_verified || !accepted_len || !err_flag) return SD_ERR_INVALID_ARG;
  if (k_max > 0 && (!conf_logits || !w || !b)) return SD_ERR_INVALID_ARG;
  if (k_max == 0) return SD_OK;
  p.conf = conf_logits;
  p.lens = draft_lens;
  p.nv = num_verified;
  p.acc = accepted_len;
  p.lr = lr;
  p.w = w;
  p.b = b;
  p.conf_out = nullptr;
  p.apply = 0;
  p.err = err_flag;
  return note(sdk::launch_calibrate(p, static_cast<cudaStream_t>(stream))) == cudaSuccess
             ? SD_OK
             : SD_ERR_CUDA;
}

sd_status sd_calibrate_apply(const float* conf_logits, const int* draft_lens, int bs, int k_max,
                             const float* w, const float* b, float* conf_out, int* err_flag,
                             void* stream) {
  sdk::CalibParams p{};
  const sd_status st = calib_shape(bs, k_max, p);
  if (st != SD_OK) return st;
  if (!draft_lens || !err_flag) return SD_ERR_INVALID_ARG;
  if (k_max > 0 && (!conf_logits || !w || !b || !conf_out)) return SD_ERR_INVALID_ARG;
  if (k_max == 0) return SD_OK;
  p.conf = conf_logits;
  p.lens = draft_lens;
  p.nv = nullptr;
  p.acc = nullptr;
  p.lr = 0.0f;
  p.w = const_cast<float*>(w);  // read only when apply = 1
  p.b = const_cast<float*>(b);
  p.conf_out = conf_out;
  p.apply = 1;
  p.err = err_flag;
  return note(sdk::launch_calibrate(p, static_cast<cudaStream_t>(stream))) == cudaSuccess
             ? SD_OK
             : SD_ERR_CUDA;
}

size_t sd_verify_workspace_bytes(int bs, int k_max) {
  if (bs < 1 || k_max < 0) return 0;
  return verify_ws_bytes(bs, k_max);
}

sd_status sd_verify_ex(const void* target_logits, const void* draft_logits, sd_dtype dt, int V,
                       const int* draft_ids, const float* uniforms, const float* temps,
                       const int* cu_seqlens, int bs, int k_max, int* accepted_len,
                       int* out_tokens, float* probs_out, int* err_flag, void* workspace,
                       size_t ws_bytes, const sd_launch_cfg* cfg, void* stream) {
  if (bs < 1 || k_max < 0) return SD_ERR_INVALID_ARG;
  if (k_max > SD_MAX_K || bs > SD_MAX_VERIFY_BS) return SD_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace)) return SD_ERR_INVALID_ARG;
  if (ws_bytes < verify_ws_bytes(bs, k_max)) return SD_ERR_SHAPE;
  if (dt != SD_F32 && dt != SD_BF16) return SD_ERR_INVALID_ARG;
  if (V < 1) return SD_ERR_INVALID_ARG;
  if (V > SD_MAX_V) return SD_ERR_UNSUPPORTED;
  if (!target_logits || !uniforms || !temps || !cu_seqlens || !err_flag || !accepted_len ||
      !out_tokens)
    return SD_ERR_INVALID_ARG;
  if (k_max > 0 && !draft_ids) return SD_ERR_INVALID_ARG;
  if (cfg && (cfg->threads < 0 || cfg->blocks < 0 || cfg->blocks_per_sm < 0))
    return SD_ERR_INVALID_ARG;
  const int elem = dt == SD_F32 ? 4 : 2;
  const bool vec = (static_cast<size_t>(V) * elem) % 16 == 0 && aligned16(target_logits) &&
                   (draft_logits == nullptr || aligned16(draft_logits));
  sdk::VerifyShape shape;
  sd_status st = shape_for(V, dt, bs, cfg, vec, &shape);
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
  p.accepted_len = accepted_len;
  p.out_tokens = out_tokens;
  p.probs_out = probs_out;
  p.err = err_flag;
  p.st_t = w.st_t;
  p.st_d = w.st_d;
  p.st_c = w.st_c;
  p.rs = w.rs;
  p.req_cnt = w.req_cnt;
  p.res_list = w.res_list;
  p.slice_cnt = w.slice_cnt;
  p.ctrl = w.ctrl;
  return note(sdk::launch_verify(p, elem, shape, static_cast<cudaStream_t>(stream))) ==
                 cudaSuccess
             ? SD_OK
             : SD_ERR_CUDA;
}

sd_status sd_verify(const void* target_logits, const void* draft_logits, sd_dtype dt, int V,
                    const int* draft_ids, const float* uniforms, const float* temps,
                    const int* cu_seqlens, int bs, int k_max, int* accepted_len, int* out_tokens,
                    float* probs_out, int* err_flag, void* workspace, size_t ws_bytes,
                    void* stream) {
  return sd_verify_ex(target_logits, draft_logits, dt, V, draft_ids, uniforms, temps, cu_seqlens,
                      bs, k_max, accepted_len, out_tokens, probs_out, err_flag, workspace,
                      ws_bytes, nullptr, stream);
}

sd_status sd_verify_launch_info(int V, sd_dtype dt, int bs, const sd_launch_cfg* req,
                                sd_launch_cfg* chosen, size_t* smem_bytes) {
  if (V < 1 || bs < 1 || (dt != SD_F32 && dt != SD_BF16) || !chosen) return SD_ERR_INVALID_ARG;
  if (bs > SD_MAX_VERIFY_BS || V > SD_MAX_V) return SD_ERR_UNSUPPORTED;
  const int elem = dt == SD_F32 ? 4 : 2;
  const bool vec = (static_cast<size_t>(V) * elem) % 16 == 0;
  sdk::VerifyShape shape;
  sd_status st = shape_for(V, dt, bs, req, vec, &shape);
  if (st != SD_OK) return st;
  chosen->threads = shape.threads;
  chosen->blocks = shape.blocks;
  chosen->blocks_per_sm = 0;
  chosen->reserved = 0;
  if (smem_bytes) *smem_bytes = shape.smem;
  return SD_OK;
}

}  // extern "C"
