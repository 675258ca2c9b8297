// sd_api.cu -- host side of the C ABI declared in include/sd.h: argument
// validation, workspace carving, launch-shape selection and kernel launches.
// No entry point allocates device memory or synchronises the stream.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
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

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace sdk {

void set_last_error(const char* msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }
void clear_last_error() { set_last_error("no error"); }

// Records why a call is refused; returns the status unchanged.
sd_status refuse(sd_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

// 2^(j/16), j = 0..15, each split into two floats (hi + lo) -- the table of
// the sampler's precise exponent.
static void exp_table(float2* tab) {
  for (int j = 0; j < 16; ++j) {
    const double t = std::exp2(static_cast<double>(j) / 16.0);
    const float hi = static_cast<float>(t);
    tab[j] = make_float2(hi, static_cast<float>(t - static_cast<double>(hi)));
  }
}

sd_status verify_setup(const void* target_logits, const void* draft_logits, sd_dtype dt, int V,
                       const int* draft_ids, const float* uniforms, const float* temps,
                       const int* cu_seqlens, int bs, int k_max, int* accepted_len,
                       int* out_tokens, float* probs_out, int* err_flag,
                       const sd_launch_cfg* cfg, VerifyCall* call) {
  if (bs < 1 || k_max < 0) return refuse(SD_ERR_INVALID_ARG, "bs=%d, k_max=%d: need bs >= 1, k_max >= 0", bs, k_max);
  if (k_max > SD_MAX_K || bs > SD_MAX_VERIFY_BS)
    return refuse(SD_ERR_UNSUPPORTED, "bs=%d, k_max=%d beyond SD_MAX_VERIFY_BS=%d / SD_MAX_K=%d", bs,
                  k_max, SD_MAX_VERIFY_BS, SD_MAX_K);
  if (dt != SD_F32 && dt != SD_BF16) return refuse(SD_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dt));
  if (V < 1) return refuse(SD_ERR_INVALID_ARG, "V=%d < 1", V);
  const int elem = dt == SD_F32 ? 4 : 2;
  if (V > SD_MAX_V || static_cast<size_t>(V) * elem > static_cast<size_t>(SD_MAX_ROW_BYTES))
    return refuse(SD_ERR_UNSUPPORTED, "V=%d (%d-byte elements) beyond SD_MAX_V / SD_MAX_ROW_BYTES", V, elem);
  if (!target_logits || !uniforms || !temps || !cu_seqlens || !err_flag || !accepted_len ||
      !out_tokens)
    return refuse(SD_ERR_INVALID_ARG, "a required pointer is NULL");
  if (k_max > 0 && !draft_ids) return refuse(SD_ERR_INVALID_ARG, "draft_ids is NULL");
  int blocks = 0, flags = 0, wait_us = 0;
  if (cfg) {
    if (cfg->blocks < 0 || cfg->wait_limit_us < 0 || cfg->reserved != 0)
      return refuse(SD_ERR_INVALID_ARG, "sd_launch_cfg: negative field or reserved != 0");
    if (cfg->flags & ~(SD_VERIFY_EARLY_EXIT | SD_VERIFY_DRAFT_PADDED | SD_VERIFY_TEST_STALL))
      return refuse(SD_ERR_INVALID_ARG, "sd_launch_cfg: unknown flag bits 0x%x", cfg->flags);
    blocks = cfg->blocks;
    flags = cfg->flags;
    wait_us = cfg->wait_limit_us;
  }
  call->vec = (static_cast<size_t>(V) * elem) % 16 == 0 && aligned16(target_logits) &&
              (draft_logits == nullptr || aligned16(draft_logits));
  call->blocks = blocks;
  const SamplerWs L = sampler_ws_layout(bs, k_max, V, elem);
  call->elem = elem;
  call->ws_need = L.total;
  call->zero_off = L.zero;
  SamplerParams& p = call->p;
  p = SamplerParams{};
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
  p.flags = flags;
  p.wait_ns = 1000ull * static_cast<uint64_t>(wait_us > 0 ? wait_us : 1000000);
  sampler_geometry(V, elem, &p.slice, &p.ncr, &p.ncd);
  exp_table(p.exp_tab);
  return SD_OK;
}

sd_status verify_shape(VerifyCall* call) {
  bool fits = false;
  if (note(choose_sampler_shape(call->p.V, call->elem, call->p.bs, call->blocks, call->vec,
                                &call->shape, &fits)) != cudaSuccess)
    return SD_ERR_CUDA;
  if (!fits)
    return refuse(SD_ERR_UNSUPPORTED, "bs=%d: the sampler's shared memory does not fit", call->p.bs);
  return SD_OK;
}

void verify_bind(VerifyCall* call, void* workspace) {
  const SamplerWs L = sampler_ws_layout(call->p.bs, call->p.k_max, call->p.V, call->elem);
  char* b = static_cast<char*>(workspace);
  SamplerParams& p = call->p;
  p.rst = reinterpret_cast<RowStat*>(b + L.rst);
  p.rs = reinterpret_cast<unsigned long long*>(b + L.rs);
  p.pc = reinterpret_cast<int*>(b + L.pc);
  p.st = reinterpret_cast<int*>(b + L.st);
  p.dl = reinterpret_cast<int*>(b + L.dl);
  p.dpc = reinterpret_cast<int*>(b + L.dpc);
  p.ctrl = reinterpret_cast<int*>(b + L.ctrl);
}

sd_status verify_launch(const VerifyCall& call, void* stream) {
  return note(launch_sampler(call.p, call.elem, call.shape, static_cast<cudaStream_t>(stream))) ==
                 cudaSuccess
             ? SD_OK
             : SD_ERR_CUDA;
}

}  // namespace sdk

extern "C" {

int sd_abi_version(void) { return 2; }

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

// Host checks of sd_plan; records the reason of a refusal.
static sd_status plan_checks(const float* conf_logits, const float* budget_conf,
                             const int* budget_draft_lens, int bs_budget, const int* draft_lens,
                             int bs, int k_max, const float* cost_table, int cost_len, int T,
                             sd_mode mode, const int* B_out, const uint8_t* slot_mask,
                             const int* num_verified, const int* cu_seqlens, const int* err_flag) {
  using sdk::refuse;
  if (bs < 1 || k_max < 0) return refuse(SD_ERR_INVALID_ARG, "bs=%d, k_max=%d", bs, k_max);
  if (k_max > SD_MAX_K) return refuse(SD_ERR_UNSUPPORTED, "k_max=%d > SD_MAX_K", k_max);
  if (mode != SD_MODE_ADAPTIVE && mode != SD_MODE_ALL_SLOTS && mode != SD_MODE_UNIFORM_K)
    return refuse(SD_ERR_INVALID_ARG, "unknown mode %d", static_cast<int>(mode));
  if (!draft_lens || !B_out || !num_verified || !cu_seqlens || !err_flag)
    return refuse(SD_ERR_INVALID_ARG, "a required pointer is NULL");
  if (k_max > 0 && !slot_mask) return refuse(SD_ERR_INVALID_ARG, "slot_mask is NULL");
  const int P = pow2ceil(k_max < 1 ? 1 : k_max);
  if (static_cast<long long>(pow2ceil(bs)) * P > SD_MAX_PLAN_SLOTS)
    return refuse(SD_ERR_UNSUPPORTED, "pow2ceil(bs)*pow2ceil(k_max) > SD_MAX_PLAN_SLOTS");
  if (mode != SD_MODE_ALL_SLOTS) {
    if (!conf_logits || !cost_table) return refuse(SD_ERR_INVALID_ARG, "conf_logits or cost_table is NULL");
    if (T < 1 || cost_len < 1) return refuse(SD_ERR_INVALID_ARG, "T=%d, cost_len=%d", T, cost_len);
    if (T >= cost_len) return refuse(SD_ERR_SHAPE, "T=%d >= cost_len=%d", T, cost_len);
    if (mode == SD_MODE_ADAPTIVE && budget_conf) {
      if (!budget_draft_lens || bs_budget < 1)
        return refuse(SD_ERR_INVALID_ARG, "budget_conf without budget_draft_lens / bs_budget");
      if (static_cast<long long>(pow2ceil(bs_budget)) * P > SD_MAX_PLAN_SLOTS)
        return refuse(SD_ERR_UNSUPPORTED, "budget set beyond SD_MAX_PLAN_SLOTS");
    }
  }
  return SD_OK;
}

sd_status sd_plan(const float* conf_logits, const float* budget_conf, const int* budget_draft_lens,
                  int bs_budget, const int* draft_lens, int bs, int k_max, const float* cost_table,
                  int cost_len, int T, sd_mode mode, int* B_out, uint8_t* slot_mask,
                  int* num_verified, int* cu_seqlens, int* err_flag, void* workspace,
                  size_t ws_bytes, void* stream) {
  (void)workspace;
  (void)ws_bytes;
  sdk::clear_last_error();
  const sd_status st = plan_checks(conf_logits, budget_conf, budget_draft_lens, bs_budget,
                                   draft_lens, bs, k_max, cost_table, cost_len, T, mode, B_out,
                                   slot_mask, num_verified, cu_seqlens, err_flag);
  if (st != SD_OK) return st;
  const int P = pow2ceil(k_max < 1 ? 1 : k_max);
  const int NPb = (mode == SD_MODE_ADAPTIVE && budget_conf) ? pow2ceil(bs_budget) * P : 0;
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
  sdk::clear_last_error();
  if (bs < 1 || k_max < 0) return sdk::refuse(SD_ERR_INVALID_ARG, "bs=%d, k_max=%d", bs, k_max);
  if (k_max > SD_MAX_K) return sdk::refuse(SD_ERR_UNSUPPORTED, "k_max=%d > SD_MAX_K", k_max);
  const int P = pow2ceil(k_max < 1 ? 1 : k_max);
  if (static_cast<long long>(pow2ceil(bs)) * P > SD_MAX_PLAN_SLOTS)
    return sdk::refuse(SD_ERR_UNSUPPORTED, "pow2ceil(bs)*pow2ceil(k_max) > SD_MAX_PLAN_SLOTS");
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
  if (!(std::isfinite(lr) && lr >= 0.0f)) return sdk::refuse(SD_ERR_INVALID_ARG, "lr not finite or < 0");
  if (!draft_lens || !num_verified || !accepted_len || !err_flag)
    return sdk::refuse(SD_ERR_INVALID_ARG, "a required pointer is NULL");
  if (k_max > 0 && (!conf_logits || !w || !b))
    return sdk::refuse(SD_ERR_INVALID_ARG, "conf_logits, w or b is NULL");
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
  if (!draft_lens || !err_flag) return sdk::refuse(SD_ERR_INVALID_ARG, "a required pointer is NULL");
  if (k_max > 0 && (!conf_logits || !w || !b || !conf_out))
    return sdk::refuse(SD_ERR_INVALID_ARG, "conf_logits, w, b or conf_out is NULL");
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

size_t sd_verify_workspace_bytes(int bs, int k_max, int V, sd_dtype dt) {
  if (bs < 1 || k_max < 0 || V < 1 || (dt != SD_F32 && dt != SD_BF16)) return 0;
  return sdk::sampler_ws_layout(bs, k_max, V, dt == SD_F32 ? 4 : 2).total;
}

sd_status sd_verify_ex(const void* target_logits, const void* draft_logits, sd_dtype dt, int V,
                       const int* draft_ids, const float* uniforms, const float* temps,
                       const int* cu_seqlens, int bs, int k_max, int* accepted_len,
                       int* out_tokens, float* probs_out, int* err_flag, void* workspace,
                       size_t ws_bytes, const sd_launch_cfg* cfg, void* stream) {
  sdk::clear_last_error();
  sdk::VerifyCall call;
  const sd_status st = sdk::verify_setup(target_logits, draft_logits, dt, V, draft_ids, uniforms,
                                         temps, cu_seqlens, bs, k_max, accepted_len, out_tokens,
                                         probs_out, err_flag, cfg, &call);
  if (st != SD_OK) return st;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return sdk::refuse(SD_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
  if (ws_bytes < call.ws_need)
    return sdk::refuse(SD_ERR_SHAPE, "ws_bytes=%zu < %zu", ws_bytes, call.ws_need);
  const sd_status sh = sdk::verify_shape(&call);
  if (sh != SD_OK) return sh;
  sdk::verify_bind(&call, workspace);
  return sdk::verify_launch(call, stream);
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
                                sd_launch_cfg* chosen, int* threads, int* buffers,
                                size_t* smem_bytes) {
  sdk::clear_last_error();
  if (V < 1 || bs < 1 || (dt != SD_F32 && dt != SD_BF16) || !chosen)
    return sdk::refuse(SD_ERR_INVALID_ARG, "invalid V, bs, dtype or NULL output");
  const int elem = dt == SD_F32 ? 4 : 2;
  if (bs > SD_MAX_VERIFY_BS || V > SD_MAX_V ||
      static_cast<size_t>(V) * elem > static_cast<size_t>(SD_MAX_ROW_BYTES))
    return sdk::refuse(SD_ERR_UNSUPPORTED, "beyond this library's limits");
  if (req && (req->blocks < 0 || req->reserved != 0))
    return sdk::refuse(SD_ERR_INVALID_ARG, "sd_launch_cfg: negative field or reserved != 0");
  const bool vec = (static_cast<size_t>(V) * elem) % 16 == 0;
  sdk::SamplerShape shape;
  bool fits = false;
  if (note(sdk::choose_sampler_shape(V, elem, bs, req ? req->blocks : 0, vec, &shape, &fits)) !=
      cudaSuccess)
    return SD_ERR_CUDA;
  if (!fits) return sdk::refuse(SD_ERR_UNSUPPORTED, "the sampler's shared memory does not fit");
  chosen->blocks = shape.blocks;
  chosen->flags = req ? req->flags : 0;
  chosen->wait_limit_us = req ? req->wait_limit_us : 0;
  chosen->reserved = 0;
  if (threads) *threads = shape.threads;
  if (buffers) *buffers = shape.nbuf;
  if (smem_bytes) *smem_bytes = shape.smem;
  return SD_OK;
}

}  // extern "C"
