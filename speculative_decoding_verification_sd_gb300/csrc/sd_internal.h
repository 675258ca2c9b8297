// sd_internal.h -- parameter blocks and launch helpers shared between the
// host API (sd_api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "sd.h"

namespace sdk {

// ---------------------------------------------------------------- planner
struct PlanParams {
  const float* conf;
  const float* budget_conf;
  const int* budget_lens;
  int bs_budget;
  const int* lens;
  int bs;
  int k_max;
  const float* cost;
  int cost_len;
  int T;
  int mode;
  int P;    // pow2ceil(max(k_max, 1)): slots reserved per request in the sort
  int NP;   // pow2ceil(bs) * P
  int NPb;  // pow2ceil(bs_budget) * P, or 0
  int* B_out;
  uint8_t* mask;
  int* num_verified;
  int* cu;
  int* err;
};

constexpr int kPlanThreads = 1024;
size_t plan_smem_bytes(const PlanParams& p);
cudaError_t launch_plan(const PlanParams& p, cudaStream_t s);

// ---------------------------------------------------------------- sampler
// Statistics of one logit row, 16 bytes: m = max logit, z = sum over the row
// of 2^((l - m) * log2(e) / tau) (tau > 0), lx = logit at the slot's draft
// token, amax = lowest index of the maximum (tau = 0; -1 if the row is bad).
struct __align__(16) RowStat {
  float m, z, lx;
  int amax;
};

struct VerifyParams {
  const void* target;
  const void* draft;
  int V;
  const int* draft_ids;
  const float* uniforms;
  const float* temps;
  const int* cu;
  int bs;
  int k_max;
  int* accepted_len;
  int* out_tokens;
  float* probs_out;
  int* err;
  RowStat* st_t;  // [bs*(k_max+1)]
  RowStat* st_d;  // [bs*k_max]
  float2* st_c;   // [bs*(k_max+1)][kStatStride] per-chunk (max, scaled sum) of target rows
  unsigned long long* rs;  // [bs][kStatStride] per-chunk residual sums (2^56 fixed point)
                           //   of the listed residual draws; zero between calls
  int* req_cnt;   // [bs]   rows finished per request; zero between calls
  int* res_list;  // [bs]   listed residual draws, 1 + (request << 4 | slot); zero between calls
  int* slice_cnt; // [bs]   slices finished per listed residual draw; zero between calls
  int* ctrl;      // [8]    rows handed out, CTAs finished, residual draws listed,
                  //        residual draws claimed, sampling requests decided;
                  //        zero between calls
};

// Statistics chunks: a row is cut into at most kStatStride chunks whose
// softmax statistics (target rows) or residual sums (listed draws) are kept,
// so a final draw reads back one chunk instead of its row.
constexpr int kStatStride = 128;

struct VerifyShape {
  int threads, blocks;
  size_t smem;
  bool vec;
};

// Chooses the launch of the sampling kernel for (V, dtype, bs) on the current
// device, honouring a user request; *fits = false when nothing fits.
cudaError_t choose_verify_shape(int V, int elem, int bs, const sd_launch_cfg* req, bool vec,
                                VerifyShape* out, bool* fits);
cudaError_t launch_verify(const VerifyParams& p, int elem, const VerifyShape& shape,
                          cudaStream_t s);

// Offset of the first workspace byte that must be zero before a call (the
// residual sums and every counter sit in [offset, sd_verify_workspace_bytes)).
size_t verify_ws_zero_offset(int bs, int k_max);
// Sets the message sd_last_error_string() returns on this host thread.
void set_last_error(const char* msg);

}  // namespace sdk
