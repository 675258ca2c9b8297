// sd_internal.h -- parameter blocks and launch helpers shared between the
// host API (sd_api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/sd.h"

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
  float* probs_out;
  int* err;
  uint8_t* ws_accept;  // [rows_cap]
  int* ws_cand;        // [rows_cap]
  int* ws_status;      // [1] 0 = rows pass ran on valid cu_seqlens
  // launch shape
  int C;            // cluster size
  int S;            // stages
  int SL;           // vocabulary slice per CTA (elements, multiple of 64)
  int stage_bytes;  // 2 * SL * elem
};

struct VerifyShape {
  int C, S, SL, threads, clusters;
  size_t smem;
  bool bulk;
};

// Chooses (threads, C, S, SL) for (V, dtype, bs) on the current device,
// honouring a user request; *fits = false when no shape fits.
cudaError_t choose_verify_shape(int V, int elem, int bs, const sd_launch_cfg* req, bool bulk,
                                VerifyShape* out, bool* fits);
cudaError_t launch_verify_rows(const VerifyParams& p, int elem, const VerifyShape& shape,
                               cudaStream_t s);
cudaError_t launch_verify_finalize(const int* draft_ids, const int* cu, int bs, int k_max,
                                   int* accepted_len, int* out_tokens, int* err,
                                   const uint8_t* ws_accept, const int* ws_cand,
                                   const int* ws_status, cudaStream_t s);
cudaError_t max_active_clusters(int elem, const VerifyShape& shape, int* n);

}  // namespace sdk
