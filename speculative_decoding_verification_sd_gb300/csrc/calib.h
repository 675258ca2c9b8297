// calib.h -- parameter block and launch helper of the online calibration of
// the per-position acceptance model, shared between the host API
// (sd_api.cu) and its kernels (in plan_kernel.cu, next to the planner whose
// length and offset helpers they use).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "sd.h"

namespace sdk {

struct CalibParams {
  const float* conf;     // [N] packed by draft_lens
  const int* lens;       // [bs] draft_lens
  const int* nv;         // [bs] num_verified (update only)
  const int* acc;        // [bs] accepted_len (update only)
  int bs;
  int k_max;
  int P;                 // pow2ceil(max(k_max, 1))
  int NP;                // pow2ceil(bs) * P
  float lr;              // update only
  float* w;              // [k_max] in/out (update), in (apply)
  float* b;              // [k_max]
  float* conf_out;       // [N] apply only: w_j * c + b_j
  int apply;             // 0: one update step, 1: write the calibrated logits
  int* err;
};

cudaError_t launch_calibrate(const CalibParams& p, cudaStream_t s);

}  // namespace sdk
