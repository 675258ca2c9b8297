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
// The sampling kernel streams every logit row with all its streaming warps:
// warp w takes bytes [w * slice, (w + 1) * slice) of the row, in chunks of
// kSegBytes (one bulk copy each).  A final draw's row(s) are taken in
// chunks of kSubBytes per row (a target and a draft chunk share a buffer).
// kSubBytes is a multiple of 512: a lane's share of a draw chunk is a whole
// number of 16-byte units.  Sixteen warps, each with two 6 KB buffers,
// hide more latency than twelve with 8 KB ones (measured).
constexpr int kSegBytes = 6144;
constexpr int kSubBytes = kSegBytes / 2;
constexpr int kMaxRowBytes = 2 << 20;          // V * elem <= 2 MiB
constexpr int kSamplerWarps = 16;              // streaming warps per CTA (plus one scheduler warp)
constexpr int kFinishWarps = 1;                // warps that finish the CTA's units (rows, draws)

// Statistics of one logit row, 32 bytes.  M = maximum, 1/Z as a
// double-float (izh + izl) with Z = sum over the row of
// 2^((l - M) * log2(e) / tau) (sampling rows), lx = the logit at the
// slot's draft token, amax = lowest argmax (greedy rows), bad = the row
// holds NaN or +inf or no finite value.
struct __align__(16) RowStat {
  float M, izh, izl, lx;
  int amax, bad, r0, r1;
};

// Control words of one call (all zero between calls).
enum {
  kCtlRow = 0,        // row units claimed
  kCtlCtas = 1,       // CTAs finished
  kCtlDraws = 2,      // final draws listed
  kCtlDrawTaken = 3,  // listed draws claimed by a CTA
  kCtlReqDone = 4,    // requests whose outputs are complete
  kCtlStop = 5,       // a bounded wait gave up in this call
  kCtlWords = 8
};

// Bits of sd_launch_cfg.flags the kernel reads (include/sd.h).
constexpr int kFlagEarlyExit = SD_VERIFY_EARLY_EXIT;
constexpr int kFlagDraftPadded = SD_VERIFY_DRAFT_PADDED;
constexpr int kFlagTestStall = SD_VERIFY_TEST_STALL;

struct SamplerParams {
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
  int flags;
  uint64_t wait_ns;  // how long a device-side wait may last before it gives up
  int slice;         // bytes of a row per streaming warp (a multiple of 16)
  int ncr;           // row chunks per warp (at most)
  int ncd;           // draw chunks per warp (at most)
  // workspace
  RowStat* rst;               // [bs*(k_max+1) + bs*k_max]: target rows, then draft rows
  unsigned long long* rs;     // [2*bs][kSamplerWarps][ncd] chunk sums of each listed draw
  int* pc;                    // [bs*(k_max+1)] per pair: rows counted, plus
                              //   skipped rows << 16                           (zero between calls)
  int* st;                    // [bs] slot decisions per request               (zero between calls)
  int* dl;                    // [2*bs] listed draws                           (zero between calls)
  int* dpc;                   // [2*bs] parts of each listed draw summed       (zero between calls)
  int* ctrl;                  // [kCtlWords]                                   (zero between calls)
  float2 exp_tab[16];         // 2^(j/16) as (hi, lo) pairs
};

// Workspace layout of the sampling kernel (each part 256-byte aligned); the
// parts from `zero` on must be zero before a call and are left zero by it.
struct SamplerWs {
  size_t rst, rs, zero, pc, st, dl, dpc, ctrl, total;
};
SamplerWs sampler_ws_layout(int bs, int k_max, int V, int elem);
// Per-warp slice of a row and the chunk counts it gives.
void sampler_geometry(int V, int elem, int* slice, int* ncr, int* ncd);

struct SamplerShape {
  int blocks, threads, nbuf;
  size_t smem;
  bool vec;
};

// Launch shape for (V, elem, bs) on the current device; *fits = false when the
// shared memory does not fit.  `blocks` = 0 asks for one CTA per SM.
cudaError_t choose_sampler_shape(int V, int elem, int bs, int blocks, bool vec,
                                 SamplerShape* out, bool* fits);
cudaError_t launch_sampler(const SamplerParams& p, int elem, const SamplerShape& shape,
                           cudaStream_t s);

// One sd_verify call after its host-side checks: kernel parameters (the
// workspace pointers still unset), launch shape, workspace size and the
// offset of its part that must be zero before a call.
struct VerifyCall {
  SamplerParams p;
  SamplerShape shape;
  int elem, blocks;
  bool vec;
  size_t ws_need, zero_off;
};

// Host-side checks and parameters of a sampling call (sd_verify_ex's
// arguments minus the workspace), with no CUDA call; records the reason of a
// refusal.  verify_shape then picks the launch shape on the current device.
sd_status verify_setup(const void* target_logits, const void* draft_logits, sd_dtype dt, int V,
                       const int* draft_ids, const float* uniforms, const float* temps,
                       const int* cu_seqlens, int bs, int k_max, int* accepted_len,
                       int* out_tokens, float* probs_out, int* err_flag,
                       const sd_launch_cfg* cfg, VerifyCall* call);
sd_status verify_shape(VerifyCall* call);
// Points the call's workspace parts into `workspace` (call->ws_need bytes).
void verify_bind(VerifyCall* call, void* workspace);
sd_status verify_launch(const VerifyCall& call, void* stream);

// Sets / clears the message sd_last_error_string() returns on this host thread.
void set_last_error(const char* msg);
void clear_last_error();
// Records why a call is refused (printf format); returns `st` unchanged.
sd_status refuse(sd_status st, const char* fmt, ...);

}  // namespace sdk
