/* sd.h -- C ABI of the GB300 verification-step library (libsdverify.so).
 *
 * One verification step of speculative decoding with adaptive verification,
 * in two stages that run entirely on one GPU:
 *
 *   sd_plan    planning stage: per-slot survival, global top-B, budget
 *              argmax against a step-cost table, varlen compaction.
 *   sd_verify  sampling stage: vocab-wide speculative rejection sampling on
 *              the compacted target/draft logits, one kernel.
 *
 * Sources (page title, section):
 *   [AV-blog]  fosworld blog "추측 디코딩과 vLLM 적응형 검증"
 *   [AV-page]  agentlenshq "vLLM DSpark을 활용한 적응형 검증(Adaptive Verification)"
 *   [DSD-page] discuss.pytorch.kr "DSD: Cohere의 하드웨어 인식 동적 추측 디코딩"
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *     caller allocates and frees every buffer; the library never allocates.
 *     Host-side state is limited to per-device launch settings applied once
 *     (shared-memory limits) and the per-thread last-error text.
 *   - Calls enqueue work on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and return without synchronising.  The return value
 *     reports host-side argument validation and launch errors only.
 *   - Problems found on the device (bad lengths, non-finite data, ...) are
 *     OR-ed into the caller's `err_flag` word (SD_DEV_ERR_* bits).  The word
 *     is sticky: the library never clears it; the caller zeroes it and reads
 *     it after any synchronisation.  A call that finds a device error still
 *     writes well-formed outputs (see each entry point), so later calls in
 *     the same stream never read out of bounds.
 *   - The planner's choice of B stays on the device; the host only ever
 *     knows the upper bound bs*(k_max+1) of target rows ([AV-blog] "켜는
 *     방법과 제약": the CPU knows only an upper bound of the lengths decided
 *     on the GPU), so every launch is sized from that bound.
 */
#ifndef SD_VERIFY_H_
#define SD_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SD_OK = 0,
  SD_ERR_INVALID_ARG = -1,  /* NULL pointer, negative size, unknown enum value */
  SD_ERR_SHAPE = -2,        /* sizes inconsistent with each other (e.g. T >= cost_len) */
  SD_ERR_UNSUPPORTED = -3,  /* valid but beyond this library's limits (SD_MAX_*) */
  SD_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed */
  SD_ERR_DEVICE_CHECK = -5  /* reserved for callers mapping err_flag to a status */
} sd_status;

typedef enum { SD_F32 = 0, SD_BF16 = 1 } sd_dtype;

typedef enum {
  SD_MODE_ADAPTIVE = 0,  /* budget chosen by the cost model ([AV-page] Budget Calculation) */
  SD_MODE_ALL_SLOTS = 1, /* every drafted slot verified (fixed-K speculative decoding) */
  SD_MODE_UNIFORM_K = 2  /* one draft length K for the batch, by goodput ([DSD-page]) */
} sd_mode;

/* Device error bits (OR-ed into *err_flag). */
#define SD_DEV_ERR_DRAFT_LENS 0x001      /* draft_lens[i] outside [0, k_max] */
#define SD_DEV_ERR_CONF 0x002            /* a confidence logit is NaN/inf */
#define SD_DEV_ERR_COST 0x004            /* a used cost entry is not finite and > 0 */
#define SD_DEV_ERR_CU_SEQLENS 0x008      /* cu_seqlens not a valid compaction */
#define SD_DEV_ERR_DRAFT_ID 0x010        /* a verified draft id outside [0, V) */
#define SD_DEV_ERR_TEMP 0x020            /* a temperature < 0 or not finite */
#define SD_DEV_ERR_UNIFORM 0x040         /* a uniform outside [0, 1) */
#define SD_DEV_ERR_LOGITS 0x080          /* a logit row holds NaN/+inf or no finite value */
#define SD_DEV_ERR_TIMEOUT 0x100         /* a bounded device-side wait gave up */
#define SD_DEV_ERR_OUTCOME 0x200         /* num_verified / accepted_len out of range (calibration) */

/* Limits of this library. */
#define SD_MAX_K 15            /* k_max <= 15: at most 16 query rows per request */
#define SD_MAX_PLAN_SLOTS 8192 /* pow2ceil(bs) * pow2ceil(k_max) <= 8192 for sd_plan */
#define SD_MAX_VERIFY_BS 4096  /* bs <= 4096 for sd_verify */
#define SD_MAX_V (1 << 20)     /* V <= 1,048,576 ... */
#define SD_MAX_ROW_BYTES (2 << 20) /* ... and V * element size <= 2 MiB (fp32: V <= 524,288) */

/* ------------------------------------------------------------------------
 * sd_plan -- planning stage of adaptive verification.
 *
 * Passages: [AV-blog] "동작" steps 1-3 (survival = product of per-position
 * acceptance estimates front to back; slots of all requests compete for the
 * budget and the chosen slots are always a contiguous prefix of each draft;
 * the number of slots maximises expected accepted tokens / expected step time
 * from a table profiled at start-up); [AV-page] "DSpark 신뢰도 스케줄링
 * 메커니즘" (Global Top-B Selection; Budget Calculation: one bonus token per
 * sampling request plus the survival of the B best slots, against the cost
 * of T non-draft plus B draft tokens; Execution Pipeline: the budget is sized
 * from the previous step's double-buffered confidences, the assignment runs
 * on the GPU without a host round trip) and "기술적 구현 및 CUDA Graphs"
 * (Cost Modeling: the cost curve is forced monotone; CUDA Graph Padding: the
 * table carries the graph-size staircase).
 *
 * Computes, with a_{i,j} = 1/(1+exp(-conf_{i,j})) and
 * s_{i,j} = prod_{m<=j} a_{i,m} (fp32):
 *   order all N = sum(draft_lens) slots by (s desc, packed index asc);
 *   cost'[n] = max(cost_table[1..n]);
 *   B* = smallest argmax over B in [0, min(N, cost_len-1-T)] of
 *        (bs + sum of the B largest s) / cost'[T+B];
 *   a slot is selected iff its rank < B*.
 *
 * SD_MODE_UNIFORM_K ([DSD-page] discuss.pytorch.kr "DSD feat. Cohere",
 * "동적 추측 디코딩(DSD)의 핵심 아이디어": one draft length for the whole
 * batch, chosen to maximise goodput = AL / ITL) computes instead, with
 * n(K) = sum_i min(K, draft_lens[i]):
 *   K* = smallest argmax over K in [0, max_i draft_lens[i]] with
 *        n(K) <= cost_len-1-T of
 *        (bs + sum_i sum_{j < min(K, draft_lens[i])} s_{i,j}) / cost'[T+n(K)];
 *   slot (i,j) is selected iff j < K*; B* = n(K*).  K* is max_i n_i.
 * The same survival s, cost' and error checks as the adaptive mode (the cost
 * entries T..T+min(N, cost_len-1-T) must be finite and > 0).
 *
 * Arguments
 *   conf_logits      [N] fp32, packed by request: slot (i,j) at
 *                    offset_i + j, offset = exclusive scan of draft_lens.
 *                    Unused (may be NULL) in SD_MODE_ALL_SLOTS.  Raw
 *                    confidence logits, or sd_calibrate_apply's calibrated
 *                    ones (the survival then uses the calibrated estimate).
 *   budget_conf      (SD_MODE_ADAPTIVE only; ignored in the other modes)
 *                    [N'] fp32 previous-step confidences packed by
 *                    budget_draft_lens [bs_budget], or NULL to size the budget
 *                    from conf_logits.  When given, B* is computed from them
 *                    (same T, R = bs) and clipped to min(N, cost_len-1-T);
 *                    the slots are still assigned by the current conf_logits.
 *   draft_lens       [bs] int32, 0 <= draft_lens[i] <= k_max.
 *   cost_table       [cost_len] fp32, cost of a step of n tokens at index n.
 *                    Unused (may be NULL) in SD_MODE_ALL_SLOTS.
 *   T                non-draft tokens of the step (>= 1 in the adaptive and
 *                    uniform-K modes).
 * Outputs
 *   B_out            [1] int32: B* (the number of verified draft slots).
 *   slot_mask        [bs*k_max] uint8: slot (i,j) at i*k_max+j, 1 = verified.
 *   num_verified     [bs] int32: n_i (a prefix of request i's draft).
 *   cu_seqlens       [bs+1] int32: cu[0] = 0, cu[i+1] = cu[i] + n_i + 1
 *                    (n_i verified drafts plus one target/bonus row).
 *   err_flag         [1] int32, sticky SD_DEV_ERR_* bits.  On a device error
 *                    the outputs describe B = 0 (n_i = 0, cu[i] = i).
 *   workspace        unused by this library (ws_bytes may be 0).
 * Limits: 1 <= bs, 0 <= k_max <= SD_MAX_K, pow2ceil(bs)*pow2ceil(k_max)
 * <= SD_MAX_PLAN_SLOTS (SD_ERR_UNSUPPORTED otherwise).  One CTA, one launch.
 * ---------------------------------------------------------------------- */
size_t sd_plan_workspace_bytes(int bs, int k_max);
sd_status sd_plan(const float* conf_logits, const float* budget_conf,
                  const int* budget_draft_lens, int bs_budget, const int* draft_lens,
                  int bs, int k_max, const float* cost_table, int cost_len, int T,
                  sd_mode mode, int* B_out, uint8_t* slot_mask, int* num_verified,
                  int* cu_seqlens, int* err_flag, void* workspace, size_t ws_bytes,
                  void* stream);

/* ------------------------------------------------------------------------
 * sd_verify -- sampling stage: speculative rejection sampling over the
 * vocabulary, one persistent kernel.
 *
 * Passages: [AV-blog] "추측 디코딩이란" (the target scores all drafted
 * positions in one pass; drafts are accepted front to back up to the first
 * mismatch, where the target's own token is inserted, so every step emits at
 * least one token), "속도, 메모리, 정확도에 주는 영향" row 정확도 (with the
 * original papers' rejection-sampling rule the output distribution equals the
 * target model's) and "참고 링크 / 논문" (Leviathan et al. 2023; Chen et al.
 * 2023); [AV-page] "현재 제한 사항" (logits are compacted after the forward).
 *
 * For request i with n_i = cu[i+1]-cu[i]-1 verified drafts, temperature
 * tau_i, target rows t_j (j = 0..n_i) and draft rows d_j (j < n_i):
 *   tau_i > 0: p_j = softmax(t_j/tau_i), q_j = softmax(d_j/tau_i);
 *              slot j accepted iff uniforms[i][j] * q_j(x_j) <= p_j(x_j)
 *              (p_j(x_j), q_j(x_j) rounded to fp32, the product in fp32).
 *   tau_i = 0: slot j accepted iff x_j == argmax t_j (lowest index on ties);
 *              draft rows are not read.
 *   a_i = first rejected slot, else n_i.
 *   final token y_i: tau_i = 0: argmax t_{a_i}; tau_i > 0: inverse CDF with
 *   u = uniforms[i][k_max] (smallest k with sum_{l<=k} w_l > u * sum w) over
 *   w = max(p_{a_i} - q_{a_i}, 0) after a rejection, or w = p_{n_i} (bonus)
 *   when every slot was accepted; if that residual has no positive mass,
 *   w = p_{a_i}.  The weights are summed in exact 64-bit fixed point (2^-56);
 *   an element heavier than 2^-10 of its row's largest weight is formed to
 *   about 1e-10 relative, the others in fp32.
 *   out_tokens[i] = (x_0 .. x_{a_i-1}, y_i, -1 ...), accepted_len[i] = a_i.
 *
 * Arguments
 *   target_logits  [rows_cap, V] fp32 or bf16, row-major, compacted: the row of
 *                  (i,j) is cu_seqlens[i]+j.  rows_cap >= bs*(k_max+1) is the
 *                  caller's allocation; only rows < cu_seqlens[bs] are read.
 *   draft_logits   [bs*k_max, V] same dtype.  Compacted: the row of (i,j) is
 *                  cu_seqlens[i]-i+j; with SD_VERIFY_DRAFT_PADDED (see
 *                  sd_verify_ex) it is i*k_max+j, the uncompacted layout a
 *                  draft forward over every drafted slot leaves.  Only rows of
 *                  requests with tau > 0 are read.  May be NULL if every
 *                  temperature is 0.
 *   dt, V          element type and vocabulary size.
 *   draft_ids      [bs*k_max] int32, indexed like the draft rows.
 *   uniforms       [bs, k_max+1] fp32 in [0,1): slot tests then the final draw.
 *   temps          [bs] fp32 >= 0.
 *   cu_seqlens     [bs+1] int32 from sd_plan (or the caller).
 * Outputs
 *   accepted_len   [bs] int32; out_tokens [bs, k_max+1] int32, -1 padded.
 *   probs_out      [bs*k_max, 2] fp32 or NULL: (p_j(x_j), q_j(x_j)) of every
 *                  verified slot of a tau > 0 request whose rows were read, at
 *                  the draft-row index (diagnostics; with early exit the slots
 *                  after the first rejection may be left untouched; entries of
 *                  greedy requests and of unverified slots are untouched).
 *   err_flag       [1] int32, sticky SD_DEV_ERR_* bits.  On SD_DEV_ERR_CU_SEQLENS
 *                  no logit is read and outputs are accepted_len = 0,
 *                  out_tokens = -1.  On SD_DEV_ERR_TIMEOUT every request's
 *                  outputs are accepted_len = 0, out_tokens = (0, -1, ...).
 *   workspace      device scratch of sd_verify_workspace_bytes(bs, k_max, V, dt)
 *                  bytes, 256-byte aligned: per-row statistics, per-chunk
 *                  sums of the final draws, per-request and per-slot
 *                  counters.  It must be zero-filled once before its
 *                  first use (e.g. cudaMemsetAsync); every call leaves the
 *                  counters at zero again.  One call at a time per workspace.
 * Layout: rows are staged with 16-byte bulk copies when V*elem is a multiple
 * of 16 and both logits base pointers are 16-byte aligned, read element by
 * element otherwise (same results, slower).
 * Limits: 1 <= bs <= SD_MAX_VERIFY_BS, 0 <= k_max <= SD_MAX_K,
 * V <= SD_MAX_V, V * elem <= SD_MAX_ROW_BYTES (SD_ERR_UNSUPPORTED otherwise).
 * ---------------------------------------------------------------------- */
size_t sd_verify_workspace_bytes(int bs, int k_max, int V, sd_dtype dt);

sd_status sd_verify(const void* target_logits, const void* draft_logits, sd_dtype dt, int V,
                    const int* draft_ids, const float* uniforms, const float* temps,
                    const int* cu_seqlens, int bs, int k_max, int* accepted_len,
                    int* out_tokens, float* probs_out, int* err_flag, void* workspace,
                    size_t ws_bytes, void* stream);

/* Options of sd_verify_ex.  Outputs never depend on `blocks`; the flags below
 * change what is read, never the accepted lengths or tokens. */
#define SD_VERIFY_EARLY_EXIT 0x1   /* skip the rows of slots after a request's known
                                      first rejection ([AV-blog] "뒤 자리 수락률이 급하게
                                      떨어지는 이유": later positions are rarely reached) */
#define SD_VERIFY_DRAFT_PADDED 0x2 /* draft rows and draft ids at i*k_max+j (uncompacted) */
#define SD_VERIFY_TEST_STALL 0x100 /* test hook: stream no row, so the end-of-call wait
                                      runs out (after wait_limit_us) and the time-out path runs */
typedef struct {
  int blocks;     /* persistent CTAs (0 = one per SM; capped at one per SM) */
  int flags;      /* SD_VERIFY_* bits */
  int wait_limit_us; /* microseconds a device-side wait may last before it gives up
                        (0 = the default, 1 s); the drain of in-flight copies at exit
                        is bounded separately */
  int reserved;   /* must be 0 */
} sd_launch_cfg;

/* sd_verify with options (cfg may be NULL: defaults). */
sd_status sd_verify_ex(const void* target_logits, const void* draft_logits, sd_dtype dt, int V,
                       const int* draft_ids, const float* uniforms, const float* temps,
                       const int* cu_seqlens, int bs, int k_max, int* accepted_len,
                       int* out_tokens, float* probs_out, int* err_flag, void* workspace,
                       size_t ws_bytes, const sd_launch_cfg* cfg, void* stream);

/* ------------------------------------------------------------------------
 * sd_verify_noalloc -- sd_verify without a caller workspace.  The pages have
 * no counterpart to this entry point.  It is for callers that cannot call
 * cudaMalloc around the verification step: a serving loop that reserved the
 * device's memory up front (weights, KV cache) and must not allocate while
 * it runs, or a host process whose allocator is owned by another framework.
 *
 * Same arguments and outputs as sd_verify, minus workspace/ws_bytes.  The
 * workspace is a file-scope device array of SD_NOALLOC_SCRATCH_BYTES inside
 * the library (static device memory, held by every device that loads the
 * library until the process exits; no allocation at call time).  Host code
 * cannot name that array directly: its device address is looked up with
 * cudaGetSymbolAddress, with the device current, on the first call on each
 * device -- make that first call before any stream capture -- and again on
 * every later call that is not being captured, so a call after a device
 * reset or from another context on the device uses the address that is
 * valid there.  A call under capture uses the address cached by the last
 * call outside capture on that device.
 * Each call first checks its arguments as sd_verify does, then clears, on
 * `stream`, the part of the scratch that must start at zero (the counters),
 * then runs the sampling kernel on it.  Calls that overlap in time on one
 * device share the scratch and race: issue them on one stream, or order them.
 * Errors: SD_ERR_UNSUPPORTED when sd_verify_workspace_bytes(bs, k_max, V, dt)
 * exceeds SD_NOALLOC_SCRATCH_BYTES (every batch sd_verify accepts fits at
 * V = 129280; at V = 2^20 bf16, about 1,900 requests at k_max = 7), with the
 * reason in sd_last_error_string(); SD_ERR_CUDA
 * when the lookup or the clear fails; otherwise as sd_verify.
 * ---------------------------------------------------------------------- */
#define SD_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB */

sd_status sd_verify_noalloc(const void* target_logits, const void* draft_logits, sd_dtype dt,
                            int V, const int* draft_ids, const float* uniforms,
                            const float* temps, const int* cu_seqlens, int bs, int k_max,
                            int* accepted_len, int* out_tokens, float* probs_out, int* err_flag,
                            void* stream);

/* Launch shape sd_verify_ex would use for (V, dt, bs) and `req` (NULL =
 * defaults) on the current device: CTAs in chosen->blocks, threads per CTA
 * and chunk buffers per CTA (two per streaming warp) in *threads and
 * *buffers, dynamic shared memory in
 * *smem_bytes (each output pointer may be NULL).  Host-only query. */
sd_status sd_verify_launch_info(int V, sd_dtype dt, int bs, const sd_launch_cfg* req,
                                sd_launch_cfg* chosen, int* threads, int* buffers,
                                size_t* smem_bytes);

/* ------------------------------------------------------------------------
 * sd_calibrate / sd_calibrate_apply -- online calibration of the
 * per-position acceptance estimate.
 *
 * Passage: [AV-blog] the table under "동작" (for model-based drafts the
 * per-position acceptance estimate comes from a small logistic model on the
 * draft's logits, corrected continuously with the verification results).
 * Model: a_{i,j} = sigmoid(w_j * c_{i,j} + b_j) of the confidence logit;
 * w = 1, b = 0 is the estimate sd_plan uses on raw logits.
 *
 * sd_calibrate: one gradient step from one step's outcomes.  Slot (i,j) was
 * observed when j < num_verified[i] and j <= accepted_len[i]; its label is 1
 * for j < accepted_len[i] (accepted) and 0 at j = accepted_len[i] (the first
 * rejection).  With m_j observed slots at position j and
 * e = sigmoid(w_j c + b_j) - label:
 *   w_j -= lr * (1/m_j) * sum e * c,   b_j -= lr * (1/m_j) * sum e
 * (the gradient of the mean logistic loss); positions with m_j = 0 keep
 * their parameters.  Sums in fp32 within a warp and fp64 across warps, in a
 * fixed order: repeated calls give identical results.
 *
 * sd_calibrate_apply: conf_out[slot] = fma(w_j, conf_logits[slot], b_j) for
 * every drafted slot, the calibrated logits to pass to sd_plan as
 * conf_logits (conf_out may equal conf_logits).
 *
 * Arguments
 *   conf_logits   [N] fp32 packed by draft_lens as for sd_plan.
 *   draft_lens    [bs] int32, 0 <= draft_lens[i] <= k_max.
 *   num_verified  [bs] int32, 0 <= num_verified[i] <= draft_lens[i] (sd_plan's).
 *   accepted_len  [bs] int32, 0 <= accepted_len[i] <= num_verified[i] (sd_verify's).
 *   lr            learning rate, finite and >= 0.
 *   w, b          [k_max] fp32 on the device, updated in place (sd_calibrate).
 *   conf_out      [N] fp32 (sd_calibrate_apply).
 *   err_flag      [1] int32, sticky bits: SD_DEV_ERR_DRAFT_LENS,
 *                 SD_DEV_ERR_OUTCOME, SD_DEV_ERR_CONF (a non-finite observed
 *                 logit).  On any of them nothing is updated (or written).
 * Limits as sd_plan: 1 <= bs, 0 <= k_max <= SD_MAX_K,
 * pow2ceil(bs)*pow2ceil(k_max) <= SD_MAX_PLAN_SLOTS.  k_max = 0 returns
 * SD_OK without a launch.  One CTA, one launch, asynchronous on `stream`.
 * ---------------------------------------------------------------------- */
sd_status sd_calibrate(const float* conf_logits, const int* draft_lens, const int* num_verified,
                       const int* accepted_len, int bs, int k_max, float lr, float* w, float* b,
                       int* err_flag, void* stream);
sd_status sd_calibrate_apply(const float* conf_logits, const int* draft_lens, int bs, int k_max,
                             const float* w, const float* b, float* conf_out, int* err_flag,
                             void* stream);

const char* sd_status_string(sd_status s);

/* The reason for the last status other than SD_OK that an entry point
 * returned on the calling host thread: the CUDA error's name and text for
 * SD_ERR_CUDA, otherwise the failed check ("no error" if none).  Every entry
 * point resets it to "no error" when it starts, so the text always belongs to
 * the thread's latest call.  The pointer stays valid until that thread's next
 * call. */
const char* sd_last_error_string(void);

int sd_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SD_VERIFY_H_ */
