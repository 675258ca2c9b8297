// plan_kernel.cu -- K1: the planning stage of adaptive verification in one
// CTA of 1024 threads, everything resident in shared memory.
//
//   survival   a = sigmoid(conf), s_j = s_{j-1} * a_j front to back
//              [fosworld blog "추측 디코딩과 vLLM 적응형 검증", "동작" step 1]
//   top-B      all slots ranked by (s desc, packed index asc); each request's
//              survival list is already sorted, so the sort is a merge of
//              pre-sorted runs (merge path, Odeh et al. 2012)
//              ["동작" step 2; agentlenshq "vLLM DSpark을 활용한 적응형 검증",
//               "DSpark 신뢰도 스케줄링 메커니즘" / Global Top-B Selection]
//   budget     B* = smallest argmax_B (R + sum of the B best s) / cost'[T+B],
//              cost' = running max of the table (forced monotone)
//              ["동작" step 3; same page, Budget Calculation, and
//               "기술적 구현 및 CUDA Graphs" / Cost Modeling, CUDA Graph Padding]
//   compaction slot mask, n_i and cu_seqlens (n_i drafts + 1 row per request)
//              [same page, Execution Pipeline: assignment on the GPU without a
//               host round trip]
//
// The prefix sums of the ranked survival values are exact integer sums of
// the fp32 keys scaled by 2^48 (at most 8192 terms <= 1, so they fit in 62
// bits); only the final division by the cost is rounded.
#include <atomic>
#include <mutex>

#include "sd_device.cuh"
#include "sd_internal.h"

namespace sdk {

namespace {

constexpr int NT = kPlanThreads;
constexpr int NW = NT / 32;
constexpr unsigned long long kSentinel = ~0ull;
constexpr float kFix = 281474976710656.0f;  // 2^48

struct PlanShared {
  unsigned long long red_u64[NW];
  float red_f32[NW];
  int red_i32[NW];
  int err;
  int B;
  unsigned long long scan_total;
};

__device__ unsigned long long block_excl_scan_u64(unsigned long long v, PlanShared& sh,
                                                  unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned long long t = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) sh.red_u64[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = sh.red_u64[lane];
    unsigned long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      unsigned long long t = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += t;
    }
    sh.red_u64[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) sh.scan_total = wi;
  }
  __syncthreads();
  const unsigned long long r = sh.red_u64[warp] + inc - v;
  if (total) *total = sh.scan_total;
  __syncthreads();
  return r;
}

__device__ int block_excl_scan_i32(int v, PlanShared& sh, int* total) {
  unsigned long long t;
  unsigned long long r = block_excl_scan_u64(static_cast<unsigned long long>(v), sh, &t);
  if (total) *total = static_cast<int>(t);
  return static_cast<int>(r);
}

__device__ unsigned long long block_max_u64(unsigned long long v, PlanShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max_u64(v);
  if (lane == 0) sh.red_u64[warp] = v;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = warp_max_u64(sh.red_u64[lane]);
    if (lane == 0) sh.scan_total = w;
  }
  __syncthreads();
  const unsigned long long r = sh.scan_total;
  __syncthreads();
  return r;
}

__device__ float block_max_f32(float v, PlanShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  if (lane == 0) sh.red_f32[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float w = warp_max(sh.red_f32[lane]);
    if (lane == 0) sh.red_f32[0] = w;
  }
  __syncthreads();
  const float r = sh.red_f32[0];
  __syncthreads();
  return r;
}

// Exclusive running maximum over the threads' values in thread order.
__device__ float block_excl_max_scan(float v, PlanShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc = fmaxf(inc, t);
  }
  if (lane == 31) sh.red_f32[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    float wi = sh.red_f32[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi = fmaxf(wi, t);
    }
    const float ex = __shfl_up_sync(kFull, wi, 1);
    sh.red_f32[lane] = lane == 0 ? -INFINITY : ex;
  }
  __syncthreads();
  const float lane_ex_raw = __shfl_up_sync(kFull, inc, 1);
  const float lane_ex = lane == 0 ? -INFINITY : lane_ex_raw;
  const float r = fmaxf(sh.red_f32[warp], lane_ex);
  __syncthreads();
  return r;
}

// Loads draft lengths, checks them and forms packed offsets off[0..n].
// Returns the total slot count N.
__device__ int load_lengths(const int* lens_g, int n, int k_max, int* lens, int* off,
                            PlanShared& sh) {
  const int chunk = (n + NT - 1) / NT;
  const int beg = min(n, static_cast<int>(threadIdx.x) * chunk);
  const int end = min(n, beg + chunk);
  int local = 0, bad = 0;
  for (int i = beg; i < end; ++i) {
    int k = lens_g[i];
    if (k < 0 || k > k_max) { bad = 1; k = 0; }
    lens[i] = k;
    local += k;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) sh.err |= SD_DEV_ERR_DRAFT_LENS;
  int total;
  int run = block_excl_scan_i32(local, sh, &total);
  for (int i = beg; i < end; ++i) {
    off[i] = run;
    run += lens[i];
  }
  if (threadIdx.x == 0) off[n] = total;
  __syncthreads();
  return total;
}

// Sort keys of n requests, P slots each: high word = ~bits(s) (s >= 0, so a
// larger survival gives a smaller key), low word = i*P + j (packed order).
// Unused slots hold the sentinel, which sorts last.  The N packed confidence
// logits are first copied to shared memory by the whole block (coalesced),
// then each thread runs the short survival product of its requests.
__device__ void build_keys(const float* conf, const int* lens, const int* off, int n, int P,
                           int N, unsigned long long* keys, float* conf_s, PlanShared& sh) {
  int bad = 0;
  for (int q = threadIdx.x; q < N; q += NT) {
    const float c = conf[q];
    if (!isfinite(c)) bad = 1;
    conf_s[q] = c;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) sh.err |= SD_DEV_ERR_CONF;
  for (int i = threadIdx.x; i < n; i += NT) {
    const int k = lens[i];
    const float* c = conf_s + off[i];
    float s = 1.0f;
    for (int j = 0; j < P; ++j) {
      unsigned long long key = kSentinel;
      if (j < k) {
        s = s * (1.0f / (1.0f + expf(-c[j])));
        key = (static_cast<unsigned long long>(~__float_as_uint(s)) << 32) |
              static_cast<unsigned long long>(i * P + j);
      }
      keys[i * P + j] = key;
    }
  }
  __syncthreads();
}

// Merge sort of n keys (power of two) whose runs of length `run` are already
// ascending.  Returns the buffer holding the result.
__device__ unsigned long long* merge_runs(unsigned long long* a, unsigned long long* b, int n,
                                          int run) {
  const int ipt = (n + NT - 1) / NT;
  for (int w = run; w < n; w <<= 1) {
    const int o_beg = static_cast<int>(threadIdx.x) * ipt;
    const int o_end = min(n, o_beg + ipt);
    for (int o = o_beg; o < o_end;) {
      const int base = (o / (2 * w)) * (2 * w);
      const int blk_end = min(base + 2 * w, o_end);
      const unsigned long long* A = a + base;
      const unsigned long long* Bv = a + base + w;
      const int k = o - base;
      // Merge path: ai = number of A elements among the first k outputs.
      int lo = max(0, k - w), hi = min(k, w);
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (A[mid] <= Bv[k - 1 - mid]) lo = mid + 1;
        else hi = mid;
      }
      int ai = lo, bi = k - lo;
      for (; o < blk_end; ++o) {
        const bool take_a = (bi >= w) || (ai < w && A[ai] <= Bv[bi]);
        b[o] = take_a ? A[ai++] : Bv[bi++];
      }
    }
    __syncthreads();
    unsigned long long* t = a;
    a = b;
    b = t;
  }
  return a;
}

// Budget argmax over B in [0, Bmax] on the sorted keys.  cm receives the
// monotone cost at T+B.  Returns B* (smallest maximiser).
__device__ int budget_argmax(const unsigned long long* sorted, int Bmax, int R, int T,
                             const float* cost, float* cm, PlanShared& sh) {
  // cost'[n] = max(cost[1..n]): the part below T is a plain maximum.
  float m0 = -INFINITY;
  for (int n = 1 + threadIdx.x; n < T; n += NT) m0 = fmaxf(m0, cost[n]);
  m0 = block_max_f32(m0, sh);
  // Running maximum over cost[T..T+Bmax] (chunked scan; entries must be > 0).
  const int cnt = Bmax + 1;
  const int chunk = (cnt + NT - 1) / NT;
  const int beg = min(cnt, static_cast<int>(threadIdx.x) * chunk);
  const int end = min(cnt, beg + chunk);
  float lm = -INFINITY;
  int bad = 0;
  for (int b = beg; b < end; ++b) {
    const float c = cost[T + b];
    if (!(isfinite(c) && c > 0.0f)) bad = 1;
    lm = fmaxf(lm, c);
    cm[b] = lm;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) sh.err |= SD_DEV_ERR_COST;
  // Exclusive running maximum across the chunks, folded into each chunk.
  const float excl = fmaxf(block_excl_max_scan(lm, sh), m0);
  for (int b = beg; b < end; ++b) cm[b] = fmaxf(cm[b], excl);
  __syncthreads();
  // E(B) = R + sum_{r<B} s_(r) in 2^-48 fixed point; objective and argmax.
  const int vchunk = (Bmax + NT - 1) / NT;
  const int vb = min(Bmax, static_cast<int>(threadIdx.x) * vchunk);
  const int ve = min(Bmax, vb + vchunk);
  unsigned long long local = 0;
  for (int r = vb; r < ve; ++r) {
    const float s = __uint_as_float(~static_cast<uint32_t>(sorted[r] >> 32));
    local += __float2ull_rn(s * kFix);
  }
  unsigned long long E = block_excl_scan_u64(local, sh, nullptr) +
                         static_cast<unsigned long long>(R) * 281474976710656ull;
  unsigned long long best = 0;
  auto consider = [&](int B, unsigned long long e) {
    const float obj = (__ull2float_rn(e) * (1.0f / kFix)) / cm[B];
    const unsigned long long key = (static_cast<unsigned long long>(__float_as_uint(obj)) << 32) |
                                   static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(B));
    best = key > best ? key : best;
  };
  if (threadIdx.x == 0) consider(0, E);
  for (int r = vb; r < ve; ++r) {
    const float s = __uint_as_float(~static_cast<uint32_t>(sorted[r] >> 32));
    E += __float2ull_rn(s * kFix);
    consider(r + 1, E);
  }
  best = block_max_u64(best, sh);
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFull));
}

__global__ void __launch_bounds__(NT, 1) plan_kernel(const PlanParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ PlanShared sh;
  const int NPm = max(p.NP, p.NPb);
  unsigned long long* keysA = reinterpret_cast<unsigned long long*>(smem);
  unsigned long long* keysB = keysA + NPm;
  float* cm = reinterpret_cast<float*>(keysB + NPm);        // [NPm + 1]
  int* lens = reinterpret_cast<int*>(cm + NPm + 1);        // [NPm / P]
  int* off = lens + NPm / p.P;                              // [NPm / P + 1]
  uint8_t* sel = reinterpret_cast<uint8_t*>(off + NPm / p.P + 1);  // [NP]

  if (threadIdx.x == 0) { sh.err = 0; sh.B = 0; }
  __syncthreads();

  const int L = p.cost_len - 1;
  const int nreq = p.NP / p.P;  // padded request count (power of two)
  // Current slots: lengths and offsets (padded requests have no slots).
  int N = load_lengths(p.lens, p.bs, p.k_max, lens, off, sh);
  for (int i = p.bs + threadIdx.x; i < nreq; i += NT) { lens[i] = 0; off[i] = N; }
  __syncthreads();

  int B = 0;
  if (p.mode == SD_MODE_ALL_SLOTS) {
    B = N;
  } else {
    if (p.budget_conf) {
      const int nb = p.NPb / p.P;
      const int Nb = load_lengths(p.budget_lens, p.bs_budget, p.k_max, lens, off, sh);
      for (int i = p.bs_budget + threadIdx.x; i < nb; i += NT) { lens[i] = 0; off[i] = Nb; }
      __syncthreads();
      if (sh.err == 0) {
        build_keys(p.budget_conf, lens, off, nb, p.P, Nb, keysA, reinterpret_cast<float*>(keysB), sh);
        const unsigned long long* sorted = merge_runs(keysA, keysB, p.NPb, p.P);
        const int Bmax_b = min(Nb, L - p.T);
        int Bb = 0;
        if (sh.err == 0) Bb = budget_argmax(sorted, Bmax_b, p.bs, p.T, p.cost, cm, sh);
        B = min(Bb, min(N, L - p.T));
      }
      // Restore the current request lengths.
      N = load_lengths(p.lens, p.bs, p.k_max, lens, off, sh);
      for (int i = p.bs + threadIdx.x; i < nreq; i += NT) { lens[i] = 0; off[i] = N; }
      __syncthreads();
    }
    if (sh.err == 0) {
      build_keys(p.conf, lens, off, nreq, p.P, N, keysA, reinterpret_cast<float*>(keysB), sh);
      const unsigned long long* sorted = merge_runs(keysA, keysB, p.NP, p.P);
      if (!p.budget_conf && sh.err == 0)
        B = budget_argmax(sorted, min(N, L - p.T), p.bs, p.T, p.cost, cm, sh);
      // Selection: the B best ranks.
      for (int q = threadIdx.x; q < p.NP; q += NT) sel[q] = 0;
      __syncthreads();
      if (sh.err == 0)
        for (int r = threadIdx.x; r < B; r += NT)
          sel[static_cast<uint32_t>(sorted[r] & 0xFFFFFFFFull)] = 1;
      __syncthreads();
    }
  }

  const bool failed = sh.err != 0;
  if (failed) B = 0;
  // Compaction: mask rows, n_i and cu_seqlens.
  const int chunk = (p.bs + NT - 1) / NT;
  const int beg = min(p.bs, static_cast<int>(threadIdx.x) * chunk);
  const int end = min(p.bs, beg + chunk);
  int local = 0;
  for (int i = beg; i < end; ++i) {
    int n = 0;
    for (int j = 0; j < p.k_max; ++j) {
      uint8_t m = 0;
      if (!failed && j < lens[i]) m = (p.mode == SD_MODE_ALL_SLOTS) ? 1 : sel[i * p.P + j];
      p.mask[static_cast<size_t>(i) * p.k_max + j] = m;
      n += m;
    }
    p.num_verified[i] = n;
    local += n + 1;
  }
  int total;
  int run = block_excl_scan_i32(local, sh, &total);
  for (int i = beg; i < end; ++i) {
    p.cu[i] = run;
    run += p.num_verified[i] + 1;
  }
  if (threadIdx.x == 0) {
    p.cu[p.bs] = total;
    p.B_out[0] = B;
    if (sh.err) raise_error(p.err, sh.err);
  }
}

}  // namespace

size_t plan_smem_bytes(const PlanParams& p) {
  const size_t NPm = static_cast<size_t>(p.NP > p.NPb ? p.NP : p.NPb);
  return 2 * NPm * 8 + (NPm + 1) * 4 + (NPm / p.P) * 4 + (NPm / p.P + 1) * 4 +
         static_cast<size_t>(p.NP) + 16;
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t s) {
  const size_t smem = plan_smem_bytes(p);
  // Raise the dynamic shared-memory limit to the device maximum once per device.
  static std::atomic<int> limit_of[64];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int lim = limit_of[dev].load(std::memory_order_acquire);
  if (lim == 0) {
    std::lock_guard<std::mutex> lk(mu);
    lim = limit_of[dev].load(std::memory_order_relaxed);
    if (lim == 0) {
      int optin = 0;
      e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
      if (e != cudaSuccess) return e;
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, plan_kernel);
      if (e != cudaSuccess) return e;
      lim = optin - static_cast<int>(fa.sharedSizeBytes);
      e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
      if (e != cudaSuccess) return e;
      limit_of[dev].store(lim, std::memory_order_release);
    }
  }
  if (smem > static_cast<size_t>(lim)) return cudaErrorInvalidValue;
  plan_kernel<<<1, NT, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace sdk
