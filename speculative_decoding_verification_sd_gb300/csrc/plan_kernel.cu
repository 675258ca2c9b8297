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
constexpr int kBuckets = 4096;     // bucket sort: buckets over the key range
constexpr int kBucketMax = 256;    // larger buckets fall back to the merge sort
constexpr float kFix = 281474976710656.0f;  // 2^48

struct PlanShared {
  unsigned long long red_u64[NW];
  float red_f32[NW];
  int red_i32[NW];
  int err;
  int B;
  unsigned long long scan_total;
  unsigned int hmin, hmax;
  int cmax;
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
    unsigned long long w = lane < NW ? sh.red_u64[lane] : 0ull;
    unsigned long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      unsigned long long t = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < NW) sh.red_u64[lane] = wi - w;  // exclusive prefix of warp totals
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

// round(s * 2^48) to nearest even for 0 <= s <= 1 (the value
// __float2ull_rn(s * 2^48) has), in integer arithmetic.
__device__ __forceinline__ unsigned long long fix48(float s) {
  const uint32_t b = __float_as_uint(s);
  const int e = static_cast<int>((b >> 23) & 0xFFu);
  if (e == 0) return 0ull;  // zero, or below 2^-126
  const unsigned long long m = (b & 0x7FFFFFu) | 0x800000u;  // s = m * 2^(e - 150)
  const int sh = e - 150 + 48;
  if (sh >= 0) return m << sh;
  if (sh < -25) return 0ull;  // s * 2^48 < 1/4
  const int k = -sh;
  const unsigned long long q = m >> k, r = m & ((1ull << k) - 1), half = 1ull << (k - 1);
  return q + ((r > half || (r == half && (q & 1ull))) ? 1ull : 0ull);
}

// x correctly rounded to fp32 (nearest even), in integer arithmetic (the
// value __ull2float_rn(x) has).
__device__ __forceinline__ float u64_to_f32(unsigned long long x) {
  if (x < (1ull << 24)) return static_cast<float>(static_cast<uint32_t>(x));
  const int k = 63 - __clzll(static_cast<long long>(x)) - 23;  // bits dropped
  unsigned long long q = x >> k;
  const unsigned long long r = x & ((1ull << k) - 1), half = 1ull << (k - 1);
  q += (r > half || (r == half && (q & 1ull))) ? 1ull : 0ull;  // q <= 2^24
  // q * 2^k: q converts exactly; the power of two goes into the exponent field
  return __uint_as_float(__float_as_uint(static_cast<float>(static_cast<uint32_t>(q))) +
                         (static_cast<uint32_t>(k) << 23));
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
      const int base = o & ~(2 * w - 1);  // w is a power of two
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

// Sort of the n (power of two) keys by distribution: each real key goes to
// one of kBuckets buckets by its high word (monotone in the key), buckets
// are laid out by an exclusive scan of their counts, and every key then
// finds its place inside its bucket by counting the bucket's smaller keys
// (keys are distinct: the low word is the slot index).  The real keys end
// up ascending in keys[0..N) (tmp is scratch); sentinels are dropped.
// Returns false (keys untouched) when a bucket holds more than kBucketMax
// keys, e.g. many equal survivals; the caller then merges the runs instead.
__device__ bool bucket_sort(unsigned long long* keys, unsigned long long* tmp, int n, int* cnt,
                            int* end, PlanShared& sh) {
  unsigned int lo = 0xFFFFFFFFu, hi = 0u;
  for (int q = threadIdx.x; q < n; q += NT) {
    const unsigned long long k = keys[q];
    if (k != kSentinel) {
      const unsigned int h = static_cast<unsigned int>(k >> 32);
      lo = min(lo, h);
      hi = max(hi, h);
    }
  }
  for (int q = threadIdx.x; q < kBuckets; q += NT) cnt[q] = 0;
  if (threadIdx.x == 0) { sh.hmin = 0xFFFFFFFFu; sh.hmax = 0u; sh.cmax = 0; }
  __syncthreads();
  lo = __reduce_min_sync(kFull, lo);
  hi = __reduce_max_sync(kFull, hi);
  if ((threadIdx.x & 31) == 0) {
    atomicMin(&sh.hmin, lo);
    atomicMax(&sh.hmax, hi);
  }
  __syncthreads();
  const unsigned int hmin = sh.hmin;
  if (hmin > sh.hmax) return true;  // no real key
  const unsigned int range = sh.hmax - hmin;
  int shift = 0;
  while ((range >> shift) >= static_cast<unsigned int>(kBuckets)) ++shift;
  for (int q = threadIdx.x; q < n; q += NT) {
    const unsigned long long k = keys[q];
    if (k != kSentinel) atomicAdd(&cnt[(static_cast<unsigned int>(k >> 32) - hmin) >> shift], 1);
  }
  __syncthreads();
  // bucket offsets (exclusive scan, kBuckets / NT consecutive buckets per thread)
  constexpr int kPer = kBuckets / NT;
  int c[kPer], local = 0, cm = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    c[q] = cnt[threadIdx.x * kPer + q];
    local += c[q];
    cm = max(cm, c[q]);
  }
  cm = __reduce_max_sync(kFull, cm);
  if ((threadIdx.x & 31) == 0) atomicMax(&sh.cmax, cm);
  int run = block_excl_scan_i32(local, sh, nullptr);  // synchronises the block
  if (sh.cmax > kBucketMax) return false;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    run += c[q];
    cnt[threadIdx.x * kPer + q] = run - c[q];  // the bucket's fill cursor
    end[threadIdx.x * kPer + q] = run;
  }
  __syncthreads();
  for (int q = threadIdx.x; q < n; q += NT) {
    const unsigned long long k = keys[q];
    if (k != kSentinel) tmp[atomicAdd(&cnt[(static_cast<unsigned int>(k >> 32) - hmin) >> shift], 1)] = k;
  }
  __syncthreads();
  const int total = end[kBuckets - 1];
  // each key's place: its bucket's start plus the bucket's keys below it
  for (int x = threadIdx.x; x < total; x += NT) {
    const unsigned long long v = tmp[x];
    const int bk = static_cast<int>((static_cast<unsigned int>(v >> 32) - hmin) >> shift);
    const int e = end[bk], b0 = bk > 0 ? end[bk - 1] : 0;
    int r = 0;
    for (int y = b0; y < e; ++y) r += tmp[y] < v;
    keys[b0 + r] = v;
  }
  __syncthreads();
  return true;
}

// Budget argmax over B in [0, Bmax] on the sorted keys.  cm[b] holds
// cost[T+b] (loaded at kernel start) and lm each thread's maximum of its share
// of cost[1..T) (lm_bad: one of those was not finite and positive).  Thread t
// owns the budgets B in [vb, ve); one combined block scan gives every thread
// its prefix of the survival sum (exact, 2^48 fixed point) and of the running
// cost maximum (the monotone cost'[n] = max(cost[1..n])).  Returns B*
// (smallest maximiser).
__device__ int budget_argmax(const unsigned long long* sorted, int Bmax, int R, float* cm,
                             float lm, int lm_bad, PlanShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cnt = Bmax + 1;
  const int chunk = (cnt + NT - 1) / NT;
  const int vb = min(cnt, static_cast<int>(threadIdx.x) * chunk);
  const int ve = min(cnt, vb + chunk);
  int bad = lm_bad;
  float cmax = -INFINITY;
  unsigned long long ls = 0;
  for (int B = vb; B < ve; ++B) {
    const float c = cm[B];
    if (!(isfinite(c) && c > 0.0f)) bad = 1;
    cmax = fmaxf(cmax, c);
    cm[B] = cmax;  // running maximum within the chunk
    if (B < Bmax) ls += fix48(__uint_as_float(~static_cast<uint32_t>(sorted[B] >> 32)));
  }
  // combined scan: exclusive sums, exclusive running maxima, total of lm
  unsigned long long si = ls;
  float mi = cmax, m0 = lm;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long ts = __shfl_up_sync(kFull, si, o);
    const float tm = __shfl_up_sync(kFull, mi, o);
    if (lane >= o) {
      si += ts;
      mi = fmaxf(mi, tm);
    }
    m0 = fmaxf(m0, __shfl_xor_sync(kFull, m0, o));
  }
  if (lane == 31) {
    sh.red_u64[warp] = si;
    sh.red_f32[warp] = mi;
  }
  if (lane == 0) sh.red_i32[warp] = __float_as_int(m0);
  if (__syncthreads_or(bad) && threadIdx.x == 0) sh.err |= SD_DEV_ERR_COST;
  if (warp == 0) {
    unsigned long long ws = lane < NW ? sh.red_u64[lane] : 0ull;
    float wm = lane < NW ? sh.red_f32[lane] : -INFINITY;
    float w0 = lane < NW ? __int_as_float(sh.red_i32[lane]) : -INFINITY;
    const unsigned long long ws_in = ws;
    const float wm_in = wm;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long ts = __shfl_up_sync(kFull, ws, o);
      const float tm = __shfl_up_sync(kFull, wm, o);
      if (lane >= o) {
        ws += ts;
        wm = fmaxf(wm, tm);
      }
      w0 = fmaxf(w0, __shfl_xor_sync(kFull, w0, o));
    }
    const float wm_ex = __shfl_up_sync(kFull, wm, 1);
    if (lane < NW) {
      sh.red_u64[lane] = ws - ws_in;                    // exclusive warp sums
      sh.red_f32[lane] = lane == 0 ? -INFINITY : wm_ex;  // exclusive warp maxima
    }
    if (lane == 0) sh.red_i32[0] = __float_as_int(w0);
    (void)wm_in;
  }
  __syncthreads();
  const float mi_up = __shfl_up_sync(kFull, mi, 1);  // every lane takes part
  const float mi_ex = lane == 0 ? -INFINITY : mi_up;
  const float mpre = fmaxf(fmaxf(sh.red_f32[warp], mi_ex), __int_as_float(sh.red_i32[0]));
  unsigned long long E = sh.red_u64[warp] + (si - ls) + static_cast<unsigned long long>(R) * 281474976710656ull;
  // objectives of this thread's budgets; the largest (smallest B on ties) wins
  unsigned long long best = 0;
  for (int B = vb; B < ve; ++B) {
    const float c = fmaxf(cm[B], mpre);
    const float obj = (u64_to_f32(E) * (1.0f / kFix)) / c;
    const unsigned long long key = (static_cast<unsigned long long>(__float_as_uint(obj)) << 32) |
                                   static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(B));
    best = key > best ? key : best;
    if (B < Bmax) E += fix48(__uint_as_float(~static_cast<uint32_t>(sorted[B] >> 32)));
  }
  best = warp_max_u64(best);
  if (threadIdx.x == 0) sh.scan_total = 0;
  __syncthreads();
  if (lane == 0) atomicMax(&sh.scan_total, best);
  __syncthreads();
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(sh.scan_total & 0xFFFFFFFFull));
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
  int* bcnt = off + NPm / p.P + 1;                          // [2 * kBuckets]
  uint8_t* sel = reinterpret_cast<uint8_t*>(bcnt + 2 * kBuckets);  // [NP]

  if (threadIdx.x == 0) { sh.err = 0; sh.B = 0; }
  const int L = p.cost_len - 1;
  // The cost table is read first, so that its loads overlap the lengths':
  // cost[T+b] for every budget b the call can reach, and each thread's
  // maximum of its share of cost[1..T).
  float lm = -INFINITY;
  int lm_bad = 0;
  if (p.mode != SD_MODE_ALL_SLOTS) {
    for (int n = 1 + threadIdx.x; n < p.T; n += NT) {
      const float c = p.cost[n];
      if (!(isfinite(c) && c > 0.0f)) lm_bad = 1;
      lm = fmaxf(lm, c);
    }
    const int bmax = min(NPm, L - p.T);
    for (int b = threadIdx.x; b <= bmax; b += NT) cm[b] = p.cost[p.T + b];
  }
  __syncthreads();

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
        const unsigned long long* sorted = bucket_sort(keysA, keysB, p.NPb, bcnt, bcnt + kBuckets, sh)
                                               ? keysA
                                               : merge_runs(keysA, keysB, p.NPb, p.P);
        const int Bmax_b = min(Nb, L - p.T);
        int Bb = 0;
        if (sh.err == 0) Bb = budget_argmax(sorted, Bmax_b, p.bs, cm, lm, lm_bad, sh);
        B = min(Bb, min(N, L - p.T));
      }
      // Restore the current request lengths.
      N = load_lengths(p.lens, p.bs, p.k_max, lens, off, sh);
      for (int i = p.bs + threadIdx.x; i < nreq; i += NT) { lens[i] = 0; off[i] = N; }
      __syncthreads();
    }
    if (sh.err == 0) {
      build_keys(p.conf, lens, off, nreq, p.P, N, keysA, reinterpret_cast<float*>(keysB), sh);
      const unsigned long long* sorted = bucket_sort(keysA, keysB, p.NP, bcnt, bcnt + kBuckets, sh)
                                             ? keysA
                                             : merge_runs(keysA, keysB, p.NP, p.P);
      if (!p.budget_conf && sh.err == 0)
        B = budget_argmax(sorted, min(N, L - p.T), p.bs, cm, lm, lm_bad, sh);
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
         static_cast<size_t>(kBuckets) * 8 + static_cast<size_t>(p.NP) + 16;
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
