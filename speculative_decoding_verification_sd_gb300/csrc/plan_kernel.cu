// plan_kernel.cu -- K1: the planning stage of adaptive verification in one
// CTA of 1024 threads, everything resident in shared memory.
//
//   survival   a = sigmoid(conf), s_j = a_0 * ... * a_j along the draft
//              [fosworld blog "추측 디코딩과 vLLM 적응형 검증", "동작" step 1]
//   top-B      all slots ranked by (s desc, packed index asc): a bucket sort
//              on the key's high word, with a merge of the per-request runs
//              (each already sorted; merge path, Odeh et al. 2012) when a
//              bucket overflows
//              ["동작" step 2; agentlenshq "vLLM DSpark을 활용한 적응형 검증",
//               "DSpark 신뢰도 스케줄링 메커니즘" / Global Top-B Selection]
//   budget     B* = smallest argmax_B (R + sum of the B best s) / cost'[T+B],
//              cost' = running max of the table (forced monotone)
//              ["동작" step 3; same page, Budget Calculation, and
//               "기술적 구현 및 CUDA Graphs" / Cost Modeling, CUDA Graph Padding]
//   uniform K  (the other planning mode) one draft length K for the batch:
//              K* = smallest argmax_K (R + survival of each request's first
//              min(K, K_i) slots) / cost'[T + their number]
//              [discuss.pytorch.kr "DSD feat. Cohere", "동적 추측 디코딩(DSD)의
//               핵심 아이디어": goodput = AL / ITL]
//   compaction slot mask, n_i and cu_seqlens (n_i drafts + 1 row per request)
//              [same page, Execution Pipeline: assignment on the GPU without a
//               host round trip]
//   calibration (calib_kernel) one online step of the per-position
//              acceptance model a = sigmoid(w_j c + b_j), and the calibrated
//              logits w_j c + b_j that the planner then takes as its input
//              [fosworld blog, the table under "동작": a small logistic model
//               on the draft's logits, corrected with the verification results]
//
// The prefix sums of the ranked survival values are exact integer sums of
// the fp32 keys scaled by 2^48 (at most 8192 terms <= 1, so they fit in 62
// bits); only the final division by the cost is rounded.
#include <atomic>
#include <mutex>

#include "calib.h"
#include "sd_device.cuh"
#include "sd_internal.h"

namespace sdk {

namespace {

constexpr int NT = kPlanThreads;
constexpr int NW = NT / 32;
constexpr unsigned long long kSentinel = ~0ull;
constexpr int kBuckets = 4096;     // bucket sort: buckets over the key range
constexpr int kBucketMax = 256;    // larger buckets fall back to the merge sort
constexpr unsigned kOneBits = 0x3F800000u;  // bit pattern of 1.0f
constexpr int kBucketShift = 15;   // 2^15 ulps a bucket: 256 buckets a binade
static_assert(kBuckets == 4 * NT, "four bucket counters a thread, moved as one 16-byte vector");
constexpr float kFix = 281474976710656.0f;  // 2^48
constexpr int kMaxP = 16;          // pow2ceil(SD_MAX_K)

struct PlanShared {
  unsigned long long tot_u64[NW];  // per-warp totals of the block scans
  float tot_f32[NW];
  float tot_m0[NW];
  int tot_i32[NW];
  int err;
  unsigned long long best;         // budget argmax (packed objective, budget)
  int cmax;                        // largest bucket of the bucket sort
  unsigned long long col_s[kMaxP]; // uniform K: survival sum of position j (2^48)
  int col_n[kMaxP];                // uniform K: requests that draft position j
};

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

template <typename U>
__device__ __forceinline__ U warp_incl_scan(U v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const U t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive block scan of non-negative ints with one barrier: each warp scans
// its values, lane 31 publishes the warp total in tot[warp], and after the
// barrier every warp adds up the totals of the warps before it (and of all
// warps) with two warp reductions.  tot must not be written again before
// every thread has passed a later barrier.
__device__ int block_scan_excl(int v, int* tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int inc = warp_incl_scan(v);
  if (lane == 31) tot[warp] = inc;
  __syncthreads();
  const unsigned w = lane < NW ? static_cast<unsigned>(tot[lane]) : 0u;
  const int before = static_cast<int>(__reduce_add_sync(kFull, lane < warp ? w : 0u));
  if (total) *total = static_cast<int>(__reduce_add_sync(kFull, w));
  return before + inc - v;
}

// Sum over the warp of values below 2^62 (the 2^48 fixed-point survival sums),
// as three 32-bit warp reductions of 24-, 24- and 14-bit pieces.
__device__ __forceinline__ unsigned long long warp_sum_u62(unsigned long long x) {
  const unsigned lo = __reduce_add_sync(kFull, static_cast<unsigned>(x & 0xFFFFFFull));
  const unsigned mid = __reduce_add_sync(kFull, static_cast<unsigned>((x >> 24) & 0xFFFFFFull));
  const unsigned hi = __reduce_add_sync(kFull, static_cast<unsigned>(x >> 48));
  return static_cast<unsigned long long>(lo) + (static_cast<unsigned long long>(mid) << 24) +
         (static_cast<unsigned long long>(hi) << 48);
}

// Maximum over the warp of floats that are >= 0 or -inf: for those, the
// order of the bit patterns read as signed ints is the order of the values.
__device__ __forceinline__ float warp_max_nonneg(float x) {
  return __int_as_float(__reduce_max_sync(kFull, __float_as_int(x)));
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

// Requests per thread in the contiguous chunks that the lengths are read in
// (bs <= pow2ceil(bs) <= SD_MAX_PLAN_SLOTS).
constexpr int kReqPer = SD_MAX_PLAN_SLOTS / NT;

struct Chunk {
  int beg, end;
};

__device__ __forceinline__ Chunk req_chunk(int n) {
  const int c = (n + NT - 1) / NT;
  const int beg = min(n, static_cast<int>(threadIdx.x) * c);
  return {beg, min(n, beg + c)};
}

// Bucket of a key with high word h = ~bits(s), 0 <= s <= 1: 256 buckets for
// each binade below 1, down to 2^-16; smaller survivals share the last
// bucket.  Monotone in h, so ascending buckets hold ascending keys.  A NaN
// survival (bad input, flagged) lands in the last bucket.
__device__ __forceinline__ int bucket_of(unsigned int h) {
  const unsigned int d = kOneBits - ~h;
  return static_cast<int>(min(d >> kBucketShift, static_cast<unsigned int>(kBuckets - 1)));
}

// Issues the loads of this thread's chunk of draft lengths into registers.
// The loads are volatile so that they stay ahead of the cost table's (whose
// use stalls the thread) and all of them travel together.
__device__ __forceinline__ void fetch_lengths(const int* g, Chunk ch, int (&r)[kReqPer]) {
#pragma unroll
  for (int q = 0; q < kReqPer; ++q) r[q] = 0;
#pragma unroll
  for (int q = 0; q < kReqPer; ++q) {
    if (ch.beg + q >= ch.end) break;
    asm volatile("ld.global.b32 %0, [%1];" : "=r"(r[q]) : "l"(g + ch.beg + q));
  }
}

// Checks the fetched lengths of n requests, stores them in lens and forms the
// packed offsets off[0..nreq] (requests n..nreq are padding with no slots).
// Returns the total slot count N.  Ends with a barrier.
__device__ int load_lengths(const int (&r)[kReqPer], Chunk ch, int n, int nreq, int k_max,
                            uint8_t* lens, int* off, PlanShared& sh) {
  int local = 0, bad = 0;
#pragma unroll
  for (int q = 0; q < kReqPer; ++q) {
    if (ch.beg + q >= ch.end) break;
    int k = r[q];
    if (k < 0 || k > k_max) { bad = 1; k = 0; }
    lens[ch.beg + q] = static_cast<uint8_t>(k);
    local += k;
  }
  if (bad) atomicOr(&sh.err, SD_DEV_ERR_DRAFT_LENS);
  int total;
  int run = block_scan_excl(local, sh.tot_i32, &total);
#pragma unroll
  for (int q = 0; q < kReqPer; ++q) {
    if (ch.beg + q >= ch.end) break;
    off[ch.beg + q] = run;
    run += lens[ch.beg + q];
  }
  for (int i = n + threadIdx.x; i <= nreq; i += NT) {
    if (i < nreq) lens[i] = 0;
    off[i] = total;
  }
  __syncthreads();
  return total;
}

// Slots per thread in the key phase (nreq * P <= SD_MAX_PLAN_SLOTS).
constexpr int kSlotPer = SD_MAX_PLAN_SLOTS / NT;

// Sort keys of nreq requests, P slots each: high word = ~bits(s) (s >= 0, so
// a larger survival gives a smaller key), low word = q = i*P + j (packed
// order).  Unused slots hold the sentinel, which sorts last.  One thread per
// slot: all of a thread's confidence logits are requested first, then each
// slot takes a_j = sigmoid(c_j) and the survival s_j = a_0 * ... * a_j comes
// from a product scan over the request's P lanes (log2 P steps: the same
// factors as the front-to-back product, associated differently, so equal to
// it within fp32 rounding).  Every real key is counted in its bucket (cnt
// holds kBuckets zeroed counters).  Ends with a barrier.
__device__ void build_keys(const float* conf, const uint8_t* lens, const int* off, int nreq, int P,
                           unsigned long long* keys, int* cnt, PlanShared& sh) {
  const int n = nreq * P;
  const int lgP = 31 - __clz(P);
  float cv[kSlotPer];
#pragma unroll
  for (int r = 0; r < kSlotPer; ++r) cv[r] = 0.0f;
#pragma unroll
  for (int r = 0; r < kSlotPer; ++r) {
    if (r * NT >= n) break;
    const int q = r * NT + static_cast<int>(threadIdx.x);
    const int i = q >> lgP, j = q & (P - 1);
    if (q < n && j < lens[i]) cv[r] = conf[off[i] + j];
  }
  int bad = 0;
#pragma unroll
  for (int r = 0; r < kSlotPer; ++r) {
    if (r * NT >= n) break;  // uniform: the scan below is warp-wide
    const int q = r * NT + static_cast<int>(threadIdx.x);
    const int i = q >> lgP, j = q & (P - 1);
    const bool real = q < n && j < lens[i];
    float s = 1.0f;
    if (real) {
      if (!isfinite(cv[r])) bad = 1;
      s = 1.0f / (1.0f + expf(-cv[r]));
    }
    for (int d = 1; d < P; d <<= 1) {
      const float t = __shfl_up_sync(kFull, s, d, P);
      if (j >= d) s *= t;
    }
    if (q < n) {
      unsigned long long key = kSentinel;
      if (real) {
        const unsigned int h = ~__float_as_uint(s);
        key = (static_cast<unsigned long long>(h) << 32) | static_cast<unsigned long long>(q);
        atomicAdd(&cnt[bucket_of(h)], 1);
      }
      keys[q] = key;
    }
  }
  if (bad) atomicOr(&sh.err, SD_DEV_ERR_CONF);
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

// Sort of the n (power of two) keys by distribution: build_keys counted each
// real key in its bucket (bucket_of, monotone in the key); buckets are laid
// out by an exclusive scan of their counts, the keys are scattered into their
// buckets, and every key then finds its place inside its bucket by counting
// the bucket's smaller keys (keys are distinct: the low word is the slot
// index).  The real keys end up ascending in keys[0..N) (tmp is scratch);
// sentinels are dropped.  After the scatter cnt[b] is the end of bucket b.
// Returns false (keys untouched) when a bucket holds more than kBucketMax
// keys, e.g. many equal survivals; the caller then merges the runs instead.
__device__ bool bucket_sort(unsigned long long* keys, unsigned long long* tmp, int n, int* cnt,
                            PlanShared& sh) {
  // bucket offsets (exclusive scan, kBuckets / NT consecutive buckets per thread)
  constexpr int kPer = 4;
  const int4 c4 = reinterpret_cast<const int4*>(cnt)[threadIdx.x];
  const int c[kPer] = {c4.x, c4.y, c4.z, c4.w};
  int local = 0, cm = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    local += c[q];
    cm = max(cm, c[q]);
  }
  cm = __reduce_max_sync(kFull, cm);
  if ((threadIdx.x & 31) == 0) atomicMax(&sh.cmax, cm);
  int run = block_scan_excl(local, sh.tot_i32, nullptr);
  if (sh.cmax > kBucketMax) return false;  // read after the scan's barrier
  int4 cur;  // the buckets' fill cursors
  cur.x = run;
  cur.y = cur.x + c[0];
  cur.z = cur.y + c[1];
  cur.w = cur.z + c[2];
  reinterpret_cast<int4*>(cnt)[threadIdx.x] = cur;
  __syncthreads();
  for (int q = threadIdx.x; q < n; q += NT) {
    const unsigned long long k = keys[q];
    if (k != kSentinel) tmp[atomicAdd(&cnt[bucket_of(static_cast<unsigned int>(k >> 32))], 1)] = k;
  }
  __syncthreads();
  const int total = cnt[kBuckets - 1];
  // each key's place: its bucket's start plus the bucket's keys below it
  for (int x = threadIdx.x; x < total; x += NT) {
    const unsigned long long v = tmp[x];
    const int bk = bucket_of(static_cast<unsigned int>(v >> 32));
    const int e = cnt[bk], b0 = bk > 0 ? cnt[bk - 1] : 0;
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
// cost maximum (the monotone cost'[n] = max(cost[1..n])).  fx is scratch for
// the fixed-point survivals (Bmax entries).  Returns B* (smallest maximiser).
// Ends with a barrier.
__device__ int budget_argmax(const unsigned long long* sorted, unsigned long long* fx, int Bmax,
                             int R, float* cm, float lm, int lm_bad, PlanShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cnt = Bmax + 1;
  // an odd chunk keeps the strided shared-memory accesses free of bank conflicts
  const int chunk = ((cnt + NT - 1) / NT) | 1;
  const int vb = min(cnt, static_cast<int>(threadIdx.x) * chunk);
  const int ve = min(cnt, vb + chunk);
  if (threadIdx.x == 0) sh.best = 0ull;
  int bad = lm_bad;
  float cmax = -INFINITY;
  unsigned long long ls = 0;
  for (int B = vb; B < ve; ++B) {
    const float c = cm[B];
    if (!(isfinite(c) && c > 0.0f)) bad = 1;
    cmax = fmaxf(cmax, c);
    cm[B] = cmax;  // running maximum within the chunk
    if (B < Bmax) {
      const unsigned long long f = fix48(__uint_as_float(~static_cast<uint32_t>(sorted[B] >> 32)));
      fx[B] = f;
      ls += f;
    }
  }
  // Combined scan: inclusive sums and running maxima within the warp; the
  // warp totals go through shared memory, and each warp adds up those of the
  // warps before it with warp reductions (costs are > 0 when valid; invalid
  // ones raise the error flag, so their order does not matter).
  unsigned long long si = ls;
  float mi = cmax;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long ts = __shfl_up_sync(kFull, si, o);
    const float tm = __shfl_up_sync(kFull, mi, o);
    if (lane >= o) {
      si += ts;
      mi = fmaxf(mi, tm);
    }
  }
  const float m0 = warp_max_nonneg(lm);
  if (lane == 31) {
    sh.tot_u64[warp] = si;
    sh.tot_f32[warp] = mi;
  }
  if (lane == 0) sh.tot_m0[warp] = m0;
  if (bad) atomicOr(&sh.err, SD_DEV_ERR_COST);
  __syncthreads();
  const bool earlier = lane < warp;
  const unsigned long long w_ex = warp_sum_u62(earlier ? sh.tot_u64[lane] : 0ull);
  const float wm_ex = warp_max_nonneg(earlier ? sh.tot_f32[lane] : -INFINITY);
  const float w0 = warp_max_nonneg(lane < NW ? sh.tot_m0[lane] : -INFINITY);
  const float mi_up = __shfl_up_sync(kFull, mi, 1);
  const float mi_ex = lane == 0 ? -INFINITY : mi_up;
  const float mpre = fmaxf(fmaxf(wm_ex, mi_ex), w0);
  unsigned long long E = w_ex + (si - ls) + static_cast<unsigned long long>(R) * 281474976710656ull;
  // objectives of this thread's budgets; the largest (smallest B on ties) wins
  unsigned long long best = 0;
  for (int B = vb; B < ve; ++B) {
    const float c = fmaxf(cm[B], mpre);
    const float obj = (u64_to_f32(E) * (1.0f / kFix)) / c;
    const unsigned long long key = (static_cast<unsigned long long>(__float_as_uint(obj)) << 32) |
                                   static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(B));
    best = key > best ? key : best;
    if (B < Bmax) E += fx[B];
  }
  // warp maximum of the packed keys: the high words first, then the low
  // words of the lanes that hold the largest high word
  const unsigned bh = __reduce_max_sync(kFull, static_cast<unsigned>(best >> 32));
  const unsigned bl = __reduce_max_sync(kFull, static_cast<unsigned>(best >> 32) == bh
                                                   ? static_cast<unsigned>(best & 0xFFFFFFFFull)
                                                   : 0u);
  if (lane == 0) atomicMax(&sh.best, (static_cast<unsigned long long>(bh) << 32) | bl);
  __syncthreads();
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(sh.best & 0xFFFFFFFFull));
}

// Uniform draft length.  keys: build_keys' output in packed order (slot
// (i, j) at i * P + j, sentinel where request i has no slot j).  The
// survival of each position j is summed over the requests (2^48 fixed
// point, exact) with the number of requests that reach it; warp K then forms
// AL(K) = R + sum_{j<K} col_s[j] and the token count n(K) = sum_{j<K}
// col_n[j], and takes the objective AL(K) / cost'[T + n(K)] for every K up
// to the longest draft whose tokens fit the table.  cm[b] holds cost[T+b]
// (b <= Bmax, each checked here) and lm each thread's maximum of its share
// of cost[1..T).  sh.col_s / sh.col_n start zeroed.  Returns K* (smallest
// maximiser) and its token count in *B; after its last barrier it only
// reads shared state that later steps do not write.
__device__ int uniform_argmax(const unsigned long long* keys, int NP, int P, int k_max, int Bmax,
                              int R, const float* cm, float lm, int lm_bad, PlanShared& sh,
                              int* B) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) sh.best = 0ull;
  // P divides NT, so every slot a thread visits has the same position j
  unsigned long long acc = 0;
  int cnt = 0;
#pragma unroll
  for (int r = 0; r < kSlotPer; ++r) {
    const int q = r * NT + static_cast<int>(threadIdx.x);
    if (q >= NP) break;
    const unsigned long long key = keys[q];
    if (key != kSentinel) {
      acc += fix48(__uint_as_float(~static_cast<uint32_t>(key >> 32)));
      ++cnt;
    }
  }
  for (int o = P; o < 32; o <<= 1) {
    acc += __shfl_xor_sync(kFull, acc, o);
    cnt += __shfl_xor_sync(kFull, cnt, o);
  }
  if (lane < P && lane < 32) {
    atomicAdd(&sh.col_s[lane], acc);
    atomicAdd(&sh.col_n[lane], cnt);
  }
  int bad = lm_bad;
  for (int b = threadIdx.x; b <= Bmax; b += NT) {
    const float c = cm[b];
    if (!(isfinite(c) && c > 0.0f)) bad = 1;
  }
  const float m0 = warp_max_nonneg(lm);
  if (lane == 0) sh.tot_m0[warp] = m0;
  if (bad) atomicOr(&sh.err, SD_DEV_ERR_COST);
  __syncthreads();
  const int K = warp;
  if (K <= k_max && (K == 0 || sh.col_n[K - 1] > 0)) {
    unsigned long long E = static_cast<unsigned long long>(R) * 281474976710656ull;
    int n = 0;
    for (int j = 0; j < K; ++j) {
      E += sh.col_s[j];
      n += sh.col_n[j];
    }
    if (n <= Bmax) {  // tokens grow with K; Bmax = min(N, cost_len-1-T)
      float c = warp_max_nonneg(lane < NW ? sh.tot_m0[lane] : -INFINITY);
      for (int b = lane; b <= n; b += 32) c = fmaxf(c, cm[b]);
      c = warp_max_nonneg(c);
      const float obj = (u64_to_f32(E) * (1.0f / kFix)) / c;
      if (lane == 0)
        atomicMax(&sh.best, (static_cast<unsigned long long>(__float_as_uint(obj)) << 32) |
                                static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(K)));
    }
  }
  __syncthreads();
  const int Ks = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(sh.best & 0xFFFFFFFFull));
  int n = 0;
  for (int j = 0; j < Ks; ++j) n += sh.col_n[j];
  *B = n;
  return Ks;
}

// Shared-memory layout of one launch (NPm = max(NP, NPb), NRm = NPm / P).
struct PlanSmem {
  unsigned long long* keysA;  // [NPm]
  unsigned long long* keysB;  // [NPm]
  float* cm;                  // [NPm + 1] cost[T+b], then its running maximum
  int* off;                   // [NRm + 1]
  int* cnt;                   // [kBuckets]
  uint8_t* lens;              // [NRm]
  uint8_t* sel;               // [NP]
};

__host__ __device__ inline size_t plan_layout(int NP, int NPb, int P, unsigned char* base,
                                              PlanSmem* m) {
  const size_t NPm = static_cast<size_t>(NP > NPb ? NP : NPb);
  const size_t NRm = NPm / static_cast<size_t>(P);
  size_t o = 0;
  auto take = [&o](size_t bytes) {  // each part starts on a 16-byte boundary
    const size_t at = o;
    o = (o + bytes + 15) / 16 * 16;
    return at;
  };
  const size_t keysA = take(NPm * 8);
  const size_t keysB = take(NPm * 8);
  const size_t cm = take((NPm + 1) * 4);
  const size_t off = take((NRm + 1) * 4);
  const size_t cnt = take(static_cast<size_t>(kBuckets) * 4);
  const size_t lens = take(NRm);
  const size_t sel = take(static_cast<size_t>(NP));
  if (m) {
    m->keysA = reinterpret_cast<unsigned long long*>(base + keysA);
    m->keysB = reinterpret_cast<unsigned long long*>(base + keysB);
    m->cm = reinterpret_cast<float*>(base + cm);
    m->off = reinterpret_cast<int*>(base + off);
    m->cnt = reinterpret_cast<int*>(base + cnt);
    m->lens = base + lens;
    m->sel = base + sel;
  }
  return o;
}

// Sorts the keys of one slot set; returns the buffer that holds them ascending.
// Both ways end with a barrier; the bucket counters are then zeroed again
// for a later build_keys (which runs after further barriers).
__device__ const unsigned long long* sort_keys(const PlanSmem& m, int n, int P, PlanShared& sh) {
  const unsigned long long* sorted =
      bucket_sort(m.keysA, m.keysB, n, m.cnt, sh) ? m.keysA : merge_runs(m.keysA, m.keysB, n, P);
  reinterpret_cast<int4*>(m.cnt)[threadIdx.x] = int4{0, 0, 0, 0};  // kBuckets == 4 * NT
  if (threadIdx.x == 0) sh.cmax = 0;
  return sorted;
}

__global__ void __launch_bounds__(NT, 1) plan_kernel(const PlanParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ PlanShared sh;
  PlanSmem m;
  plan_layout(p.NP, p.NPb, p.P, smem, &m);
  const int NPm = max(p.NP, p.NPb);
  const int nreq = p.NP / p.P;  // padded request counts (powers of two)
  const int nb = p.NPb / p.P;
  const int L = p.cost_len - 1;
  const bool adaptive = p.mode != SD_MODE_ALL_SLOTS;  // a cost-driven mode
  const bool uniform = p.mode == SD_MODE_UNIFORM_K;

  // Every global input the first steps need is requested at once: the draft
  // lengths (current, and those of the budget set) into registers, cost[T+b]
  // for every budget b the call can reach into shared memory, and each
  // thread's maximum of its share of cost[1..T).
  const Chunk cc = req_chunk(p.bs);
  int rc[kReqPer], rb[kReqPer];
  fetch_lengths(p.lens, cc, rc);
  Chunk cb = {0, 0};
  if (p.budget_conf) {
    cb = req_chunk(p.bs_budget);
    fetch_lengths(p.budget_lens, cb, rb);
  }
  float lm = -INFINITY;
  int lm_bad = 0;
  if (adaptive) {
    const int bmax = min(NPm, L - p.T);
    for (int b = threadIdx.x; b <= bmax; b += NT) cp_async4(m.cm + b, p.cost + p.T + b);
    for (int n = 1 + threadIdx.x; n < p.T; n += NT) {
      const float c = p.cost[n];
      if (!(isfinite(c) && c > 0.0f)) lm_bad = 1;
      lm = fmaxf(lm, c);
    }
  }
  if (p.NP >= 16) {  // sel starts on a 16-byte boundary
    for (int q = threadIdx.x; q < p.NP / 16; q += NT) reinterpret_cast<int4*>(m.sel)[q] = int4{0, 0, 0, 0};
  } else if (threadIdx.x < p.NP) {
    m.sel[threadIdx.x] = 0;
  }
  reinterpret_cast<int4*>(m.cnt)[threadIdx.x] = int4{0, 0, 0, 0};  // kBuckets == 4 * NT
  if (threadIdx.x == 0) {
    sh.err = 0;
    sh.cmax = 0;
  }
  if (threadIdx.x < kMaxP) {
    sh.col_s[threadIdx.x] = 0ull;
    sh.col_n[threadIdx.x] = 0;
  }
  cp_async_wait_all();
  __syncthreads();

  // Current slots: lengths and offsets.
  int N = load_lengths(rc, cc, p.bs, nreq, p.k_max, m.lens, m.off, sh);

  int B = 0;
  int Ks = p.k_max;  // slots j < Ks of each draft, where no top-B mask applies
  if (!adaptive) {
    B = N;
  } else if (uniform) {
    if (sh.err == 0) {
      build_keys(p.conf, m.lens, m.off, nreq, p.P, m.keysA, m.cnt, sh);
      if (sh.err == 0)
        Ks = uniform_argmax(m.keysA, p.NP, p.P, p.k_max, min(N, L - p.T), p.bs, m.cm, lm, lm_bad,
                            sh, &B);
    }
  } else {
    if (p.budget_conf) {
      const int Nb = load_lengths(rb, cb, p.bs_budget, nb, p.k_max, m.lens, m.off, sh);
      if (sh.err == 0) {
        build_keys(p.budget_conf, m.lens, m.off, nb, p.P, m.keysA, m.cnt, sh);
        const unsigned long long* sorted = sort_keys(m, p.NPb, p.P, sh);
        const int Bmax_b = min(Nb, L - p.T);
        int Bb = 0;
        if (sh.err == 0)
          Bb = budget_argmax(sorted, sorted == m.keysA ? m.keysB : m.keysA, Bmax_b, p.bs, m.cm,
                             lm, lm_bad, sh);
        B = min(Bb, min(N, L - p.T));
      }
      // Back to the current request lengths.
      N = load_lengths(rc, cc, p.bs, nreq, p.k_max, m.lens, m.off, sh);
    }
    if (sh.err == 0) {
      build_keys(p.conf, m.lens, m.off, nreq, p.P, m.keysA, m.cnt, sh);
      const unsigned long long* sorted = sort_keys(m, p.NP, p.P, sh);
      if (!p.budget_conf && sh.err == 0)
        B = budget_argmax(sorted, sorted == m.keysA ? m.keysB : m.keysA, min(N, L - p.T), p.bs,
                          m.cm, lm, lm_bad, sh);
      // Selection: the B best ranks.
      if (sh.err == 0)
        for (int r = threadIdx.x; r < B; r += NT)
          m.sel[static_cast<uint32_t>(sorted[r] & 0xFFFFFFFFull)] = 1;
      __syncthreads();
    }
  }

  const bool failed = sh.err != 0;
  if (failed) B = 0;
  // Compaction: slot mask, n_i and cu_seqlens, one thread per chunk of requests.
  int nv[kReqPer], local = 0;
#pragma unroll
  for (int q = 0; q < kReqPer; ++q) nv[q] = 0;
#pragma unroll
  for (int q = 0; q < kReqPer; ++q) {
    const int i = cc.beg + q;
    if (i >= cc.end) break;
    const int k = failed ? 0 : m.lens[i];
    uint8_t* mrow = p.mask + static_cast<size_t>(i) * p.k_max;
    for (int j = 0; j < p.k_max; ++j) {
      const uint8_t v = j < k ? (adaptive && !uniform ? m.sel[i * p.P + j] : static_cast<uint8_t>(j < Ks))
                              : uint8_t{0};
      mrow[j] = v;
      nv[q] += v;
    }
    p.num_verified[i] = nv[q];
    local += nv[q] + 1;
  }
  int total;
  int run = block_scan_excl(local, sh.tot_i32, &total);
#pragma unroll
  for (int q = 0; q < kReqPer; ++q) {
    if (cc.beg + q >= cc.end) break;
    p.cu[cc.beg + q] = run;
    run += nv[q] + 1;
  }
  if (threadIdx.x == 0) {
    p.cu[p.bs] = total;
    p.B_out[0] = B;
    if (sh.err) raise_error(p.err, sh.err);
  }
}

// Online calibration of the per-position acceptance model a = sigmoid(w_j c
// + b_j), one CTA.
// apply = 0: one gradient step on the mean logistic loss of the slots the
//   step observed: slot (i, j) with j < num_verified[i] and j <=
//   accepted_len[i], label 1 below accepted_len[i] and 0 at it (the first
//   rejection); positions without observations keep their parameters.  One
//   thread per slot i * P + j as in the planner's key phase, so each thread
//   sees a single position; the per-position sums go through warp shuffles
//   and then over the warps in a fixed order in fp64, so the result does not
//   depend on timing.  The parameters are written after the last barrier and
//   only when no input check failed.
// apply = 1: conf_out[slot] = fma(w_j, c, b_j) for every drafted slot (may
//   be in place); nothing is written when a draft length is out of range.
__global__ void __launch_bounds__(NT, 1) calib_kernel(const CalibParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ PlanShared sh;
  __shared__ float part_e[NW][kMaxP];
  __shared__ float part_ec[NW][kMaxP];
  __shared__ int part_n[NW][kMaxP];
  const int nreq = p.NP / p.P;
  int* off = reinterpret_cast<int*>(smem);                               // [nreq + 1]
  uint8_t* lens = smem + static_cast<size_t>(nreq + 1) * sizeof(int);  // [nreq]
  const Chunk cc = req_chunk(p.bs);
  int rc[kReqPer];
  fetch_lengths(p.lens, cc, rc);
  if (threadIdx.x == 0) sh.err = 0;
  __syncthreads();
  load_lengths(rc, cc, p.bs, nreq, p.k_max, lens, off, sh);
  const bool ok = sh.err == 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lgP = 31 - __clz(p.P);
  const int j = static_cast<int>(threadIdx.x) & (p.P - 1);  // P divides NT
  float wj = 0.0f, bj = 0.0f;
  if (ok && j < p.k_max) {
    wj = p.w[j];
    bj = p.b[j];
  }
  float se = 0.0f, sec = 0.0f;
  int n = 0, bad = 0;
  if (ok && !p.apply) {  // every request's outcome, also those with no drafted slot
    for (int i = cc.beg; i < cc.end; ++i) {
      const int nv = p.nv[i], ac = p.acc[i];
      if (nv < 0 || nv > lens[i] || ac < 0 || ac > nv) bad |= SD_DEV_ERR_OUTCOME;
    }
  }
  if (ok) {
    for (int r = 0; r < kSlotPer; ++r) {
      const int q = r * NT + static_cast<int>(threadIdx.x);
      if (q >= p.NP) break;
      const int i = q >> lgP;
      if (i >= p.bs || j >= lens[i]) continue;
      const int at = off[i] + j;
      const float c = p.conf[at];
      if (p.apply) {
        p.conf_out[at] = fmaf(wj, c, bj);
        continue;
      }
      const int nv = p.nv[i], ac = p.acc[i];
      if (nv < 0 || nv > lens[i] || ac < 0 || ac > nv) {
        bad |= SD_DEV_ERR_OUTCOME;
        continue;
      }
      if (j >= min(nv, ac + 1)) continue;  // never tested
      if (!isfinite(c)) {
        bad |= SD_DEV_ERR_CONF;
        continue;
      }
      const float e = 1.0f / (1.0f + expf(-fmaf(wj, c, bj))) - (j < ac ? 1.0f : 0.0f);
      se += e;
      sec = fmaf(e, c, sec);
      ++n;
    }
  }
  if (p.apply) {  // uniform over the block: no barrier follows
    if (threadIdx.x == 0 && sh.err) raise_error(p.err, sh.err);
    return;
  }
  for (int o = p.P; o < 32; o <<= 1) {  // lanes with the same position
    se += __shfl_xor_sync(kFull, se, o);
    sec += __shfl_xor_sync(kFull, sec, o);
    n += __shfl_xor_sync(kFull, n, o);
  }
  if (lane < p.P) {
    part_e[warp][lane] = se;
    part_ec[warp][lane] = sec;
    part_n[warp][lane] = n;
  }
  if (bad) atomicOr(&sh.err, bad);
  __syncthreads();
  if (static_cast<int>(threadIdx.x) < p.k_max) {  // thread j holds w_j, b_j
    double E = 0.0, EC = 0.0;
    int m = 0;
    for (int v = 0; v < NW; ++v) {
      E += static_cast<double>(part_e[v][threadIdx.x]);
      EC += static_cast<double>(part_ec[v][threadIdx.x]);
      m += part_n[v][threadIdx.x];
    }
    if (sh.err == 0 && m > 0) {
      const double lr = static_cast<double>(p.lr);
      p.w[threadIdx.x] = static_cast<float>(static_cast<double>(wj) - lr * (EC / m));
      p.b[threadIdx.x] = static_cast<float>(static_cast<double>(bj) - lr * (E / m));
    }
  }
  if (threadIdx.x == 0 && sh.err) raise_error(p.err, sh.err);
}

}  // namespace

size_t plan_smem_bytes(const PlanParams& p) {
  return plan_layout(p.NP, p.NPb, p.P, nullptr, nullptr);
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

cudaError_t launch_calibrate(const CalibParams& p, cudaStream_t s) {
  const int nreq = p.NP / p.P;
  // offsets and lengths of the padded requests: at most 8193 * 4 + 8192 bytes
  const size_t smem = static_cast<size_t>(nreq + 1) * sizeof(int) + static_cast<size_t>(nreq);
  if (smem > 32 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        calib_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  calib_kernel<<<1, NT, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace sdk
