// sampler.cu -- the sampling stage (sd_verify): speculative rejection
// sampling over the whole vocabulary in one persistent kernel.
//
// Rule (the original papers cited by the fosworld blog "추측 디코딩과 vLLM
// 적응형 검증" under "참고 링크 / 논문"; greedy form in "추측 디코딩이란";
// distribution-preserving per "속도, 메모리, 정확도에 주는 영향", row 정확도):
//   tau > 0: accept slot j iff u_j * q_j(x_j) <= p_j(x_j); at the first
//            rejection draw from max(p - q, 0) normalised; after a fully
//            accepted prefix draw a bonus token from p of the next row.
//   tau = 0: accept iff x_j == argmax p_j; the correction/bonus is the argmax.
//
// Design (GB300).  Every logit row is cut into 8 KB segments.  The work list
// is ordered by slot position ("waves"): wave j holds, for every request that
// verifies slot j, its target row t_j and (tau > 0) its draft row d_j, then
// the rows t_j that are a request's bonus row, then greedy requests' rows.
// One persistent CTA per SM: a producer warp claims blocks of segments from a
// global counter and streams each segment with one bulk copy into a ring of
// shared-memory buffers; eight consumer warps take the buffers in order and
// reduce each segment to partial softmax statistics (or an argmax).  The
// consumer that counts a pair's last segment combines the pair's statistics
// and takes slot j's accept decision at once; the decision that settles a
// request (its first rejection with every earlier slot accepted, or a fully
// accepted prefix and its bonus row) lists the request's final draw.  The
// draw's row(s) were streamed moments before, so its sub-chunks are read
// again from L2, not HBM; their inverse-CDF weights are summed in exact
// 64-bit fixed point, and the consumer that counts the last sub-chunk finds
// the crossing sub-chunk and walks it.  With SD_VERIFY_EARLY_EXIT the
// producer skips rows of slots after a request's known first rejection.
//
// Precision.  Row statistics use the hardware base-2 exponent on an argument
// d * s2 with d = l - m exact and s2 = log2(e)/tau carried in two floats; the
// per-segment sums are compensated and combined in fp64.  A final draw's
// weights are fp32 except where an element weighs more than 2^-12 of its
// row's maximum: there the weight is formed in double-float from a 16-entry
// table of 2^(j/16) and a short series (Tang's table-driven method), so the
// elements that carry the distribution's mass match the fp64 definition to
// about 1e-10.
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>

#include "sd_device.cuh"
#include "sd_internal.h"

namespace sdk {

namespace {

constexpr int kNC = 8;                    // consumer warps per CTA
constexpr int kThreads = (kNC + 1) * 32;  // + the producer warp
constexpr int kMaxBufs = 24;              // ring buffers per CTA (at most)
constexpr int kRowBlock = 4;              // segments per row claim
constexpr int kSubBlock = 4;              // sub-chunks per draw claim
constexpr uint64_t kDrainNs = 2000000000ull;  // bound of the exit drain of in-flight copies (2 s)
constexpr uint32_t kPollHintNs = 10000;       // suspend hint of one poll of an mbarrier (10 us)
constexpr float kBigT = -12.0f;           // weights above 2^-12 of the row maximum: precise
constexpr float kTwo56 = 72057594037927936.0f;
constexpr float kTwo64 = 18446744073709551616.0f;
// log2(e) and ln(2), each split into two floats (hi + lo).
constexpr float kLog2eHi = 1.44269502162933349609375f;
constexpr float kLog2eLo = 1.925963033500011079e-08f;
constexpr float kLn2Hi = 0.693147182464599609375f;
constexpr float kLn2Lo = -1.904654299957768e-09f;
constexpr double kLog2eD = 1.4426950408889634074;

// Item kinds handed from the producer to the consumers.
enum { kEnd = 0, kRow = 1, kSkip = 2, kSub = 3 };
// Kinds of a final draw.
enum { kDrawResid = 0, kDrawP = 1 };

struct Desc {
  int kind;
  int a;  // kRow / kSkip: i | j << 12 | draft << 16;  kSub: draw index e
  int b;  // kRow: segment;  kSkip: segments skipped;  kSub: sub-chunk
  int c;  // kSub: the draw's list entry (1 + (i << 6 | a << 2 | kind))
};

// ---------------------------------------------------------------------------
// Memory-order and arithmetic helpers.

__device__ __forceinline__ int ld_relaxed(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ int atom_or_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.or.acq_rel.gpu.global.b32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Device-wide nanosecond clock: every wait below gives up after a bound in
// time, not in polls (one poll of an mbarrier may suspend the thread).
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// One poll of an mbarrier phase, suspending the thread at most ~hint ns.
__device__ __forceinline__ bool mbar_poll(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kPollHintNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Knuth's two-sum and the fast variant (|a| >= |b|): s + e = a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}

// s2 = log2(e) / tau as s2h + s2l with s2h rounded down, so s2l > 0 and an
// argument d * s2h + d * s2l of a masked element (d = -inf) stays -inf.
__device__ __forceinline__ void scale_of(float tau, float& s2h, float& s2l) {
  s2h = fminf(__fdiv_rd(kLog2eHi, tau), 3.0e38f);
  const float r = __fmaf_rn(-s2h, tau, kLog2eHi);  // exact remainder
  s2l = fmaxf(__fdiv_rn(__fadd_rn(r, kLog2eLo), tau), 1.0e-45f);
}

// Neumaier's compensated sum of non-negative terms.
__device__ __forceinline__ void comp_add(float& s, float& c, float x) {
  const float t = __fadd_rn(s, x);
  c = __fadd_rn(c, s >= x ? __fadd_rn(__fsub_rn(s, t), x) : __fadd_rn(__fsub_rn(x, t), s));
  s = t;
}

// 2^t for t = th + tl <= 0 in double-float (relative error ~1e-10), Tang's
// table-driven method: t = n + j/16 + r with |r| <= 1/32, 2^(j/16) from a
// table of (hi, lo) pairs, 2^r = e^x (x = r ln 2) from its series to x^5.
// Weights below 2^-120 are returned as 0.
__device__ __forceinline__ void exp2_precise(float th, float tl, const float2* tab, float& wh,
                                             float& wl) {
  if (!(th > -120.0f)) {
    wh = 0.0f;
    wl = 0.0f;
    return;
  }
  const float kf = rintf(__fmul_rn(th, 16.0f));
  const int k = __float2int_rn(kf);
  const int j = k & 15, n = k >> 4;  // k = 16 n + j
  const float r = __fadd_rn(__fsub_rn(th, __fmul_rn(kf, 0.0625f)), tl);
  const float xh = __fmul_rn(r, kLn2Hi);
  const float xl = __fadd_rn(__fmaf_rn(r, kLn2Hi, -xh), __fmul_rn(r, kLn2Lo));
  const float P = __fmaf_rn(xh, __fmaf_rn(xh, __fmaf_rn(xh, 1.0f / 120.0f, 1.0f / 24.0f), 1.0f / 6.0f),
                            0.5f);
  const float q = __fmaf_rn(__fmul_rn(xh, xh), P, xl);
  float sh, se;
  fast_two_sum(1.0f, xh, sh, se);
  const float sl = __fadd_rn(se, q);
  const float2 T = tab[j];
  const float ph = __fmul_rn(T.x, sh);
  const float pl = __fadd_rn(__fmaf_rn(T.x, sh, -ph), __fmaf_rn(T.x, sl, __fmul_rn(T.y, sh)));
  const float sc = __int_as_float((127 + n) << 23);  // 2^n, n >= -120
  wh = __fmul_rn(ph, sc);
  wl = __fmul_rn(pl, sc);
}

// ---------------------------------------------------------------------------
// Element types: a 16-byte vector is one "unit" of VE elements.

template <typename T>
struct ET;

template <>
struct ET<uint16_t> {  // bf16 bit patterns
  using V = uint4;
  static constexpr int VE = 8;
  __device__ __forceinline__ static void unpack(const uint4& r, float (&f)[8]) {
    f[0] = bf_lo(r.x); f[1] = bf_hi(r.x); f[2] = bf_lo(r.y); f[3] = bf_hi(r.y);
    f[4] = bf_lo(r.z); f[5] = bf_hi(r.z); f[6] = bf_lo(r.w); f[7] = bf_hi(r.w);
  }
  __device__ __forceinline__ static float vmax_nan(const uint4& r) {
    const uint32_t m = bmax2_nan(bmax2_nan(r.x, r.y), bmax2_nan(r.z, r.w));
    return fmax_nan(bf_lo(m), bf_hi(m));
  }
  __device__ __forceinline__ static float at(const void* base, long long k) {
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(base)[k]) << 16);
  }
  __device__ __forceinline__ static float ldg(const void* base, long long k) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(base) + k)) << 16);
  }
};

template <>
struct ET<float> {
  using V = float4;
  static constexpr int VE = 4;
  __device__ __forceinline__ static void unpack(const float4& r, float (&f)[4]) {
    f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w;
  }
  __device__ __forceinline__ static float vmax_nan(const float4& r) {
    return fmax_nan(fmax_nan(r.x, r.y), fmax_nan(r.z, r.w));
  }
  __device__ __forceinline__ static float at(const void* base, long long k) {
    return static_cast<const float*>(base)[k];
  }
  __device__ __forceinline__ static float ldg(const void* base, long long k) {
    return __ldg(static_cast<const float*>(base) + k);
  }
};

// Unit q (elements [q*VE, q*VE+VE)) of a region of n elements that starts at
// `src`: the staged shared-memory copy (vector path, n a multiple of VE), a
// global row read through L2 (`l2`), or single elements of a global row
// (element path; positions >= n read as -inf).
template <typename T, bool VEC>
__device__ __forceinline__ void load_unit(const void* src, int q, int n, bool l2,
                                          float (&f)[ET<T>::VE]) {
  using E = ET<T>;
  if constexpr (VEC) {
    const typename E::V* v = static_cast<const typename E::V*>(src) + q;
    if (l2) {
      if constexpr (sizeof(T) == 2) E::unpack(__ldcg(reinterpret_cast<const uint4*>(v)), f);
      else E::unpack(__ldcg(reinterpret_cast<const float4*>(v)), f);
    } else {
      E::unpack(*v, f);
    }
    (void)n;
  } else {
#pragma unroll
    for (int e = 0; e < E::VE; ++e) {
      const int k = q * E::VE + e;
      f[e] = k < n ? E::ldg(src, k) : -INFINITY;
    }
    (void)l2;
  }
}

// ---------------------------------------------------------------------------
// Final-draw weights.  A draw from p weighs element k with p_k; a residual
// draw with max(p_k - q_k, 0); in 2^56 fixed point.  A unit's value is the
// fixed-point value of the fp32 sum (in element order) of its elements that
// weigh less than 2^-12 of their row's maximum, plus the double-float value
// of each heavier element.  The sub-chunk sums and the walk of the crossing
// sub-chunk use these same functions, so the walk retraces the sums exactly.
struct DrawCtx {
  float Mt, Md, s2h, s2l;
  float izth, iztl, izdh, izdl;  // 1 / Z as (hi, lo)
  bool resid;
};

// fp32 weight of one element; *big when it must be formed precisely.
__device__ __forceinline__ float elem_fast(const DrawCtx& c, float lt, float ld, bool& big) {
  const float dt = __fsub_rn(lt, c.Mt);
  const float tt = __fmaf_rn(dt, c.s2h, __fmul_rn(dt, c.s2l));
  const float wt = exp2_ftz(tt);
  big = tt > kBigT;
  if (!c.resid) return __fmaf_rn(wt, c.izth, __fmul_rn(wt, c.iztl));
  const float dd = __fsub_rn(ld, c.Md);
  const float td = __fmaf_rn(dd, c.s2h, __fmul_rn(dd, c.s2l));
  const float wd = exp2_ftz(td);
  big = big || td > kBigT;
  const float qd = __fmaf_rn(wd, c.izdh, __fmul_rn(wd, c.izdl));
  return fmaxf(__fmaf_rn(wt, c.izth, __fmaf_rn(wt, c.iztl, -qd)), 0.0f);
}

// (w / Z) of one element in double-float from its logit l, row max M.
__device__ __forceinline__ void prob_precise(float l, float M, float s2h, float s2l, float izh,
                                             float izl, const float2* tab, float& ph, float& pl) {
  float dh, dl;
  two_sum(l, -M, dh, dl);
  const float th = __fmul_rn(dh, s2h);
  const float tl = __fadd_rn(__fmaf_rn(dh, s2h, -th), __fmaf_rn(dh, s2l, __fmul_rn(dl, s2h)));
  float wh, wl;
  exp2_precise(th, tl, tab, wh, wl);
  ph = __fmul_rn(wh, izh);
  pl = __fadd_rn(__fmaf_rn(wh, izh, -ph), __fmaf_rn(wh, izl, __fmul_rn(wl, izh)));
}

// Fixed-point weight of one heavy element.
__device__ __forceinline__ unsigned long long elem_precise(const DrawCtx& c, float lt, float ld,
                                                           const float2* tab) {
  float ph, pl;
  prob_precise(lt, c.Mt, c.s2h, c.s2l, c.izth, c.iztl, tab, ph, pl);
  if (c.resid) {
    float qh, ql;
    prob_precise(ld, c.Md, c.s2h, c.s2l, c.izdh, c.izdl, tab, qh, ql);
    float rh, re;
    two_sum(ph, -qh, rh, re);
    const float rl = __fadd_rn(re, __fsub_rn(pl, ql));
    fast_two_sum(rh, rl, ph, pl);  // |rl| small against rh unless both are tiny
  }
  if (!(ph > 0.0f)) return 0ull;
  const long long v = __float2ll_rn(__fmul_rn(ph, kTwo56)) + __float2ll_rn(__fmul_rn(pl, kTwo56));
  return v > 0 ? static_cast<unsigned long long>(v) : 0ull;
}

template <int VE>
__device__ __forceinline__ unsigned long long unit_fast(const DrawCtx& c, const float (&ft)[VE],
                                                        const float (&fd)[VE], uint32_t& bigm) {
  float s = 0.0f;
  bigm = 0;
#pragma unroll
  for (int e = 0; e < VE; ++e) {
    bool big;
    const float r = elem_fast(c, ft[e], fd[e], big);
    if (big) bigm |= 1u << e;
    else s = __fadd_rn(s, r);
  }
  return __float2ull_rn(__fmul_rn(s, kTwo56));
}

template <int VE>
__device__ __forceinline__ unsigned long long unit_value(const DrawCtx& c, const float (&ft)[VE],
                                                         const float (&fd)[VE], const float2* tab) {
  uint32_t bm;
  unsigned long long v = unit_fast<VE>(c, ft, fd, bm);
#pragma unroll
  for (int e = 0; e < VE; ++e)
    if ((bm >> e) & 1u) v += elem_precise(c, ft[e], fd[e], tab);
  return v;
}

// ---------------------------------------------------------------------------
// Per-CTA context: the work-list tables built in the prologue.

struct Cta {
  const int* order;  // [bs]: sampling requests by n desc, then greedy ones by n desc
  const int* WS;     // [nw+1] first unit of wave j
  const int* Pj;     // [nw] sampling requests with n > j
  const int* Ej;     // [nw] sampling requests with n == j
  int nsamp, nw, U, BPU, BPD;
  const float2* tab;  // shared-memory copy of the exponent table
};

struct Loc {
  int i, j, isd;
};

__device__ __forceinline__ Loc locate(const Cta& C, int u) {
  int j = 0;
  while (j + 1 < C.nw && C.WS[j + 1] <= u) ++j;
  const int r = u - C.WS[j];
  const int P = C.Pj[j], E = C.Ej[j];
  Loc L;
  L.j = j;
  if (r < 2 * P) {
    L.i = C.order[r >> 1];
    L.isd = r & 1;
  } else if (r < 2 * P + E) {
    L.i = C.order[P + (r - 2 * P)];
    L.isd = 0;
  } else {
    L.i = C.order[C.nsamp + (r - 2 * P - E)];
    L.isd = 0;
  }
  return L;
}

// Temperature of request i as the kernel uses it: invalid values and
// sampling without draft logits fall back to greedy (flagged in the prologue).
__device__ __forceinline__ float eff_tau(const SamplerParams& p, int i) {
  const float t = __ldg(p.temps + i);
  return (t > 0.0f && isfinite(t) && p.draft != nullptr) ? t : 0.0f;
}

__device__ __forceinline__ long long trow_of(const SamplerParams& p, int i, int j) {
  return static_cast<long long>(__ldg(p.cu + i)) + j;
}
__device__ __forceinline__ long long drow_of(const SamplerParams& p, int i, int j) {
  return (p.flags & kFlagDraftPadded) ? static_cast<long long>(i) * p.k_max + j
                                      : static_cast<long long>(__ldg(p.cu + i)) - i + j;
}
__device__ __forceinline__ int n_of(const SamplerParams& p, int i) {
  return __ldg(p.cu + i + 1) - __ldg(p.cu + i) - 1;
}

// Request state: bit j (j < 15) slot j accepted, bit 15 the bonus row's
// statistics are in, bit 16 + j slot j rejected.  Returns the accepted
// length once the state settles the request, else -1.
__device__ __forceinline__ int settled(int s, int n) {
  const uint32_t A = static_cast<uint32_t>(s) & 0x7FFFu;
  const uint32_t R = (static_cast<uint32_t>(s) >> 16) & 0x7FFFu;
  if (R) {
    const int a = __ffs(R) - 1;
    const uint32_t need = (1u << a) - 1u;
    return (A & need) == need ? a : -1;
  }
  const uint32_t need = (1u << n) - 1u;
  return ((A & need) == need && (s & 0x8000)) ? n : -1;
}

// ---------------------------------------------------------------------------
// The kernel.

template <typename T, bool VEC>
struct Sampler {
  using E = ET<T>;
  static constexpr int VE = E::VE;
  static constexpr int kSegE = kSegBytes / static_cast<int>(sizeof(T));  // elements per segment
  static constexpr int kSubE = kSubBytes / static_cast<int>(sizeof(T));  // elements per sub-chunk
  static constexpr int kUPL = kSubE / VE / 32;                           // sub-chunk units per lane

  const SamplerParams& p;
  const Cta& C;
  unsigned char* ring;
  uint64_t* full;
  uint64_t* empty;
  Desc* desc;
  int* ticket;
  volatile int* seen;  // [nbuf] phases of each buffer whose wait has passed
  volatile int* stop;
  int lane;

  __device__ size_t row_bytes() const { return static_cast<size_t>(p.V) * sizeof(T); }
  __device__ const char* trow_ptr(long long r) const {
    return static_cast<const char*>(p.target) + static_cast<size_t>(r) * row_bytes();
  }
  __device__ const char* drow_ptr(long long r) const {
    return static_cast<const char*>(p.draft) + static_cast<size_t>(r) * row_bytes();
  }

  __device__ void halt() const {
    if (lane == 0) {
      raise_error(p.err, SD_DEV_ERR_TIMEOUT);
      atomicExch(p.ctrl + kCtlStop, 1);
      *stop = 1;
    }
  }

  // ---- consumer: one segment of a row --------------------------------------
  // Writes the segment's record; returns nothing (the caller counts it).
  __device__ void segment(const void* src, int n_el, bool greedy, float tau, int xo,
                          SegRec* rec, int e0) const {
    const int nu = (n_el + VE - 1) / VE;
    SegRec out;
    out.lx = 0.0f;
    if (greedy) {
      float best = -INFINITY;
      int bidx = INT_MAX, bad = 0;
      for (int q = lane; q < nu; q += 32) {
        float f[VE];
        float vm;
        if constexpr (VEC) {
          const typename E::V raw = static_cast<const typename E::V*>(src)[q];
          vm = E::vmax_nan(raw);
          if (vm > best) {
            E::unpack(raw, f);
            int e = VE - 1;
#pragma unroll
            for (int k = VE - 1; k >= 0; --k)
              if (f[k] == vm) e = k;
            best = vm;
            bidx = q * VE + e;
          }
        } else {
          load_unit<T, false>(src, q, n_el, false, f);
          vm = f[0];
#pragma unroll
          for (int k = 1; k < VE; ++k) vm = fmax_nan(vm, f[k]);
          if (vm > best) {
            int e = VE - 1;
#pragma unroll
            for (int k = VE - 1; k >= 0; --k)
              if (f[k] == vm) e = k;
            best = vm;
            bidx = q * VE + e;
          }
        }
        bad |= (vm != vm) | (vm == INFINITY);
      }
      unsigned long long key = bidx == INT_MAX ? 0ull
          : (static_cast<unsigned long long>(ordered_bits(best)) << 32) |
                static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(bidx));
      key = warp_max_u64(key);
      bad = __any_sync(kFull, bad);
      out.m = key ? __uint_as_float((static_cast<uint32_t>(key >> 32) & 0x80000000u)
                                        ? (static_cast<uint32_t>(key >> 32) & 0x7FFFFFFFu)
                                        : ~static_cast<uint32_t>(key >> 32))
                  : -INFINITY;
      out.w2 = key ? static_cast<uint32_t>(e0) + (0xFFFFFFFFu - static_cast<uint32_t>(key)) : 0u;
      out.w3 = bad ? 1u : 0u;
    } else {
      float vm = -INFINITY;
      for (int q = lane; q < nu; q += 32) {
        if constexpr (VEC) {
          vm = fmax_nan(vm, E::vmax_nan(static_cast<const typename E::V*>(src)[q]));
        } else {
          float f[VE];
          load_unit<T, false>(src, q, n_el, false, f);
#pragma unroll
          for (int k = 0; k < VE; ++k) vm = fmax_nan(vm, f[k]);
        }
      }
      const float m = warp_max_nan(vm);
      double z = 0.0;
      if (isfinite(m)) {
        float s2h, s2l;
        scale_of(tau, s2h, s2l);
        float ks = 0.0f, kc = 0.0f;
        for (int q = lane; q < nu; q += 32) {
          float f[VE];
          load_unit<T, VEC>(src, q, n_el, false, f);
          float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int k = 0; k < VE; k += 2) {
            const float2 d = __fadd2_rn(make_float2(f[k], f[k + 1]), make_float2(-m, -m));
            const float2 t = __ffma2_rn(d, make_float2(s2h, s2h),
                                        __fmul2_rn(d, make_float2(s2l, s2l)));
            acc = __fadd2_rn(acc, make_float2(exp2_ftz(t.x), exp2_ftz(t.y)));
          }
          comp_add(ks, kc, __fadd_rn(acc.x, acc.y));
        }
        z = warp_sum_f64(static_cast<double>(ks) + static_cast<double>(kc));
      }
      out.m = m;
      const unsigned long long zb = static_cast<unsigned long long>(__double_as_longlong(z));
      out.w2 = static_cast<uint32_t>(zb);
      out.w3 = static_cast<uint32_t>(zb >> 32);
    }
    if (lane == 0) {
      if (xo >= 0 && xo < n_el) {
        if constexpr (VEC) out.lx = E::at(src, xo);
        else out.lx = E::ldg(src, xo);
      }
      __stcg(reinterpret_cast<uint4*>(rec), *reinterpret_cast<const uint4*>(&out));
    }
  }

  // ---- consumer: pair (i, j) complete -----------------------------------
  // Combines a row's segment records: max M (NaN/+inf/no finite value ->
  // bad), Z in fp64, lx, and the lowest argmax (greedy).
  __device__ void combine(const SegRec* recs, bool greedy, double s2d, int xseg, float& M,
                          double& Z, float& lx, int& amax, int& bad) const {
    float mv = -INFINITY;
    int b = 0;
    unsigned long long key = 0ull;
    for (int s = lane; s < p.nseg; s += 32) {
      const uint4 r = __ldcg(reinterpret_cast<const uint4*>(recs + s));
      const float m = __uint_as_float(r.x);
      b |= (m != m) | (m == INFINITY);
      if (greedy) {
        b |= r.w != 0u;
        if (m != -INFINITY && m == m)
          key = max(key, (static_cast<unsigned long long>(ordered_bits(m)) << 32) |
                             static_cast<unsigned long long>(0xFFFFFFFFu - r.z));
      }
      mv = fmaxf(mv, m);
    }
    b = __any_sync(kFull, b);
    M = warp_max(mv);
    if (M == -INFINITY) b = 1;
    bad = b;
    amax = -1;
    if (greedy) {
      key = warp_max_u64(key);
      amax = key ? static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key)) : -1;
      Z = 1.0;
    } else {
      double z = 0.0;
      if (!b) {
        for (int s = lane; s < p.nseg; s += 32) {
          const uint4 r = __ldcg(reinterpret_cast<const uint4*>(recs + s));
          const float m = __uint_as_float(r.x);
          if (m != -INFINITY) {
            const double zs = __longlong_as_double(static_cast<long long>(
                (static_cast<unsigned long long>(r.w) << 32) | r.z));
            z += zs * exp2((static_cast<double>(m) - static_cast<double>(M)) * s2d);
          }
        }
      }
      Z = warp_sum_f64(z);
    }
    lx = 0.0f;
    if (xseg >= 0) lx = __uint_as_float(__ldcg(reinterpret_cast<const unsigned int*>(recs + xseg) + 1));
  }

  // Writes every output of request i except a residual or bonus draw's
  // token (written by the draw's finish); counts one event of request i
  // and the request as done when `done`.
  __device__ void write_prefix(int i, int a, int y, bool write_y) const {
    const int k1 = p.k_max + 1;
    int* o = p.out_tokens + static_cast<size_t>(i) * k1;
    for (int j = lane; j < k1; j += 32) {
      if (j < a) o[j] = __ldg(p.draft_ids + drow_of(p, i, j));
      else if (j > a) o[j] = -1;
      else if (write_y) o[j] = y;
    }
    if (lane == 0) p.accepted_len[i] = a;
  }

  // Event of request i (pair decisions and the final token): the last one
  // resets the request's words for the next call.
  __device__ void event(int i, int n, int count) const {
    if (lane == 0) {
      const int old = atom_add_acq_rel(p.ev + i, count);
      if (old + count == n + 2) {
        p.st[i] = 0;
        p.ev[i] = 0;
      }
    }
  }

  __device__ void request_done(int i, int n) const {
    __syncwarp();
    if (lane == 0) red_release_add(p.ctrl + kCtlReqDone, 1);
    event(i, n, 1);
  }

  __device__ static void red_release_add(int* q, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(q), "r"(v) : "memory");
  }

  // `skipped`: early exit dropped some of the pair's segments (its slot is
  // after the request's first rejection), so it has no statistics.
  __device__ void pair_finish(int i, int j, bool skipped) const {
    const int n = n_of(p, i);
    const float tau = eff_tau(p, i);
    const bool greedy = !(tau > 0.0f);
    const bool has_d = !greedy && j < n;
    const int pid = i * (p.k_max + 1) + j;
    int bits = 0;
    int xseg = -1, x = -1;
    bool x_ok = false;
    if (j < n) {
      x = __ldg(p.draft_ids + drow_of(p, i, j));
      x_ok = x >= 0 && x < p.V;
      if (x_ok) xseg = x / kSegE;
    }
    if (!skipped) {
      const double s2d = greedy ? 0.0 : kLog2eD / static_cast<double>(tau);
      float Mt, Md = 0.0f, lxt, lxd = 0.0f;
      double Zt, Zd = 1.0;
      int amax, badt, badd = 0, dummy;
      combine(p.seg_t + static_cast<size_t>(trow_of(p, i, j)) * p.nseg, greedy, s2d, xseg, Mt, Zt,
              lxt, amax, badt);
      if (has_d)
        combine(p.seg_d + static_cast<size_t>(drow_of(p, i, j)) * p.nseg, false, s2d, xseg, Md, Zd,
                lxd, dummy, badd);
      const int bad = badt | badd;
      if (lane == 0) {
        PairStat ps;
        ps.Mt = Mt;
        ps.Md = Md;
        ps.amax = amax;
        ps.bad = bad;
        ps.Zt = Zt;
        ps.Zd = Zd;
        __stcg(reinterpret_cast<uint4*>(p.ps + pid), *reinterpret_cast<const uint4*>(&ps));
        __stcg(reinterpret_cast<uint4*>(p.ps + pid) + 1, *(reinterpret_cast<const uint4*>(&ps) + 1));
        if (bad) raise_error(p.err, SD_DEV_ERR_LOGITS);
        if (j < n && !x_ok) raise_error(p.err, SD_DEV_ERR_DRAFT_ID);
        if (j == n) {
          bits = 0x8000;  // the bonus row is in
        } else if (greedy) {
          const bool acc = !bad && x_ok && x == amax;
          bits = acc ? (1 << j) : (1 << (16 + j));
        } else {
          bool acc = false;
          float pf = 0.0f, qf = 0.0f;
          const float u = p.uniforms[static_cast<size_t>(i) * (p.k_max + 1) + j];
          if (!(u >= 0.0f && u < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
          if (!bad && x_ok) {
            // p(x) = 2^((lx - M) s2) / Z in fp64, rounded to fp32; the
            // comparison u * q <= p is taken in fp32 on those values
            pf = static_cast<float>(
                exp2((static_cast<double>(lxt) - static_cast<double>(Mt)) * s2d) / Zt);
            qf = static_cast<float>(
                exp2((static_cast<double>(lxd) - static_cast<double>(Md)) * s2d) / Zd);
            acc = __fmul_rn(u, qf) <= pf;
          }
          if (p.probs_out) {
            const size_t dr = static_cast<size_t>(drow_of(p, i, j));
            p.probs_out[2 * dr] = pf;
            p.probs_out[2 * dr + 1] = qf;
          }
          bits = acc ? (1 << j) : (1 << (16 + j));
        }
      }
    }
    // reset the pair's counter for the next call (every segment was counted)
    if (lane == 0) p.pc[pid] = 0;
    int old = 0;
    if (lane == 0 && bits) old = atom_or_acq_rel(p.st + i, bits);
    old = __shfl_sync(kFull, old, 0);
    bits = __shfl_sync(kFull, bits, 0);
    const int now = settled(old | bits, n);
    const bool settles = bits && settled(old, n) < 0 && now >= 0;
    if (settles) settle(i, n, now, greedy);
    event(i, n, 1);
  }

  // Request i has its accepted length a: write the outputs, or list its draw.
  __device__ void settle(int i, int n, int a, bool greedy) const {
    const int pid = i * (p.k_max + 1) + a;
    const uint4 w0 = __ldcg(reinterpret_cast<const uint4*>(p.ps + pid));
    const int amax = static_cast<int>(w0.z);
    const int bad = static_cast<int>(w0.w);
    if (greedy) {
      write_prefix(i, a, bad || amax < 0 ? 0 : amax, true);
      request_done(i, n);
      return;
    }
    if (bad) {  // flagged already; a well-formed token
      write_prefix(i, a, 0, true);
      request_done(i, n);
      return;
    }
    write_prefix(i, a, 0, false);
    __syncwarp();
    list_draw(i, a, a < n ? kDrawResid : kDrawP);
  }

  __device__ void list_draw(int i, int a, int kind) const {
    if (lane == 0) {
      const int e = atomicAdd(p.ctrl + kCtlDraws, 1);
      st_release(p.dl + e, 1 + ((i << 6) | (a << 2) | kind));
    }
  }

  // ---- consumer: draws ----------------------------------------------------
  __device__ DrawCtx draw_ctx(int i, int a, int kind) const {
    const int pid = i * (p.k_max + 1) + a;
    const uint4 w0 = __ldcg(reinterpret_cast<const uint4*>(p.ps + pid));
    const uint4 w1 = __ldcg(reinterpret_cast<const uint4*>(p.ps + pid) + 1);
    const double Zt = __longlong_as_double(static_cast<long long>((static_cast<unsigned long long>(w1.y) << 32) | w1.x));
    const double Zd = __longlong_as_double(static_cast<long long>((static_cast<unsigned long long>(w1.w) << 32) | w1.z));
    DrawCtx c;
    c.Mt = __uint_as_float(w0.x);
    c.Md = __uint_as_float(w0.y);
    scale_of(eff_tau(p, i), c.s2h, c.s2l);
    const double izt = 1.0 / Zt, izd = 1.0 / Zd;
    c.izth = static_cast<float>(izt);
    c.iztl = static_cast<float>(izt - static_cast<double>(c.izth));
    c.izdh = static_cast<float>(izd);
    c.izdl = static_cast<float>(izd - static_cast<double>(c.izdh));
    c.resid = kind == kDrawResid;
    return c;
  }

  // Fixed-point sum of sub-chunk s of draw (i, a, kind); the data is in the
  // staged buffer `buf` (vector path) or read from the rows (element path).
  __device__ unsigned long long sub_sum(const DrawCtx& c, const void* tsrc, const void* dsrc,
                                        int n_el) const {
    const int nu = (n_el + VE - 1) / VE;
    unsigned long long acc = 0ull;
    uint64_t bigm = 0ull;
#pragma unroll
    for (int k = 0; k < kUPL; ++k) {
      const int q = lane + 32 * k;
      if (q < nu) {
        float ft[VE], fd[VE];
        load_unit<T, VEC>(tsrc, q, n_el, false, ft);
        if (c.resid) load_unit<T, VEC>(dsrc, q, n_el, false, fd);
        else {
#pragma unroll
          for (int e = 0; e < VE; ++e) fd[e] = 0.0f;
        }
        uint32_t bm;
        acc += unit_fast<VE>(c, ft, fd, bm);
        bigm |= static_cast<uint64_t>(bm) << (k * VE);
      }
    }
    while (bigm) {
      const int bit = __ffsll(static_cast<long long>(bigm)) - 1;
      bigm &= bigm - 1;
      const int q = lane + 32 * (bit / VE);
      const int k = q * VE + bit % VE;
      const float lt = VEC ? E::at(tsrc, k) : E::ldg(tsrc, k);
      const float ld = c.resid ? (VEC ? E::at(dsrc, k) : E::ldg(dsrc, k)) : 0.0f;
      acc += elem_precise(c, lt, ld, C.tab);
    }
    return warp_sum_u64(acc);
  }

  // Finish of draw e (every sub-chunk summed): threshold floor(u * S), the
  // crossing sub-chunk, then the walk of its units and elements.
  __device__ void finish(int e, int i, int a, int kind) const {
    const int n = n_of(p, i);
    const unsigned long long* rs = p.rs + static_cast<size_t>(e) * p.nsub;
    const int spl = (p.nsub + 31) / 32;
    const int b0 = min(p.nsub, lane * spl), b1 = min(p.nsub, b0 + spl);
    unsigned long long ls = 0ull;
    for (int s = b0; s < b1; ++s) ls += __ldcg(rs + s);
    // inclusive scan over lanes
    unsigned long long inc = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    const unsigned long long S = __shfl_sync(kFull, inc, 31);
    const float u = p.uniforms[static_cast<size_t>(i) * (p.k_max + 1) + p.k_max];
    if (lane == 0 && !(u >= 0.0f && u < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
    if (S == 0ull) {
      if (kind == kDrawResid) {  // no residual mass in fp32: draw from p of the same row
        __syncwarp();
        if (lane == 0) p.dc[e] = 0;
        list_draw(i, a, kDrawP);
        if (lane == 0) p.dl[e] = 0;
        return;
      }
      if (lane == 0) raise_error(p.err, SD_DEV_ERR_LOGITS);
      finish_token(e, i, n, a, 0);
      return;
    }
    const float uc = fminf(fmaxf(u, 0.0f), 0.99999994f);
    const unsigned long long th = __umul64hi(__float2ull_rn(__fmul_rn(uc, kTwo64)), S);
    // the lane whose block holds the crossing
    const unsigned hit = __ballot_sync(kFull, inc > th);
    const int L = __ffs(hit) - 1;  // exists: inc[31] = S > th
    unsigned long long before = __shfl_sync(kFull, inc - ls, L);
    int c = 0;
    if (lane == L) {
      c = b1 - 1;
      unsigned long long run = before;
      for (int s = b0; s < b1; ++s) {
        const unsigned long long v = __ldcg(rs + s);
        if (run + v > th) {
          c = s;
          break;
        }
        run += v;
      }
      before = run;
    }
    c = __shfl_sync(kFull, c, L);
    before = __shfl_sync(kFull, before, L);
    const int y = walk(draw_ctx(i, a, kind), i, a, kind, c, th - before);
    finish_token(e, i, n, a, y);
  }

  __device__ void finish_token(int e, int i, int n, int a, int y) const {
    if (lane == 0) {
      p.out_tokens[static_cast<size_t>(i) * (p.k_max + 1) + a] = y;
      p.dl[e] = 0;
      p.dc[e] = 0;
    }
    request_done(i, n);
  }

  // The element of sub-chunk c where the running weight passes th (from the
  // sub-chunk's start); past the last element's weight, the last positive one.
  __device__ int walk(const DrawCtx& c, int i, int a, int kind, int sc, unsigned long long th) const {
    const int k0 = sc * kSubE;
    const int n_el = min(kSubE, p.V - k0);
    const int nu = (n_el + VE - 1) / VE;
    const char* tb = trow_ptr(trow_of(p, i, a)) + static_cast<size_t>(k0) * sizeof(T);
    const char* db = c.resid ? drow_ptr(drow_of(p, i, a)) + static_cast<size_t>(k0) * sizeof(T) : tb;
    (void)kind;
    unsigned long long v[kUPL];
    unsigned long long ls = 0ull;
    int lastu = -1;
#pragma unroll
    for (int k = 0; k < kUPL; ++k) {
      const int q = lane * kUPL + k;
      v[k] = 0ull;
      if (q < nu) {
        float ft[VE], fd[VE];
        load_unit<T, VEC>(tb, q, n_el, true, ft);
        if (c.resid) load_unit<T, VEC>(db, q, n_el, true, fd);
        else {
#pragma unroll
          for (int e = 0; e < VE; ++e) fd[e] = 0.0f;
        }
        v[k] = unit_value<VE>(c, ft, fd, C.tab);
        if (v[k]) lastu = q;
      }
      ls += v[k];
    }
    unsigned long long inc = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    const unsigned hit = __ballot_sync(kFull, inc > th);
    int q = -1;
    unsigned long long rem = 0ull;
    if (hit) {
      const int L = __ffs(hit) - 1;
      if (lane == L) {
        unsigned long long run = inc - ls;
        q = lane * kUPL + kUPL - 1;
#pragma unroll
        for (int k = 0; k < kUPL; ++k) {
          if (q == lane * kUPL + kUPL - 1 && run + v[k] > th) {
            q = lane * kUPL + k;
            rem = th - run;
          }
          run += v[k];
        }
      }
      q = __shfl_sync(kFull, q, L);
      rem = __shfl_sync(kFull, rem, L);
    } else {
      q = __reduce_max_sync(kFull, static_cast<unsigned>(lastu + 1)) - 1;
      rem = ~0ull;
      if (q < 0) return k0;
    }
    // elements of unit q, each with its own fixed-point weight
    int pick = -1;
    if (lane == 0) {
      float ft[VE], fd[VE];
      load_unit<T, VEC>(tb, q, n_el, true, ft);
      if (c.resid) load_unit<T, VEC>(db, q, n_el, true, fd);
      else {
#pragma unroll
        for (int e = 0; e < VE; ++e) fd[e] = 0.0f;
      }
      unsigned long long run = 0ull;
      int last = -1;
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        bool big;
        const float r = elem_fast(c, ft[e], fd[e], big);
        const unsigned long long w = big ? elem_precise(c, ft[e], fd[e], C.tab)
                                         : __float2ull_rn(__fmul_rn(r, kTwo56));
        if (w > 0ull) last = e;
        if (pick < 0 && run + w > rem) pick = e;
        run += w;
      }
      if (pick < 0) pick = last >= 0 ? last : 0;
      pick = k0 + q * VE + pick;
    }
    return __shfl_sync(kFull, pick, 0);
  }

  // ---- consumer loop ---------------------------------------------------------
  __device__ bool wait_full(int b, uint32_t par) const {
    if (mbar_poll(&full[b], par)) return true;
    const uint64_t end = now_ns() + p.wait_ns;
    for (;;) {
      if (mbar_poll(&full[b], par)) return true;
      if (*stop || now_ns() > end) return false;
    }
  }

  // Ticket t is phase m = t / nbuf of buffer b = t % nbuf.  A consumer can
  // run a whole ring ahead of a slow copy (the items between may complete at
  // once), and a parity wait on phase m while phase m - 1 is still pending
  // would return on phase m - 2.  So the consumer first waits until the
  // consumer of phase m - 1 has passed its own wait.
  __device__ bool wait_turn(int b, int m) const {
    if (seen[b] >= m) return true;
    const uint64_t end = now_ns() + p.wait_ns;
    for (;;) {
      if (seen[b] >= m) return true;
      if (*stop || now_ns() > end) return false;
      __nanosleep(32);
    }
  }

  __device__ void consume() const {
    for (;;) {
      int t = 0;
      if (lane == 0) t = atomicAdd(ticket, 1);
      t = __shfl_sync(kFull, t, 0);
      const int b = t % p.nbuf;
      const int m = t / p.nbuf;
      bool ok = false;
      if (lane == 0) {
        ok = wait_turn(b, m) && wait_full(b, static_cast<uint32_t>(m) & 1u);
        if (ok) seen[b] = m + 1;
      }
      ok = __shfl_sync(kFull, ok, 0);
      if (!ok) {
        halt();
        return;
      }
      __syncwarp();  // lane 0's wait (acquire) covers the warp's reads
      const Desc d = desc[b];
      if (d.kind == kEnd) return;
      const void* buf = ring + static_cast<size_t>(b) * kSegBytes;
      if (d.kind == kRow || d.kind == kSkip) {
        const int i = d.a & 0xFFF, j = (d.a >> 12) & 0xF, isd = (d.a >> 16) & 1;
        const int n = n_of(p, i);
        const float tau = eff_tau(p, i);
        const bool greedy = !(tau > 0.0f);
        const int pid = i * (p.k_max + 1) + j;
        // One atomic counts the item: its segments, and (a skip item) one
        // unit at bit 16, so the count that completes the pair also says
        // whether any of its segments were dropped.
        int add = 1;
        if (d.kind == kRow) {
          const int s = d.b;
          const int e0 = s * kSegE;
          const int n_el = min(kSegE, p.V - e0);
          int xo = -1;
          if (j < n) {
            const int x = __ldg(p.draft_ids + drow_of(p, i, j));
            if (x >= e0 && x < e0 + n_el) xo = x - e0;
          }
          const long long r = isd ? drow_of(p, i, j) : trow_of(p, i, j);
          const void* src = VEC ? buf : static_cast<const void*>((isd ? drow_ptr(r) : trow_ptr(r)) +
                                                                 static_cast<size_t>(e0) * sizeof(T));
          SegRec* rec = (isd ? p.seg_d : p.seg_t) + static_cast<size_t>(r) * p.nseg + s;
          segment(src, n_el, greedy, tau, xo, rec, e0);
        } else {
          add = d.b + (1 << 16);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[b]);
        const int total = p.nseg * ((!greedy && j < n) ? 2 : 1);
        int now = 0;
        if (lane == 0) now = atom_add_acq_rel(p.pc + pid, add) + add;
        now = __shfl_sync(kFull, now, 0);
        if ((now & 0xFFFF) == total) {
          __syncwarp();
          pair_finish(i, j, (now >> 16) != 0);
        }
      } else {  // kSub
        const int e = d.a, s = d.b;
        const int code = d.c - 1;
        const int i = (code >> 6) & 0xFFF, a = (code >> 2) & 0xF, kind = code & 3;
        const DrawCtx c = draw_ctx(i, a, kind);
        const int k0 = s * kSubE;
        const int n_el = min(kSubE, p.V - k0);
        const void* tsrc;
        const void* dsrc;
        if constexpr (VEC) {
          tsrc = buf;
          dsrc = static_cast<const char*>(buf) + kSubBytes;
        } else {
          tsrc = trow_ptr(trow_of(p, i, a)) + static_cast<size_t>(k0) * sizeof(T);
          dsrc = c.resid ? static_cast<const void*>(drow_ptr(drow_of(p, i, a)) + static_cast<size_t>(k0) * sizeof(T))
                         : tsrc;
        }
        const unsigned long long sum = sub_sum(c, tsrc, dsrc, n_el);
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty[b]);
          __stcg(p.rs + static_cast<size_t>(e) * p.nsub + s, sum);
        }
        __syncwarp();
        int old = 0;
        if (lane == 0) old = atom_add_acq_rel(p.dc + e, 1);
        old = __shfl_sync(kFull, old, 0);
        if (old == p.nsub - 1) {
          __syncwarp();
          finish(e, i, a, kind);
        }
      }
    }
  }

  // ---- producer (lane 0 of the producer warp) ------------------------------
  struct Prod {
    int k = 0;             // items published
    bool rows_done = false;
    int held = -1;         // a claimed draw block whose draw is not listed yet
    int rb_next = -1;      // the next row block, claimed one step ahead
    // the row block in hand
    int seg = 0, seg_end = 0;
    Loc loc{};
    long long row = 0;
    bool greedy = false;
  };

  // Waits until buffer b may be refilled for item k.
  __device__ bool wait_empty(int k) const {
    if (k < p.nbuf) return true;
    const int b = k % p.nbuf;
    const uint32_t par = static_cast<uint32_t>(k / p.nbuf - 1) & 1u;
    if (mbar_poll(&empty[b], par)) return true;
    const uint64_t end = now_ns() + p.wait_ns;
    for (;;) {
      if (mbar_poll(&empty[b], par)) return true;
      if (*stop || now_ns() > end) return false;
    }
  }

  __device__ bool publish(Prod& P, const Desc& d, const char* src0, uint32_t bytes0,
                          const char* src1, uint32_t bytes1, bool evict) const {
    if (!wait_empty(P.k)) return false;
    const int b = P.k % p.nbuf;
    desc[b] = d;
    unsigned char* dst = ring + static_cast<size_t>(b) * kSegBytes;
    if (VEC && (bytes0 + bytes1) > 0) {
      mbar_arrive_expect_tx(&full[b], bytes0 + bytes1);
      const uint64_t pol = evict ? policy_evict_first() : policy_evict_normal();
      if (bytes0) bulk_load(dst, src0, bytes0, &full[b], pol);
      if (bytes1) bulk_load(dst + kSubBytes, src1, bytes1, &full[b], pol);
    } else {
      mbar_arrive(&full[b]);
    }
    ++P.k;
    return true;
  }

  __device__ static uint64_t policy_evict_normal() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
  }

  // Takes the next row block into P (returns 1), or finds the rows done
  // (0), or gives up on a wait (-1).  A block that early exit drops is
  // handed out as one skip item and never left in P.
  __device__ int next_row_block(Prod& P) const {
    const int total = C.U * C.BPU;
    for (;;) {
      const int rb = P.rb_next;
      if (rb < 0 || rb >= total || (p.flags & kFlagTestStall)) {
        P.rows_done = true;
        P.seg = P.seg_end = 0;
        return 0;
      }
      P.rb_next = atomicAdd(p.ctrl + kCtlRowBlk, 1);  // one step ahead
      const int u = rb / C.BPU, g = rb - u * C.BPU;
      P.loc = locate(C, u);
      P.seg = g * kRowBlock;
      P.seg_end = min(p.nseg, P.seg + kRowBlock);
      const int i = P.loc.i, j = P.loc.j;
      P.greedy = !(eff_tau(p, i) > 0.0f);
      P.row = P.loc.isd ? drow_of(p, i, j) : trow_of(p, i, j);
      if (p.flags & kFlagEarlyExit) {
        const int a = settled(ld_relaxed(p.st + i), n_of(p, i));
        if (a >= 0 && j > a) {  // after the request's first rejection: not needed
          Desc d{kSkip, i | (j << 12) | (P.loc.isd << 16), P.seg_end - P.seg, 0};
          P.seg = P.seg_end = 0;
          if (!publish(P, d, nullptr, 0, nullptr, 0, false)) return -1;
          continue;
        }
      }
      return 1;
    }
  }

  __device__ void produce() const {
    Prod P;
    P.rb_next = atomicAdd(p.ctrl + kCtlRowBlk, 1);
    const size_t rbytes = row_bytes();
    uint64_t idle_end = 0;  // while nothing is handed out: when to give up
    bool failed = false;
    for (;;) {
      if (*stop) {
        failed = true;
        break;
      }
      // 1. blocks of listed draws first
      const int nd = ld_relaxed(p.ctrl + kCtlDraws);
      if (P.held < 0 && ld_relaxed(p.ctrl + kCtlDrawBlk) < nd * C.BPD)
        P.held = atomicAdd(p.ctrl + kCtlDrawBlk, 1);
      if (P.held >= 0 && P.held / C.BPD < ld_relaxed(p.ctrl + kCtlDraws)) {
        const int e = P.held / C.BPD, blk = P.held - e * C.BPD;
        P.held = -1;
        int code = ld_acquire(p.dl + e);
        for (const uint64_t end = now_ns() + p.wait_ns; code == 0 && now_ns() <= end;)
          code = ld_acquire(p.dl + e);
        if (code == 0) {
          failed = true;
          break;
        }
        const int cc = code - 1;
        const int i = (cc >> 6) & 0xFFF, a = (cc >> 2) & 0xF, kind = cc & 3;
        const char* tb = trow_ptr(trow_of(p, i, a));
        const char* db = kind == kDrawResid ? drow_ptr(drow_of(p, i, a)) : nullptr;
        const int s1 = min(p.nsub, (blk + 1) * kSubBlock);
        for (int s = blk * kSubBlock; s < s1; ++s) {
          const size_t off = static_cast<size_t>(s) * kSubBytes;
          const uint32_t by = static_cast<uint32_t>(min(static_cast<size_t>(kSubBytes), rbytes - off));
          Desc d{kSub, e, s, code};
          if (!publish(P, d, tb + off, VEC ? by : 0u, db ? db + off : nullptr, (VEC && db) ? by : 0u,
                       true)) {
            failed = true;
            break;
          }
        }
        if (failed) break;
        idle_end = 0;
        continue;
      }
      // 2. row segments
      if (!P.rows_done) {
        if (P.seg >= P.seg_end) {
          const int got = next_row_block(P);
          if (got < 0 || *stop) {
            failed = true;
            break;
          }
          if (got == 0) continue;
        }
        const int s = P.seg++;
        const size_t off = static_cast<size_t>(s) * kSegBytes;
        const uint32_t by = static_cast<uint32_t>(min(static_cast<size_t>(kSegBytes), rbytes - off));
        const char* base = P.loc.isd ? drow_ptr(P.row) : trow_ptr(P.row);
        Desc d{kRow, P.loc.i | (P.loc.j << 12) | (P.loc.isd << 16), s, 0};
        if (!publish(P, d, base + off, VEC ? by : 0u, nullptr, 0u, P.greedy)) {
          failed = true;
          break;
        }
        idle_end = 0;
        continue;
      }
      // 3. nothing to hand out: done once every request's outputs are in
      if (ld_acquire(p.ctrl + kCtlReqDone) >= p.bs) break;
      const uint64_t t = now_ns();
      if (idle_end == 0) idle_end = t + p.wait_ns;
      if (t > idle_end) {
        failed = true;
        break;
      }
      __nanosleep(128);
    }
    if (failed) halt();
    // one end marker per consumer warp
    for (int w = 0; w < kNC && !*stop; ++w) {
      Desc d{kEnd, 0, 0, 0};
      if (!publish(P, d, nullptr, 0, nullptr, 0, false)) {
        halt();
        break;
      }
    }
    // No bulk copy may be in flight when the CTA exits: wait for the last
    // item of every buffer (a copy of valid memory always lands; the bound
    // does not depend on the caller's wait limit).
    const uint64_t drain_end = now_ns() + kDrainNs;
    for (int k = max(0, P.k - p.nbuf); k < P.k; ++k) {
      const int b = k % p.nbuf;
      const uint32_t par = static_cast<uint32_t>(k / p.nbuf) & 1u;
      while (!mbar_poll(&full[b], par) && now_ns() <= drain_end) {
      }
    }
  }
};

// ---------------------------------------------------------------------------

template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads, 1) sampler_kernel(const __grid_constant__ SamplerParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t s_full[kMaxBufs], s_empty[kMaxBufs];
  __shared__ Desc s_desc[kMaxBufs];
  __shared__ int s_ticket, s_stop, s_bad, s_last;
  __shared__ int s_seen[kMaxBufs];
  __shared__ int s_hist[32], s_base[32];
  __shared__ int s_WS[SD_MAX_K + 3], s_P[SD_MAX_K + 2], s_E[SD_MAX_K + 2];
  __shared__ float2 s_tab[16];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bs = p.bs, K1 = p.k_max + 1;
  unsigned char* ring = smem;
  int* order = reinterpret_cast<int*>(smem + static_cast<size_t>(p.nbuf) * kSegBytes);  // [bs]
  // the ring doubles as scratch for the request lengths while the tables are built
  int* nscr = reinterpret_cast<int*>(smem);  // [bs] bin of request i

  if (tid == 0) {
    s_bad = 0;
    s_ticket = 0;
    s_stop = 0;
  }
  if (tid < 32) s_hist[tid] = 0;
  if (tid < kMaxBufs) s_seen[tid] = 0;
  if (tid < 16) s_tab[tid] = p.exp_tab[tid];
  __syncthreads();

  // ---- per-call checks of the compaction (the same verdict in every CTA)
  int bad = 0;
  if (tid == 0 && __ldg(p.cu) != 0) bad = 1;
  for (int i = tid; i < bs; i += kThreads) {
    const int d = __ldg(p.cu + i + 1) - __ldg(p.cu + i);
    if (d < 1 || d > K1) bad = 1;
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0) {
      if (tid == 0) raise_error(p.err, SD_DEV_ERR_CU_SEQLENS);
      for (int i = tid; i < bs; i += kThreads) {
        p.accepted_len[i] = 0;
        for (int j = 0; j < K1; ++j) p.out_tokens[static_cast<size_t>(i) * K1 + j] = -1;
      }
    }
    return;  // nothing read, no counter touched
  }

  // ---- temperatures (flagged once), bins: sampling first, n descending
  int badt = 0;
  for (int i = tid; i < bs; i += kThreads) {
    const float t = __ldg(p.temps + i);
    if (!(t >= 0.0f) || !isfinite(t)) badt |= SD_DEV_ERR_TEMP;
    else if (t > 0.0f && p.draft == nullptr) badt |= SD_DEV_ERR_LOGITS;
    const int n = __ldg(p.cu + i + 1) - __ldg(p.cu + i) - 1;
    const int bin = (eff_tau(p, i) > 0.0f ? 0 : 16) + (15 - n);
    nscr[i] = bin;
    atomicAdd(&s_hist[bin], 1);
  }
  if (badt && blockIdx.x == 0) raise_error(p.err, badt);
  __syncthreads();
  if (warp == 0) {
    const int h = s_hist[lane];
    int inc = h;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    s_base[lane] = inc - h;  // next position of bin `lane`
    __syncwarp();
    // stable scatter of the requests into their bins, 32 at a time
    for (int c0 = 0; c0 < bs; c0 += 32) {
      const int i = c0 + lane;
      const int bin = i < bs ? nscr[i] : -1 - lane;  // past the end: a group of its own
      const unsigned same = __match_any_sync(kFull, bin);
      const unsigned below = same & ((1u << lane) - 1u);
      const int pos = i < bs ? s_base[bin] + __popc(below) : 0;
      __syncwarp();
      if (i < bs) {
        order[pos] = i;
        if (below == 0u) s_base[bin] += __popc(same);  // one lane per bin advances it
      }
      __syncwarp();
    }
    // wave tables: sampling requests with n at s_hist[15 - n], greedy at s_hist[31 - n]
    if (lane == 0) {
      int ws = 0;
      for (int j = 0; j < K1; ++j) {
        int Pgt = 0, Gge = 0;
        for (int n = j + 1; n <= SD_MAX_K; ++n) Pgt += s_hist[15 - n];
        for (int n = j; n <= SD_MAX_K; ++n) Gge += s_hist[31 - n];
        s_P[j] = Pgt;
        s_E[j] = s_hist[15 - j];
        s_WS[j] = ws;
        ws += 2 * Pgt + s_hist[15 - j] + Gge;
      }
      s_WS[K1] = ws;
    }
  }
  // the bins were kept in the ring; later bulk copies write there
  fence_proxy_async();
  // One thread initialises every ring barrier and then fences: the fence
  // makes the initialising thread's own inits visible to the bulk copies'
  // completions (async proxy), so the inits and the fence share a thread.
  if (tid == 0) {
    for (int b = 0; b < p.nbuf; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  Cta C;
  C.order = order;
  C.WS = s_WS;
  C.Pj = s_P;
  C.Ej = s_E;
  C.nsamp = 0;
  for (int b = 0; b < 16; ++b) C.nsamp += s_hist[b];
  C.nw = K1;
  C.U = s_WS[K1];
  C.BPU = (p.nseg + kRowBlock - 1) / kRowBlock;
  C.BPD = (p.nsub + kSubBlock - 1) / kSubBlock;
  C.tab = s_tab;

  Sampler<T, VEC> S{p, C, ring, s_full, s_empty, s_desc, &s_ticket, s_seen, &s_stop, lane};
  if (warp < kNC) {
    S.consume();
  } else {
    if (lane == 0) S.produce();
    // The CTA barrier below is warp-aligned: the producer warp reaches it
    // converged, after lane 0 has drained its copies.
    __syncwarp();
  }

  // ---- the last CTA out resets the call's control words (and, after a
  // wait gave up, every counter and the outputs, to well-formed values)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(p.ctrl + kCtlCtas, 1) == static_cast<int>(gridDim.x) - 1;
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    if (ld_acquire(p.ctrl + kCtlStop)) {
      const int pairs = bs * K1;
      for (int q = tid; q < pairs; q += kThreads) p.pc[q] = 0;
      for (int i = tid; i < bs; i += kThreads) {
        p.st[i] = 0;
        p.ev[i] = 0;
        p.accepted_len[i] = 0;
        for (int j = 0; j < K1; ++j)
          p.out_tokens[static_cast<size_t>(i) * K1 + j] = j == 0 ? 0 : -1;
      }
      for (int e = tid; e < 2 * bs; e += kThreads) {
        p.dl[e] = 0;
        p.dc[e] = 0;
      }
    }
    __syncthreads();
    if (tid < kCtlWords) p.ctrl[tid] = 0;
    __threadfence();
  }
}

template <typename T, bool VEC>
void* kfn() {
  return reinterpret_cast<void*>(&sampler_kernel<T, VEC>);
}

void* pick(int elem, bool vec) {
  static void* const t[4] = {kfn<float, true>(), kfn<float, false>(), kfn<uint16_t, true>(),
                             kfn<uint16_t, false>()};
  return t[(elem == 4 ? 0 : 2) + (vec ? 0 : 1)];
}

// Raises the kernel's dynamic shared-memory limit once per (kernel, device).
cudaError_t prepare(void* fn, int* limit) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> lim_of[4][kMaxDev];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int slot = -1;
  for (int k = 0; k < 4; ++k)
    if (fn == pick(k < 2 ? 4 : 2, (k & 1) == 0)) slot = k;
  if (slot < 0 || dev < 0 || dev >= kMaxDev) return cudaErrorInvalidValue;
  int lim = lim_of[slot][dev].load(std::memory_order_acquire);
  if (lim == 0) {
    std::lock_guard<std::mutex> lk(mu);
    lim = lim_of[slot][dev].load(std::memory_order_relaxed);
    if (lim == 0) {
      int optin = 0;
      e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
      if (e != cudaSuccess) return e;
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, fn);
      if (e != cudaSuccess) return e;
      lim = optin - static_cast<int>(fa.sharedSizeBytes);
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
      if (e != cudaSuccess) return e;
      lim_of[slot][dev].store(lim, std::memory_order_release);
    }
  }
  *limit = lim;
  return cudaSuccess;
}

}  // namespace

SamplerWs sampler_ws_layout(int bs, int k_max, int V, int elem) {
  auto al = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
  const size_t rows_t = static_cast<size_t>(bs) * (k_max + 1);
  const size_t rows_d = static_cast<size_t>(bs) * k_max;
  const size_t rb = static_cast<size_t>(V) * elem;
  const size_t nseg = (rb + kSegBytes - 1) / kSegBytes;
  const size_t nsub = (rb + kSubBytes - 1) / kSubBytes;
  SamplerWs L;
  L.seg_t = 0;
  L.seg_d = al(L.seg_t + rows_t * nseg * sizeof(SegRec));
  L.ps = al(L.seg_d + rows_d * nseg * sizeof(SegRec));
  L.rs = al(L.ps + rows_t * sizeof(PairStat));
  L.zero = al(L.rs + 2 * static_cast<size_t>(bs) * nsub * 8);
  L.pc = L.zero;
  L.st = al(L.pc + rows_t * 4);
  L.ev = al(L.st + static_cast<size_t>(bs) * 4);
  L.dl = al(L.ev + static_cast<size_t>(bs) * 4);
  L.dc = al(L.dl + 2 * static_cast<size_t>(bs) * 4);
  L.ctrl = al(L.dc + 2 * static_cast<size_t>(bs) * 4);
  L.total = al(L.ctrl + kCtlWords * 4);
  return L;
}

cudaError_t choose_sampler_shape(int V, int elem, int bs, int blocks, bool vec,
                                 SamplerShape* out, bool* fits) {
  *fits = false;
  (void)V;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  void* fn = pick(elem, vec);
  int lim = 0;
  e = prepare(fn, &lim);
  if (e != cudaSuccess) return e;
  const size_t tables = (static_cast<size_t>(bs) * 4 + 127) & ~static_cast<size_t>(127);
  if (tables + 4 * static_cast<size_t>(kSegBytes) > static_cast<size_t>(lim)) return cudaSuccess;
  int nbuf = static_cast<int>((static_cast<size_t>(lim) - tables) / kSegBytes);
  nbuf = std::min(nbuf, kMaxBufs);
  // A consumer waits on its buffer's phase by parity, which is unambiguous
  // only while no consumer can run a whole ring ahead of the producer.
  if (nbuf < kNC + 2) return cudaSuccess;
  // the ring also holds the request bins while the tables are built
  if (static_cast<size_t>(nbuf) * kSegBytes < static_cast<size_t>(bs) * 4) return cudaSuccess;
  out->nbuf = nbuf;
  out->threads = kThreads;
  out->blocks = blocks > 0 ? std::min(blocks, sms) : sms;
  out->smem = static_cast<size_t>(nbuf) * kSegBytes + tables;
  out->vec = vec;
  *fits = true;
  return cudaSuccess;
}

cudaError_t launch_sampler(const SamplerParams& p, int elem, const SamplerShape& shape,
                           cudaStream_t s) {
  void* fn = pick(elem, shape.vec);
  int lim = 0;
  cudaError_t e = prepare(fn, &lim);
  if (e != cudaSuccess) return e;
  if (shape.smem > static_cast<size_t>(lim)) return cudaErrorInvalidValue;
  void* args[] = {const_cast<SamplerParams*>(&p)};
  e = cudaLaunchKernel(fn, dim3(shape.blocks), dim3(shape.threads), args, shape.smem, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace sdk
