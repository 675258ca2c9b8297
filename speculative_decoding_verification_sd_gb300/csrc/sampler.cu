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
// Design (GB300).  One persistent CTA per SM: a scheduler warp claims units
// of work into a small queue in shared memory, and sixteen streaming warps
// take every unit together.  A unit is one logit row (claimed in slot order,
// "waves": slot j's rows of every request before slot j + 1's) or one final
// draw.  Streaming warp w copies its own slice of the unit's row(s) with
// bulk copies into two buffers of its own (the next chunk lands while the
// current one is reduced, across unit boundaries) and reduces each chunk to
// softmax statistics or an argmax.  A finishing warp takes the units in
// order once all sixteen have counted their part: it combines a row's
// partials and counts the row into its (request, slot) pair; the row that
// completes a pair takes the slot's accept decision, and the decision that
// settles a request lists the request's final draw.  A draw is a unit like a
// row: every streaming warp sums its slice's inverse-CDF weights in exact
// 64-bit fixed point, and the finishing warp finds the crossing chunk and
// walks it.  The finish's global round trips (atomics, statistics loads) so
// stay off the streaming warps.  With SD_VERIFY_EARLY_EXIT the scheduler
// drops rows of slots after a request's settled first rejection before they
// are streamed.
//
// Precision.  Row statistics use the hardware base-2 exponent on an argument
// d * s2 with d = l - m exact and s2 = log2(e)/tau carried in two floats; the
// per-chunk sums are compensated and combined in double-float.  A final
// draw's weights are fp32 except where an element weighs more than 2^-10 of
// its row's maximum: there the weight is formed in double-float from a
// 16-entry table of 2^(j/16) and a short series (Tang's table-driven
// method), so the elements that carry the distribution's mass match the
// fp64 definition to about 1e-10.  No fp64 arithmetic is used: this GPU
// runs it, and 64-bit conversions, at 1/64 of the fp32 rate.
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>

#include "sd_device.cuh"
#include "sd_internal.h"

namespace sdk {

namespace {

constexpr int kNW = kSamplerWarps;         // streaming warps per CTA
constexpr int kFin = kFinishWarps;         // finishing warps per CTA
constexpr int kThreads = (kNW + 1 + kFin) * 32;  // + the scheduler warp
constexpr int kQ = 4;                      // positions of the per-CTA unit queue
constexpr int kChunk = kSegBytes;          // bytes of a row chunk (one bulk copy)
constexpr int kHalf = kSubBytes;           // bytes per row of a draw chunk
constexpr uint64_t kDrainNs = 2000000000ull;  // bound of the exit drain of in-flight copies (2 s)
constexpr float kBigT = -10.0f;           // weights above 2^-10 of the row maximum: precise
constexpr int kHeavyList = 128;           // per-warp list of heavy elements handled in one pass
constexpr float kTwo64 = 18446744073709551616.0f;
// log2(e) and ln(2), each split into two floats (hi + lo).
constexpr float kLog2eHi = 1.44269502162933349609375f;
constexpr float kLog2eLo = 1.925963033500011079e-08f;
constexpr float kLn2Hi = 0.693147182464599609375f;
constexpr float kLn2Lo = -1.904654299957768e-09f;

// Units of work handed from the scheduler warp to the streaming warps.
enum { kUEnd = 0, kURow = 1, kUDraw = 2 };
// Kinds of a final draw.
enum { kDrawResid = 0, kDrawP = 1 };

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
// One poll of an mbarrier phase (the hardware may hold the thread briefly
// while the phase is incomplete; no suspend hint, which measurably left
// warps asleep well after their phase had completed).
__device__ __forceinline__ bool mbar_poll(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
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

// Double-float (hi + lo) sum and product, ~2^-44 relative; fast_two_sum
// needs |hi| of the result to dominate, which holds for these non-negative
// sums and products.
__device__ __forceinline__ void ff_add(float ah, float al, float bh, float bl, float& sh, float& sl) {
  float s, e;
  two_sum(ah, bh, s, e);
  e = __fadd_rn(e, __fadd_rn(al, bl));
  fast_two_sum(s, e, sh, sl);
}
__device__ __forceinline__ void ff_mul(float ah, float al, float bh, float bl, float& ph, float& pl) {
  const float p = __fmul_rn(ah, bh);
  const float c = __fmaf_rn(ah, bl, __fmaf_rn(al, bh, __fmaf_rn(ah, bh, -p)));
  fast_two_sum(p, c, ph, pl);
}
// 1 / (zh + zl) as a double-float: a rounded reciprocal and one correction.
__device__ __forceinline__ void ff_recip(float zh, float zl, float& ih, float& il) {
  ih = __frcp_rn(zh);
  const float e = __fmaf_rn(-zl, ih, __fmaf_rn(-zh, ih, 1.0f));
  il = __fmul_rn(e, ih);
}
__device__ __forceinline__ void warp_sum_ff(float& h, float& l) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(kFull, h, o), ol = __shfl_xor_sync(kFull, l, o);
    ff_add(h, l, oh, ol, h, l);
  }
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
// global row read through the read-only path (`gmem`; the walk's re-reads of
// one chunk then hit L1), or single elements of a global row (element path;
// positions >= n read as -inf).
template <typename T, bool VEC>
__device__ __forceinline__ void load_unit(const void* src, int q, int n, bool gmem,
                                          float (&f)[ET<T>::VE]) {
  using E = ET<T>;
  if constexpr (VEC) {
    const typename E::V* v = static_cast<const typename E::V*>(src) + q;
    if (gmem) {
      if constexpr (sizeof(T) == 2) E::unpack(__ldg(reinterpret_cast<const uint4*>(v)), f);
      else E::unpack(__ldg(reinterpret_cast<const float4*>(v)), f);
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
    (void)gmem;
  }
}

// ---------------------------------------------------------------------------
// Final-draw weights.  A draw from p weighs element k with p_k; a residual
// draw with max(p_k - q_k, 0); in 2^56 fixed point.  A unit's value is the
// fixed-point value of the fp32 sum (in element order) of its elements that
// weigh less than 2^-10 of their row's maximum, plus the double-float value
// of each heavier element.  The sub-chunk sums and the walk of the crossing
// sub-chunk use these same functions, so the walk retraces the sums exactly.
struct DrawCtx {
  float Mt, Md, s2h, s2l;
  float izth, iztl, izdh, izdl;  // 1 / Z as (hi, lo)
  bool resid;
};

// x * 2^56 truncated to an integer (0 <= x < 256) from two 32-bit
// conversions: this GPU converts to 64-bit integers at 1/8 of the 32-bit
// rate.  y = x * 2^24 and its fraction are exact, so for x >= 2^-32 the
// result is x * 2^56 exactly.
__device__ __forceinline__ unsigned long long fixed56(float x) {
  const float y = __fmul_rn(x, 16777216.0f);
  const float yt = truncf(y);
  const uint32_t hi = __float2uint_rz(yt);
  const uint32_t lo = __float2uint_rz(__fmul_rn(__fsub_rn(y, yt), 4294967296.0f));
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

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
  // The table-driven exponent leaves its series' tail in the low word, up
  // to ~2^-12 of the high one: renormalise so |pl| <= ulp(ph) / 2, then ph
  // at 2^-56 and the small correction pl at 2^-48 (|pl * 2^48| <= 2^24).
  fast_two_sum(ph, pl, ph, pl);
  const long long v = static_cast<long long>(fixed56(ph)) +
                      static_cast<long long>(__float2int_rn(__fmul_rn(pl, 281474976710656.0f))) * 256ll;
  return v > 0 ? static_cast<unsigned long long>(v) : 0ull;
}

// Two elements at once in packed fp32x2 arithmetic; each half is rounded
// exactly as elem_fast rounds its element (the packed operations are the
// same IEEE operations per half).
__device__ __forceinline__ float2 pair_fast(const DrawCtx& c, float2 lt, float2 ld, bool& b0, bool& b1) {
  const float2 dt = __fadd2_rn(lt, make_float2(-c.Mt, -c.Mt));
  const float2 tt = __ffma2_rn(dt, make_float2(c.s2h, c.s2h), __fmul2_rn(dt, make_float2(c.s2l, c.s2l)));
  const float2 wt = make_float2(exp2_ftz(tt.x), exp2_ftz(tt.y));
  b0 = tt.x > kBigT;
  b1 = tt.y > kBigT;
  if (!c.resid)
    return __ffma2_rn(wt, make_float2(c.izth, c.izth), __fmul2_rn(wt, make_float2(c.iztl, c.iztl)));
  const float2 dd = __fadd2_rn(ld, make_float2(-c.Md, -c.Md));
  const float2 td = __ffma2_rn(dd, make_float2(c.s2h, c.s2h), __fmul2_rn(dd, make_float2(c.s2l, c.s2l)));
  const float2 wd = make_float2(exp2_ftz(td.x), exp2_ftz(td.y));
  b0 = b0 || td.x > kBigT;
  b1 = b1 || td.y > kBigT;
  const float2 qd = __ffma2_rn(wd, make_float2(c.izdh, c.izdh), __fmul2_rn(wd, make_float2(c.izdl, c.izdl)));
  const float2 r = __ffma2_rn(wt, make_float2(c.izth, c.izth),
                              __ffma2_rn(wt, make_float2(c.iztl, c.iztl), make_float2(-qd.x, -qd.y)));
  return make_float2(fmaxf(r.x, 0.0f), fmaxf(r.y, 0.0f));
}

// A unit's fast value: the fixed-point value of the fp32 sum (a balanced
// tree, in element order) of its elements that weigh less than 2^-10 of
// their row's maximum; *bigm marks the others.
template <int VE>
__device__ __forceinline__ unsigned long long unit_fast(const DrawCtx& c, const float (&ft)[VE],
                                                        const float (&fd)[VE], uint32_t& bigm) {
  float r[VE];
  bigm = 0;
#pragma unroll
  for (int e = 0; e < VE; e += 2) {
    bool b0, b1;
    const float2 pr = pair_fast(c, make_float2(ft[e], ft[e + 1]), make_float2(fd[e], fd[e + 1]), b0, b1);
    r[e] = b0 ? 0.0f : pr.x;
    r[e + 1] = b1 ? 0.0f : pr.y;
    bigm |= (b0 ? 1u << e : 0u) | (b1 ? 1u << (e + 1) : 0u);
  }
#pragma unroll
  for (int w = 1; w < VE; w *= 2)
#pragma unroll
    for (int e = 0; e < VE; e += 2 * w) r[e] = __fadd_rn(r[e], r[e + w]);
  return fixed56(r[0]);
}

// ---------------------------------------------------------------------------
// Per-CTA context: the work-list tables built in the prologue.

struct Cta {
  const int* order;  // [bs]: sampling requests by n desc, then greedy ones by n desc
  const int* WS;     // [nw+1] first unit of wave j
  const int* Pj;     // [nw] sampling requests with n > j
  const int* Ej;     // [nw] sampling requests with n == j
  int nsamp, nw, U;
  int dshift;         // a final draw is split into 1 << dshift units (the same in every CTA)
  int dper;           // draw chunks per warp in one part: ceil(ncd >> dshift)
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

// One unit of the per-CTA queue.
struct Unit {
  int kind;
  int a;  // row: i | j << 12 | draft << 16;  draw: the draw's index e
  int b;  // row: the row's index;  draw: its list entry 1 + (i << 6 | a << 2 | kind)
  int c;  // draw: which of its 1 << C.dshift parts
};

// What a streaming warp needs of a unit.
struct UInfo {
  int kind;
  int i, j, n;
  bool isd, greedy;
  float tau;
  const char* src_t;  // row unit: the row;  draw: the target row t_a
  const char* src_d;  // residual draw: the draft row d_a (else null)
  int e, a, dkind;    // draw unit
  int part;           // draw unit: which part of the draw's chunks
  int x;              // row unit of a slot j < n: the slot's draft token (else -1)
};

// A published unit as the scheduler decoded it: the unit, its exponent
// scale (sampling rows), a draw's context and uniform.  The scheduler runs
// ahead of the streaming warps, so their global loads leave the critical path.
struct QInfo {
  UInfo f;
  float s2h, s2l;
  DrawCtx dc;
  float du;
};

template <typename T, bool VEC>
struct Sampler {
  using E = ET<T>;
  static constexpr int VE = E::VE;
  static constexpr int kUPL = kHalf / static_cast<int>(sizeof(T)) / VE / 32;  // draw-chunk units per lane

  const SamplerParams& p;
  Cta C;
  // per-CTA queue in shared memory
  Unit* q_ent;         // [kQ]
  volatile int* q_seq; // [kQ] position published in each slot
  volatile int* q_fin; // [kQ] position whose unit is complete in each slot
  int* q_cnt;          // [kQ] streaming warps done with the slot's position (grows by kNW a use)
  volatile int* q_end; // position of the END unit once published (else INT_MAX)
  QInfo* q_inf;        // [kQ] the decoded unit of each published position
  uint4* q_rec;        // [kQ][kNW] per-warp partial statistics of a row unit
  unsigned char* bufs; // [kNW][2][kChunk]
  unsigned short* heavy;  // [kNW][kHeavyList] heavy elements of a draw chunk
  uint64_t* full;      // [kNW][2]
  volatile int* stop;
  int lane, warp;
  int R;               // row bytes

  __device__ const char* trow_ptr(long long r) const {
    return static_cast<const char*>(p.target) + static_cast<size_t>(r) * static_cast<size_t>(R);
  }
  __device__ const char* drow_ptr(long long r) const {
    return static_cast<const char*>(p.draft) + static_cast<size_t>(r) * static_cast<size_t>(R);
  }
  __device__ int sl_begin(int w) const { return min(w * p.slice, R); }
  __device__ int sl_end(int w) const { return min((w + 1) * p.slice, R); }
  __device__ int nchunks(int kind, int w) const {
    const int len = sl_end(w) - sl_begin(w);
    const int cb = kind == kURow ? kChunk : kHalf;
    return len > 0 ? (len + cb - 1) / cb : 0;
  }
  // Warp w's chunks of unit f: [cbase, cbase + ucount) of its slice (a draw
  // part takes its share of every warp's draw chunks).
  __device__ int cbase(const UInfo& f, int w) const {
    if (f.kind == kURow) return 0;
    return min(f.part * C.dper, nchunks(kUDraw, w));
  }
  __device__ int ucount(const UInfo& f, int w) const {
    if (f.kind == kURow) return nchunks(kURow, w);
    return min((f.part + 1) * C.dper, nchunks(kUDraw, w)) - cbase(f, w);
  }

  __device__ void halt() const {
    if (lane == 0) {
      raise_error(p.err, SD_DEV_ERR_TIMEOUT);
      atomicExch(p.ctrl + kCtlStop, 1);
      *stop = 1;
    }
  }

  __device__ UInfo info(const Unit& u) const {
    UInfo f;
    f.kind = u.kind;
    f.src_d = nullptr;
    f.x = -1;
    f.e = f.a = f.dkind = f.part = 0;
    f.isd = false;
    if (u.kind == kURow) {
      f.i = u.a & 0xFFF;
      f.j = (u.a >> 12) & 0xF;
      f.isd = ((u.a >> 16) & 1) != 0;
      f.n = n_of(p, f.i);
      f.tau = eff_tau(p, f.i);
      f.greedy = !(f.tau > 0.0f);
      f.src_t = f.isd ? drow_ptr(u.b) : trow_ptr(u.b);
      if (f.j < f.n) f.x = __ldg(p.draft_ids + drow_of(p, f.i, f.j));
    } else {
      f.e = u.a;
      f.part = u.c;
      const int code = u.b - 1;
      f.i = (code >> 6) & 0xFFF;
      f.a = (code >> 2) & 0xF;
      f.dkind = code & 3;
      f.j = f.a;
      f.n = n_of(p, f.i);
      f.tau = eff_tau(p, f.i);
      f.greedy = false;
      f.src_t = trow_ptr(trow_of(p, f.i, f.a));
      if (f.dkind == kDrawResid) f.src_d = drow_ptr(drow_of(p, f.i, f.a));
    }
    return f;
  }

  // ---- per-warp bulk copies ----------------------------------------------
  __device__ unsigned char* buf_of(int g) const {
    return bufs + (static_cast<size_t>(warp) * 2 + (g & 1)) * kChunk;
  }
  __device__ uint64_t* bar_of(int g) const { return full + warp * 2 + (g & 1); }

  // Lane 0: chunk c of unit f into buffer g & 1 (vector path only).  Every
  // row is copied evict-first: the final draws' second reads mostly miss L2
  // anyway, and the small per-call data (the planner's inputs, the counters)
  // then stays resident.
  __device__ void issue(const UInfo& f, int c, int g, uint64_t pol_first) const {
    const int cb = f.kind == kURow ? kChunk : kHalf;
    const int off = sl_begin(warp) + (cbase(f, warp) + c) * cb;
    const uint32_t by = static_cast<uint32_t>(min(cb, sl_end(warp) - off));
    unsigned char* dst = buf_of(g);
    uint64_t* bar = bar_of(g);
    if (f.kind == kURow) {
      mbar_arrive_expect_tx(bar, by);
      bulk_load(dst, f.src_t + off, by, bar, pol_first);
    } else {
      mbar_arrive_expect_tx(bar, f.src_d ? 2 * by : by);
      bulk_load(dst, f.src_t + off, by, bar, pol_first);
      if (f.src_d) bulk_load(dst + kHalf, f.src_d + off, by, bar, pol_first);
    }
  }

  // Lane 0: waits for chunk g's copy (bounded).
  __device__ bool wait_chunk(int g) const {
    uint64_t* bar = bar_of(g);
    const uint32_t par = static_cast<uint32_t>(g >> 1) & 1u;
    if (mbar_poll(bar, par)) return true;
    const uint64_t end = now_ns() + p.wait_ns;
    for (;;) {
      if (mbar_poll(bar, par)) return true;
      if (*stop || now_ns() > end) return false;
    }
  }

  // ---- row chunks -----------------------------------------------------------
  // Per-warp partial of a row unit: sampling rows keep (m, z = zh + zl) with
  // z = sum of 2^((l - m) s2) over the chunks so far; greedy rows keep the
  // key (ordered value << 32 | ~index) of the best element and a bad flag.
  struct Part {
    float m, zh, zl, lx;
    unsigned long long key;
    int bad;
  };

  // Rescales the double-float z = (zh, zl), taken relative to m_from, to
  // m_to >= m_from: z * 2^((m_from - m_to) s2).
  __device__ void rescale(float& zh, float& zl, float m_from, float m_to, float s2h, float s2l) const {
    float dh, dl;
    two_sum(m_from, -m_to, dh, dl);
    const float th = __fmul_rn(dh, s2h);
    const float tl = __fadd_rn(__fmaf_rn(dh, s2h, -th), __fmaf_rn(dh, s2l, __fmul_rn(dl, s2h)));
    float fh, fl;
    exp2_precise(th, tl, C.tab, fh, fl);
    ff_mul(zh, zl, fh, fl, zh, zl);
  }

  // One chunk of a row unit: n_el elements at src (staged copy or global
  // row), e0 = the chunk's first element in the row.  Lane-private: each
  // lane folds its own elements into its running partial (no shuffle here);
  // the warp combines its lanes once per unit (unit_record).
  __device__ void row_chunk(const void* src, int n_el, int e0, const UInfo& f, float s2h, float s2l,
                            Part& P) const {
    const int nu = (n_el + VE - 1) / VE;
    if (f.greedy) {
      float best = -INFINITY;
      int bidx = INT_MAX, bad = 0;
      for (int q = lane; q < nu; q += 32) {
        float fv[VE];
        float vm;
        if constexpr (VEC) {
          const typename E::V raw = static_cast<const typename E::V*>(src)[q];
          vm = E::vmax_nan(raw);
          if (vm > best) {
            E::unpack(raw, fv);
            int e = VE - 1;
#pragma unroll
            for (int k = VE - 1; k >= 0; --k)
              if (fv[k] == vm) e = k;
            best = vm;
            bidx = q * VE + e;
          }
        } else {
          load_unit<T, false>(src, q, n_el, false, fv);
          vm = fv[0];
#pragma unroll
          for (int k = 1; k < VE; ++k) vm = fmax_nan(vm, fv[k]);
          if (vm > best) {
            int e = VE - 1;
#pragma unroll
            for (int k = VE - 1; k >= 0; --k)
              if (fv[k] == vm) e = k;
            best = vm;
            bidx = q * VE + e;
          }
        }
        bad |= (vm != vm) | (vm == INFINITY);
      }
      const unsigned long long key = bidx == INT_MAX ? 0ull
          : (static_cast<unsigned long long>(ordered_bits(best)) << 32) |
                static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(e0 + bidx));
      P.key = max(P.key, key);
      P.bad |= bad;
      return;
    }
    // four units per step, each with its own dependency chain
    const int nq = nu > lane ? (nu - lane + 31) / 32 : 0;  // units q = lane + 32 t, t < nq
    float cm4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    {
      int t = 0;
      for (; t + 4 <= nq; t += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u) cm4[u] = fmax_nan(cm4[u], unit_max(src, lane + 32 * (t + u), n_el));
      }
      for (; t < nq; ++t) cm4[0] = fmax_nan(cm4[0], unit_max(src, lane + 32 * t, n_el));
    }
    const float cm = fmax_nan(fmax_nan(cm4[0], cm4[1]), fmax_nan(cm4[2], cm4[3]));
    if (f.x >= e0 && f.x < e0 + n_el && lane == 0) {
      if constexpr (VEC) P.lx = E::at(src, f.x - e0);
      else P.lx = E::ldg(src, f.x - e0);
    }
    if (!(cm == cm) || cm == INFINITY) {  // NaN or +inf: the row is bad
      P.bad = 1;
      return;
    }
    if (P.bad || cm == -INFINITY) return;  // nothing finite in the lane's part
    if (cm > P.m) {  // the lane's reference maximum rises: rescale its sum
      if (P.m != -INFINITY) rescale(P.zh, P.zl, P.m, cm, s2h, s2l);
      P.m = cm;
    }
    const float m = P.m;
    // the lane's compensated sum, continued, and a second chain beside it
    float ks = P.zh, kc = P.zl, ks2 = 0.0f, kc2 = 0.0f;
    int t = 0;
    for (; t + 4 <= nq; t += 4) {
      float a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = unit_exp_sum(src, lane + 32 * (t + u), n_el, m, s2h, s2l);
      comp_add(ks, kc, __fadd_rn(a[0], a[1]));
      comp_add(ks2, kc2, __fadd_rn(a[2], a[3]));
    }
    for (; t < nq; ++t) comp_add(ks, kc, unit_exp_sum(src, lane + 32 * t, n_el, m, s2h, s2l));
    fast_two_sum(ks, kc, ks, kc);
    if (ks2 > 0.0f) {
      fast_two_sum(ks2, kc2, ks2, kc2);
      ff_add(ks, kc, ks2, kc2, ks, kc);
    }
    P.zh = ks;
    P.zl = kc;
  }

  // Maximum (NaN-propagating) of unit q of a chunk.
  __device__ __forceinline__ float unit_max(const void* src, int q, int n_el) const {
    if constexpr (VEC) {
      (void)n_el;
      return E::vmax_nan(static_cast<const typename E::V*>(src)[q]);
    } else {
      float fv[VE];
      load_unit<T, false>(src, q, n_el, false, fv);
      float vm = fv[0];
#pragma unroll
      for (int k = 1; k < VE; ++k) vm = fmax_nan(vm, fv[k]);
      return vm;
    }
  }

  // fp32 sum of 2^((l - m) s2) over unit q's elements (pairs in fp32x2).
  __device__ __forceinline__ float unit_exp_sum(const void* src, int q, int n_el, float m, float s2h,
                                                float s2l) const {
    float fv[VE];
    load_unit<T, VEC>(src, q, n_el, false, fv);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < VE; k += 2) {
      const float2 d = __fadd2_rn(make_float2(fv[k], fv[k + 1]), make_float2(-m, -m));
      const float2 t = __ffma2_rn(d, make_float2(s2h, s2h), __fmul2_rn(d, make_float2(s2l, s2l)));
      acc = __fadd2_rn(acc, make_float2(exp2_ftz(t.x), exp2_ftz(t.y)));
    }
    return __fadd_rn(acc.x, acc.y);
  }

  // The warp's record of a row unit from its lanes' partials (warp-wide):
  // greedy rows the best key and the bad flag; sampling rows the maximum
  // (NaN when a lane saw NaN or +inf), the double-float sum relative to it,
  // and the draft token's logit (lane 0).
  __device__ uint4 unit_record(const UInfo& f, const Part& P, float s2h, float s2l) const {
    const int bad = __any_sync(kFull, P.bad != 0);
    if (f.greedy) {
      const unsigned long long key = warp_max_u64(P.key);
      return make_uint4(static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32),
                        static_cast<uint32_t>(bad), 0u);
    }
    const float M = warp_max(P.m);
    float zh = 0.0f, zl = 0.0f;
    if (!bad && P.m != -INFINITY) {
      zh = P.zh;
      zl = P.zl;
      fast_two_sum(zh, zl, zh, zl);
      if (P.m != M) rescale(zh, zl, P.m, M, s2h, s2l);
    }
    warp_sum_ff(zh, zl);
    return make_uint4(__float_as_uint(bad ? NAN : M), __float_as_uint(zh), __float_as_uint(zl),
                      __float_as_uint(P.lx));
  }

  // ---- outputs and per-request bookkeeping --------------------------------
  // Writes every output of request i except a final draw's token (written
  // when the draw finishes).
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

  // Request i's outputs are all written: counted for the schedulers' end
  // test (the outputs themselves are read only after the kernel).
  __device__ void request_done() const {
    __syncwarp();
    if (lane == 0) atomicAdd(p.ctrl + kCtlReqDone, 1);
  }

  __device__ void list_draw(int i, int a, int kind) const {
    if (lane == 0) {
      const int e = atomicAdd(p.ctrl + kCtlDraws, 1);
      if (e < 2 * p.bs) st_release(p.dl + e, 1 + ((i << 6) | (a << 2) | kind));
      else raise_error(p.err, SD_DEV_ERR_TIMEOUT);  // cannot happen: at most two draws a request
    }
  }

  __device__ const RowStat* tstat(int i, int j) const { return p.rst + trow_of(p, i, j); }
  __device__ const RowStat* dstat(int i, int j) const {
    return p.rst + static_cast<size_t>(p.bs) * (p.k_max + 1) + drow_of(p, i, j);
  }

  // ---- row unit complete: combine the warps' partials ---------------------
  // Called by the finishing warp once every part is in; writes the row's
  // statistics and counts the row into its pair.
  // r = warp `lane`'s record (lanes < kNW), read before the slot was released.
  __device__ void row_finish(const uint4 r, const UInfo& f) const {
    RowStat rs;
    rs.izh = 1.0f;
    rs.izl = 0.0f;
    rs.lx = 0.0f;
    rs.amax = -1;
    rs.r0 = rs.r1 = 0;
    if (f.greedy) {
      // record: key (lo, hi), bad
      const unsigned long long key = lane < kNW
          ? (static_cast<unsigned long long>(r.y) << 32) | r.x : 0ull;
      const int bad = __any_sync(kFull, lane < kNW && r.z != 0u);
      const unsigned long long best = warp_max_u64(key);
      rs.amax = best ? static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best)) : -1;
      const uint32_t ob = static_cast<uint32_t>(best >> 32);
      rs.M = best ? __uint_as_float((ob & 0x80000000u) ? (ob & 0x7FFFFFFFu) : ~ob) : -INFINITY;
      rs.bad = bad || best == 0ull;
    } else {
      // record: m (NaN when the warp saw NaN or +inf), zh, zl, lx
      const float m = lane < kNW ? __uint_as_float(r.x) : -INFINITY;
      int bad = __any_sync(kFull, m != m);
      const float M = warp_max(m == m ? m : -INFINITY);
      if (M == -INFINITY) bad = 1;
      float zh = 0.0f, zl = 0.0f;
      if (!bad && m != -INFINITY) {
        float s2h, s2l;
        scale_of(f.tau, s2h, s2l);
        zh = __uint_as_float(r.y);
        zl = __uint_as_float(r.z);
        rescale(zh, zl, m, M, s2h, s2l);
      }
      warp_sum_ff(zh, zl);
      rs.M = M;
      rs.bad = bad;
      if (!bad) ff_recip(zh, zl, rs.izh, rs.izl);
      // lx: kept by the warp whose slice holds the draft token
      if (f.x >= 0 && f.x < p.V) {
        const int wx = static_cast<int>((static_cast<long long>(f.x) * sizeof(T)) / p.slice);
        rs.lx = __shfl_sync(kFull, __uint_as_float(r.w), wx);
      }
    }
    const size_t row = f.isd ? static_cast<size_t>(p.bs) * (p.k_max + 1) + drow_of(p, f.i, f.j)
                             : static_cast<size_t>(trow_of(p, f.i, f.j));
    if (lane == 0) {
      __stcg(reinterpret_cast<uint4*>(p.rst + row), *reinterpret_cast<const uint4*>(&rs));
      __stcg(reinterpret_cast<uint4*>(p.rst + row) + 1, *(reinterpret_cast<const uint4*>(&rs) + 1));
    }
    count_row(f.i, f.j, f.n, f.greedy, 1);
  }

  // Counts `add` into pair (i, j): a row (1) or a skipped row (1 + 1 << 16);
  // the count that completes the pair finishes it (warp-wide).
  __device__ void count_row(int i, int j, int n, bool greedy, int add) const {
    const int pid = i * (p.k_max + 1) + j;
    const int total = (!greedy && j < n) ? 2 : 1;
    int now = 0;
    if (lane == 0) now = atom_add_acq_rel(p.pc + pid, add) + add;
    now = __shfl_sync(kFull, now, 0);
    if ((now & 0xFFFF) == total) {
      __syncwarp();
      pair_finish(i, j, (now >> 16) != 0);
    }
  }

  // ---- pair (i, j) complete ------------------------------------------------
  // `skipped`: early exit dropped one of its rows (the slot is after the
  // request's first rejection), so it has no decision.
  __device__ void pair_finish(int i, int j, bool skipped) const {
    const int n = n_of(p, i);
    const float tau = eff_tau(p, i);
    const bool greedy = !(tau > 0.0f);
    const bool has_d = !greedy && j < n;
    const int pid = i * (p.k_max + 1) + j;
    int bits = 0;
    int tam = -1, tbad = 0, dbad = 0;  // slot j's argmax and bad flags, for settle
    if (!skipped && lane == 0) {
      RowStat t, d;
      *reinterpret_cast<uint4*>(&t) = __ldcg(reinterpret_cast<const uint4*>(tstat(i, j)));
      *(reinterpret_cast<uint4*>(&t) + 1) = __ldcg(reinterpret_cast<const uint4*>(tstat(i, j)) + 1);
      d.M = 0.0f;
      d.izh = 1.0f;
      d.izl = 0.0f;
      d.lx = 0.0f;
      d.bad = 0;
      if (has_d) {
        *reinterpret_cast<uint4*>(&d) = __ldcg(reinterpret_cast<const uint4*>(dstat(i, j)));
        *(reinterpret_cast<uint4*>(&d) + 1) = __ldcg(reinterpret_cast<const uint4*>(dstat(i, j)) + 1);
      }
      const int bad = t.bad | d.bad;
      tam = t.amax;
      tbad = t.bad;
      dbad = d.bad;
      int x = -1;
      bool x_ok = false;
      if (j < n) {
        x = __ldg(p.draft_ids + drow_of(p, i, j));
        x_ok = x >= 0 && x < p.V;
      }
      if (bad) raise_error(p.err, SD_DEV_ERR_LOGITS);
      if (j < n && !x_ok) raise_error(p.err, SD_DEV_ERR_DRAFT_ID);
      if (j == n) {
        bits = 0x8000;  // the bonus row is in
      } else if (greedy) {
        const bool acc = !bad && x_ok && x == t.amax;
        bits = acc ? (1 << j) : (1 << (16 + j));
      } else {
        bool acc = false;
        float pf = 0.0f, qf = 0.0f;
        const float u = p.uniforms[static_cast<size_t>(i) * (p.k_max + 1) + j];
        if (!(u >= 0.0f && u < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
        if (!bad && x_ok) {
          // p(x) = 2^((lx - M) s2) / Z in double-float, rounded once to
          // fp32; the comparison u * q <= p is taken in fp32 on those values
          float s2h, s2l, h, l;
          scale_of(tau, s2h, s2l);
          prob_precise(t.lx, t.M, s2h, s2l, t.izh, t.izl, C.tab, h, l);
          pf = __fadd_rn(h, l);
          prob_precise(d.lx, d.M, s2h, s2l, d.izh, d.izl, C.tab, h, l);
          qf = __fadd_rn(h, l);
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
    // reset the pair's counter for the next call (every row was counted)
    if (lane == 0) p.pc[pid] = 0;
    int old = 0;
    if (lane == 0 && bits) old = atom_or_acq_rel(p.st + i, bits);
    old = __shfl_sync(kFull, old, 0);
    bits = __shfl_sync(kFull, bits, 0);
    const int now = settled(old | bits, n);
    const bool settles = bits && settled(old, n) < 0 && now >= 0;
    if (settles) {
      tam = __shfl_sync(kFull, tam, 0);
      tbad = __shfl_sync(kFull, tbad, 0);
      dbad = __shfl_sync(kFull, dbad, 0);
      settle(i, n, now, greedy, j, tam, tbad | (has_d ? dbad : 0));
    }
  }

  // Request i has its accepted length a: write the outputs, or list its draw.
  // The pair (i, j) that settled it passes its rows' argmax and bad flags,
  // used when a == j (the usual case) instead of reloading them.
  __device__ void settle(int i, int n, int a, bool greedy, int j, int jamax, int jbad) const {
    int bad, amax;
    if (a == j) {
      bad = jbad;
      amax = jamax;
    } else {
      const uint4 t1 = __ldcg(reinterpret_cast<const uint4*>(tstat(i, a)) + 1);
      bad = static_cast<int>(t1.y);
      if (!greedy && a < n) bad |= static_cast<int>(__ldcg(reinterpret_cast<const uint4*>(dstat(i, a)) + 1).y);
      amax = static_cast<int>(t1.x);
    }
    if (greedy) {
      write_prefix(i, a, bad || amax < 0 ? 0 : amax, true);
      request_done();
      return;
    }
    if (bad) {  // flagged already; a well-formed token
      write_prefix(i, a, 0, true);
      request_done();
      return;
    }
    write_prefix(i, a, 0, false);
    __syncwarp();
    list_draw(i, a, a < n ? kDrawResid : kDrawP);
  }

  // ---- final draws -----------------------------------------------------------
  __device__ DrawCtx draw_ctx(int i, int a, int kind) const {
    const uint4 t0 = __ldcg(reinterpret_cast<const uint4*>(tstat(i, a)));
    DrawCtx c;
    c.Mt = __uint_as_float(t0.x);
    c.izth = __uint_as_float(t0.y);
    c.iztl = __uint_as_float(t0.z);
    c.Md = 0.0f;
    c.izdh = 0.0f;
    c.izdl = 0.0f;
    c.resid = kind == kDrawResid;
    if (c.resid) {
      const uint4 d0 = __ldcg(reinterpret_cast<const uint4*>(dstat(i, a)));
      c.Md = __uint_as_float(d0.x);
      c.izdh = __uint_as_float(d0.y);
      c.izdl = __uint_as_float(d0.z);
    }
    scale_of(eff_tau(p, i), c.s2h, c.s2l);
    return c;
  }

  // Fixed-point sum of one draw chunk of n_el elements (target at tsrc,
  // draft at dsrc for a residual draw).
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
    // The heavy elements, compacted into the warp's list and spread over all
    // lanes (a lane's own count varies a lot; the warp's total is small).
    unsigned short* hl = heavy + warp * kHeavyList;
    for (;;) {
      const int cnt = __popcll(bigm);
      int off = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, off, o);
        if (lane >= o) off += t;
      }
      const int total = __shfl_sync(kFull, off, 31);
      if (total == 0) break;
      off -= cnt;  // exclusive
      while (bigm && off < kHeavyList) {
        const int bit = __ffsll(static_cast<long long>(bigm)) - 1;
        bigm &= bigm - 1;
        hl[off++] = static_cast<unsigned short>((lane + 32 * (bit / VE)) * VE + bit % VE);
      }
      __syncwarp();
      const int nl = min(total, kHeavyList);
      for (int n = lane; n < nl; n += 32) {
        const int k = hl[n];
        const float lt = VEC ? E::at(tsrc, k) : E::ldg(tsrc, k);
        const float ld = c.resid ? (VEC ? E::at(dsrc, k) : E::ldg(dsrc, k)) : 0.0f;
        acc += elem_precise(c, lt, ld, C.tab);
      }
      __syncwarp();
    }
    return warp_sum_u64(acc);
  }

  __device__ void finish_token(int e, int i, int n, int a, int y) const {
    if (lane == 0) {
      p.out_tokens[static_cast<size_t>(i) * (p.k_max + 1) + a] = y;
      p.dl[e] = 0;
    }
    request_done();
  }

  // Draw unit complete (every warp's chunk sums are in): threshold
  // floor(u * S), the crossing chunk, then the walk of its units and elements.
  __device__ void draw_finish(const UInfo& f, const DrawCtx& dcx, float u) const {
    const int e = f.e, i = f.i, a = f.a, kind = f.dkind, n = f.n;
    const unsigned long long* rs = p.rs + static_cast<size_t>(e) * kNW * p.ncd;
    const int total = kNW * p.ncd;
    const int spl = (total + 31) / 32;
    const int b0 = min(total, lane * spl), b1 = min(total, b0 + spl);
    // lane's chunk sums (chunks past a warp's slice weigh 0): held in
    // registers when they fit, so the crossing search below reloads nothing
    constexpr int kHeld = 8;
    const bool held = spl <= kHeld;
    unsigned long long hv[kHeld];
    unsigned long long ls = 0ull;
    if (held) {
#pragma unroll
      for (int t = 0; t < kHeld; ++t) {
        const int q = b0 + t;
        hv[t] = (q < b1 && q % p.ncd < nchunks(kUDraw, q / p.ncd)) ? __ldcg(rs + q) : 0ull;
        ls += hv[t];
      }
    } else {
      for (int q = b0; q < b1; ++q)
        if (q % p.ncd < nchunks(kUDraw, q / p.ncd)) ls += __ldcg(rs + q);
    }
    unsigned long long inc = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    const unsigned long long S = __shfl_sync(kFull, inc, 31);
    if (lane == 0 && !(u >= 0.0f && u < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
    if (S == 0ull) {
      if (kind == kDrawResid) {  // no residual mass in fp32: draw from p of the same row
        __syncwarp();
        if (lane == 0) p.dl[e] = 0;
        list_draw(i, a, kDrawP);
        return;
      }
      if (lane == 0) raise_error(p.err, SD_DEV_ERR_LOGITS);
      finish_token(e, i, n, a, 0);
      return;
    }
    const float uc = fminf(fmaxf(u, 0.0f), 0.99999994f);
    const unsigned long long th = __umul64hi(__float2ull_rn(__fmul_rn(uc, kTwo64)), S);
    // the lane whose range holds the crossing
    const unsigned hit = __ballot_sync(kFull, inc > th);
    const int L = __ffs(hit) - 1;  // exists: inc[31] = S > th
    unsigned long long before = __shfl_sync(kFull, inc - ls, L);
    int cq = 0;
    if (lane == L) {
      cq = b1 - 1;
      unsigned long long run = before;
      if (held) {
        bool found = false;
#pragma unroll
        for (int t = 0; t < kHeld; ++t) {
          if (!found && b0 + t < b1) {
            if (run + hv[t] > th) {
              cq = b0 + t;
              found = true;
            } else {
              run += hv[t];
            }
          }
        }
      } else {
        for (int q = b0; q < b1; ++q) {
          const unsigned long long v = q % p.ncd < nchunks(kUDraw, q / p.ncd) ? __ldcg(rs + q) : 0ull;
          if (run + v > th) {
            cq = q;
            break;
          }
          run += v;
        }
      }
      before = run;
    }
    cq = __shfl_sync(kFull, cq, L);
    before = __shfl_sync(kFull, before, L);
    const int w = cq / p.ncd, cc = cq % p.ncd;
    const int off = sl_begin(w) + cc * kHalf;
    const int n_el = min(kHalf, sl_end(w) - off) / static_cast<int>(sizeof(T));
    const int y = walk(dcx, i, a, off / static_cast<int>(sizeof(T)), n_el, th - before);
    finish_token(e, i, n, a, y);
  }

  // The element of the chunk of n_el elements at k0 where the running weight
  // passes th (from the chunk's start); past the last element's weight, the
  // last positive one.
  __device__ int walk(const DrawCtx& c, int i, int a, int k0, int n_el, unsigned long long th) const {
    const int nu = (n_el + VE - 1) / VE;
    const char* tb = trow_ptr(trow_of(p, i, a)) + static_cast<size_t>(k0) * sizeof(T);
    const char* db = c.resid ? drow_ptr(drow_of(p, i, a)) + static_cast<size_t>(k0) * sizeof(T) : tb;
    unsigned long long v[kUPL];
    uint64_t bigm = 0ull;
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
        uint32_t bm;
        v[k] = unit_fast<VE>(c, ft, fd, bm);
        bigm |= static_cast<uint64_t>(bm) << (k * VE);
      }
    }
    while (bigm) {  // the heavy elements, four per pass, each added to its unit
      int kk[4], ku[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        kk[t] = -1;
        ku[t] = -1;
        if (bigm) {
          const int bit = __ffsll(static_cast<long long>(bigm)) - 1;
          bigm &= bigm - 1;
          ku[t] = bit / VE;
          kk[t] = (lane * kUPL + ku[t]) * VE + bit % VE;
        }
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int k = kk[t] < 0 ? 0 : kk[t];
        const float lt = E::ldg(tb, k);
        const float ld = c.resid ? E::ldg(db, k) : 0.0f;
        const unsigned long long pv = elem_precise(c, lt, ld, C.tab);
#pragma unroll
        for (int u2 = 0; u2 < kUPL; ++u2) v[u2] += ku[t] == u2 ? pv : 0ull;
      }
    }
    unsigned long long ls = 0ull;
    int lastu = -1;
#pragma unroll
    for (int k = 0; k < kUPL; ++k) {
      ls += v[k];
      if (v[k]) lastu = lane * kUPL + k;
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
    // the elements of unit q, one per lane (lanes < VE), each with its own
    // fixed-point weight; the first whose running weight passes rem
    unsigned long long w = 0ull;
    {
      float ft[VE], fd[VE];
      load_unit<T, VEC>(tb, q, n_el, true, ft);
      if (c.resid) load_unit<T, VEC>(db, q, n_el, true, fd);
      else {
#pragma unroll
        for (int e = 0; e < VE; ++e) fd[e] = 0.0f;
      }
      float lt = ft[0], ld = fd[0];
#pragma unroll
      for (int e = 1; e < VE; ++e)
        if (lane == e) {
          lt = ft[e];
          ld = fd[e];
        }
      bool big;
      const float r = elem_fast(c, lt, ld, big);
      w = big ? elem_precise(c, lt, ld, C.tab) : fixed56(r);
      if (lane >= VE) w = 0ull;
    }
    unsigned long long run = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(kFull, run, o);
      if (lane >= o) run += t;
    }
    const unsigned pass = __ballot_sync(kFull, lane < VE && run > rem);
    const unsigned pos = __ballot_sync(kFull, lane < VE && w > 0ull);
    const int e = pass ? __ffs(pass) - 1 : (pos ? 31 - __clz(pos) : 0);
    return k0 + q * VE + e;
  }

  // ---- streaming warps -------------------------------------------------------
  // Waits (lane 0, bounded) until position k is published in its slot.
  __device__ bool wait_entry(int k) const {
    bool ok = true;
    if (lane == 0 && q_seq[k % kQ] != k) {
      const uint64_t end = now_ns() + p.wait_ns;
      for (;;) {
        if (q_seq[k % kQ] == k) break;
        if (*stop || now_ns() > end) {
          ok = false;
          break;
        }
        __nanosleep(64);
      }
    }
    ok = __shfl_sync(kFull, ok, 0) != 0;
    __threadfence_block();  // the entry's fields after its published position
    __syncwarp();
    return ok;
  }

  // Warp w's part of position k is done: its record (row units) and the
  // count the finishing warp waits on.
  __device__ void finalize(int k, const UInfo& f, const Part& P, float s2h, float s2l) const {
    const int slot = k % kQ;
    uint4 r = make_uint4(0u, 0u, 0u, 0u);
    if (f.kind == kURow) r = unit_record(f, P, s2h, s2l);
    if (lane == 0) {
      if (f.kind == kURow) {
        q_rec[slot * kNW + warp] = r;
      } else {
        __threadfence();  // the chunk sums, read back through L2 by the finishing warp
      }
      __threadfence_block();
      atomicAdd(q_cnt + slot, 1);
    }
    __syncwarp();
  }

  // ---- finishing warps ---------------------------------------------------------
  // Finishing warp f takes positions f, f + kFin, ... in order: once every
  // streaming warp has counted its part, it finishes the unit (a row's
  // statistics and its pair; a draw's threshold and walk) and releases the
  // slot.  The streaming warps never wait on these global round trips.
  __device__ void finish_units(int f0) const {
    for (int k = f0;; k += kFin) {
      const int slot = k % kQ;
      // position k published, or END published before it
      int ok = 1;
      if (lane == 0 && q_seq[slot] != k) {
        const uint64_t end = now_ns() + p.wait_ns;
        for (;;) {
          if (q_seq[slot] == k) break;
          if (*q_end < k || *stop) {
            ok = 0;
            break;
          }
          if (now_ns() > end) {
            ok = -1;
            break;
          }
          __nanosleep(64);
        }
      }
      ok = __shfl_sync(kFull, ok, 0);
      if (ok < 0) halt();
      if (ok <= 0) break;
      __threadfence_block();
      __syncwarp();
      const Unit u = q_ent[slot];
      if (u.kind == kUEnd) break;
      const UInfo f = q_inf[slot].f;
      const DrawCtx dcx = q_inf[slot].dc;
      const float du = q_inf[slot].du;
      // every streaming warp done with position k
      if (lane == 0) {
        const int need = kNW * (k / kQ + 1);
        volatile int* cnt = q_cnt + slot;
        const uint64_t end = now_ns() + p.wait_ns;
        while (*cnt < need) {
          if (*stop || now_ns() > end) {
            ok = 0;
            break;
          }
          __nanosleep(32);
        }
      }
      ok = __shfl_sync(kFull, ok, 0);
      if (!ok) {
        halt();
        break;
      }
      __threadfence_block();
      __syncwarp();
      if (f.kind == kURow) {
        const uint4 r = lane < kNW ? q_rec[slot * kNW + lane] : make_uint4(0u, 0u, 0u, 0u);
        row_finish(r, f);
      } else {
        // one part: every chunk sum came from this CTA's warps; two parts:
        // the second part to finish (in either CTA) walks the draw
        bool last = true;
        if (C.dshift) {
          int parts = 0;
          if (lane == 0) {
            __threadfence();
            parts = atom_add_acq_rel(p.dpc + f.e, 1) + 1;
            if (parts == 2) p.dpc[f.e] = 0;
          }
          last = __shfl_sync(kFull, parts, 0) == 2;
        }
        if (last) draw_finish(f, dcx, du);
      }
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        q_fin[slot] = k;
      }
    }
  }

  __device__ static Part fresh_part() {
    Part P;
    P.m = -INFINITY;
    P.zh = P.zl = P.lx = 0.0f;
    P.key = 0ull;
    P.bad = 0;
    return P;
  }

  __device__ void stream() const {
    const uint64_t pol_first = policy_evict_first();
    int ik = 0, ic = 0, gi = 0;  // issue cursor: position, its next chunk; chunks issued
    int ck = 0, cc = 0, gc = 0;  // compute cursor: position, its next chunk; chunks computed
    bool iend = false, fi_ok = false, fc_ok = false;
    UInfo fi{}, fc{};
    Part P = fresh_part();
    float s2h = 0.0f, s2l = 0.0f;
    DrawCtx dctx{};
    for (;;) {
      // 1. keep two chunks in flight, across unit boundaries (vector path)
      if constexpr (VEC) {
        while (!iend && gi - gc < 2) {
          if (!fi_ok) {
            int pub = 0;
            if (lane == 0) pub = q_seq[ik % kQ] == ik;
            if (!__shfl_sync(kFull, pub, 0)) break;
            __threadfence_block();
            __syncwarp();
            const Unit u = q_ent[ik % kQ];
            if (u.kind == kUEnd) {
              iend = true;
              break;
            }
            fi = q_inf[ik % kQ].f;
            fi_ok = true;
            ic = 0;
          }
          if (ic >= ucount(fi, warp)) {
            ++ik;
            fi_ok = false;
            continue;
          }
          if (lane == 0) issue(fi, ic, gi, pol_first);
          ++ic;
          ++gi;
        }
      }
      // 2. the compute cursor's unit
      if (!fc_ok) {
        if (!wait_entry(ck)) {
          halt();
          break;
        }
        const Unit u = q_ent[ck % kQ];
        if (u.kind == kUEnd) break;
        const QInfo& qi = q_inf[ck % kQ];
        fc = qi.f;
        fc_ok = true;
        cc = 0;
        P = fresh_part();
        if (fc.kind == kURow) {
          s2h = qi.s2h;
          s2l = qi.s2l;
        } else {
          dctx = qi.dc;
        }
      }
      if (cc < ucount(fc, warp)) {
        const int cb = fc.kind == kURow ? kChunk : kHalf;
        const int off = sl_begin(warp) + (cbase(fc, warp) + cc) * cb;
        const int n_el = min(cb, sl_end(warp) - off) / static_cast<int>(sizeof(T));
        const void* st_src;
        const void* sd_src;
        if constexpr (VEC) {
          if (gc == gi) continue;  // its copy is issued in step 1 of the next pass
          int ok = 1;
          if (lane == 0) ok = wait_chunk(gc);
          if (!__shfl_sync(kFull, ok, 0)) {
            halt();
            break;
          }
          __syncwarp();
          st_src = buf_of(gc);
          sd_src = buf_of(gc) + kHalf;
        } else {
          st_src = fc.src_t + off;
          sd_src = fc.src_d ? fc.src_d + off : nullptr;
        }
        if (fc.kind == kURow) {
          row_chunk(st_src, n_el, off / static_cast<int>(sizeof(T)), fc, s2h, s2l, P);
        } else {
          const unsigned long long sum = sub_sum(dctx, st_src, sd_src, n_el);
          if (lane == 0) __stcg(p.rs + (static_cast<size_t>(fc.e) * kNW + warp) * p.ncd + cbase(fc, warp) + cc, sum);
        }
        if constexpr (VEC) fence_proxy_async();  // this buffer's reads before the copy into it
        __syncwarp();
        ++gc;
        ++cc;
        continue;
      }
      finalize(ck, fc, P, s2h, s2l);
      ++ck;
      fc_ok = false;
    }
    // No bulk copy may be in flight when the warp leaves.
    if constexpr (VEC) {
      if (lane == 0) {
        const uint64_t end = now_ns() + kDrainNs;
        for (int g = gc; g < gi; ++g)
          while (!mbar_poll(bar_of(g), static_cast<uint32_t>(g >> 1) & 1u) && now_ns() <= end) {
          }
      }
      __syncwarp();
    }
  }

  // ---- scheduler warp (lane 0) -----------------------------------------------
  // Pair (i, j)'s row dropped by early exit: counted with the skip mark; the
  // count that completes the pair ends it without a decision.
  __device__ void skip_row(int i, int j, int n) const {
    const bool greedy = !(eff_tau(p, i) > 0.0f);
    const int pid = i * (p.k_max + 1) + j;
    const int total = (!greedy && j < n) ? 2 : 1;
    const int add = 1 + (1 << 16);
    const int now = atom_add_acq_rel(p.pc + pid, add) + add;
    if ((now & 0xFFFF) == total) p.pc[pid] = 0;
  }

  struct Sched {
    int rb_next = -1;  // the next row unit, claimed one step ahead
    bool rows_done = false;
    int held = -1;     // a claimed draw index not listed yet
    int taken_seen = 0;
  };

  // The next unit for the queue: rows in slot order, else parts of listed
  // draws; END once every request's outputs are in (or a wait gave up).
  __device__ Unit claim(Sched& S) const {
    uint64_t idle_end = 0;
    for (;;) {
      if (*stop) return Unit{kUEnd, 0, 0, 0};
      // rows in slot order first: every decision, and so every draw, waits on them
      while (!S.rows_done) {
        const int rb = S.rb_next;
        if (rb < 0 || rb >= C.U || (p.flags & kFlagTestStall)) {
          S.rows_done = true;
          break;
        }
        S.rb_next = atomicAdd(p.ctrl + kCtlRow, 1);
        const Loc L = locate(C, rb);
        const int n = n_of(p, L.i);
        if (p.flags & kFlagEarlyExit) {
          const int a = settled(ld_relaxed(p.st + L.i), n);
          if (a >= 0 && L.j > a) {  // after the request's first rejection: not needed
            skip_row(L.i, L.j, n);
            continue;
          }
        }
        const long long row = L.isd ? drow_of(p, L.i, L.j) : trow_of(p, L.i, L.j);
        return Unit{kURow, L.i | (L.j << 12) | (L.isd << 16), static_cast<int>(row), 0};
      }
      // then parts of listed draws
      const int nd = ld_relaxed(p.ctrl + kCtlDraws);
      if (S.held < 0 && S.taken_seen < (nd << C.dshift)) {
        S.held = atomicAdd(p.ctrl + kCtlDrawTaken, 1);  // a part of a draw
        S.taken_seen = S.held + 1;
        if (S.held >= (2 * p.bs << C.dshift)) S.held = -1;  // past the draw list (never listed)
      }
      if (S.held >= 0 && (S.held >> C.dshift) < nd) {
        const int e = S.held >> C.dshift;
        int code = ld_acquire(p.dl + e);
        for (const uint64_t end = now_ns() + p.wait_ns; code == 0 && now_ns() <= end;)
          code = ld_acquire(p.dl + e);
        if (code == 0) {
          halt();
          return Unit{kUEnd, 0, 0, 0};
        }
        const Unit u{kUDraw, e, code, S.held & ((1 << C.dshift) - 1)};
        S.held = -1;
        return u;
      }
      if (ld_acquire(p.ctrl + kCtlReqDone) >= p.bs) return Unit{kUEnd, 0, 0, 0};
      const uint64_t t = now_ns();
      if (idle_end == 0) {
        idle_end = t + p.wait_ns;
      } else if (t > idle_end) {
        halt();
        return Unit{kUEnd, 0, 0, 0};
      }
      __nanosleep(200);
    }
  }

  __device__ void schedule() const {
    Sched S;
    S.rb_next = atomicAdd(p.ctrl + kCtlRow, 1);
    for (int k = 0;; ++k) {
      const int slot = k % kQ;
      bool ok = true;
      if (k >= kQ && q_fin[slot] != k - kQ) {  // the slot's previous unit must be complete
        const uint64_t end = now_ns() + p.wait_ns;
        while (q_fin[slot] != k - kQ) {
          if (*stop || now_ns() > end) {
            ok = false;
            break;
          }
          __nanosleep(64);
        }
      }
      if (!ok) halt();
      const Unit u = ok ? claim(S) : Unit{kUEnd, 0, 0, 0};
      if (u.kind != kUEnd) {
        QInfo qi;
        qi.f = info(u);
        qi.s2h = qi.s2l = 0.0f;
        qi.dc = DrawCtx{};
        qi.du = 0.0f;
        if (qi.f.kind == kURow) {
          if (!qi.f.greedy) scale_of(qi.f.tau, qi.s2h, qi.s2l);
        } else {
          qi.dc = draw_ctx(qi.f.i, qi.f.a, qi.f.dkind);
          qi.du = p.uniforms[static_cast<size_t>(qi.f.i) * (p.k_max + 1) + p.k_max];
        }
        q_inf[slot] = qi;
      }
      q_ent[slot] = u;
      if (u.kind == kUEnd) *q_end = k;  // finishing warps waiting on later positions leave
      __threadfence_block();
      q_seq[slot] = k;
      if (u.kind == kUEnd) break;
    }
  }
};

// ---------------------------------------------------------------------------

template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads, 1) sampler_kernel(const __grid_constant__ SamplerParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t s_full[kNW * 2];
  __shared__ Unit s_ent[kQ];
  __shared__ QInfo s_inf[kQ];
  __shared__ int s_seq[kQ], s_fin[kQ], s_cnt[kQ];
  __shared__ uint4 s_rec[kQ * kNW];
  __shared__ int s_stop, s_last, s_end;
  __shared__ int s_hist[32], s_base[32];
  __shared__ int s_WS[SD_MAX_K + 3], s_P[SD_MAX_K + 2], s_E[SD_MAX_K + 2];
  __shared__ float2 s_tab[16];
  __shared__ unsigned short s_heavy[kNW * kHeavyList];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bs = p.bs, K1 = p.k_max + 1;
  unsigned char* bufs = smem;
  int* order = reinterpret_cast<int*>(smem + static_cast<size_t>(kNW) * 2 * kChunk);  // [bs]
  // the buffers double as scratch for the request lengths while the tables are built
  int* nscr = reinterpret_cast<int*>(smem);  // [bs] bin of request i

  if (tid == 0) {
    s_stop = 0;
    s_end = INT_MAX;
  }
  if (tid < 32) s_hist[tid] = 0;
  if (tid < kQ) {
    s_seq[tid] = -1;
    s_fin[tid] = -1;
    s_cnt[tid] = 0;
  }
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
  // the bins were kept in the buffers; later bulk copies write there
  fence_proxy_async();
  // One thread initialises every buffer barrier and then fences: the fence
  // makes the initialising thread's own inits visible to the bulk copies'
  // completions (async proxy), so the inits and the fence share a thread.
  if (tid == 0) {
    for (int b = 0; b < 2 * kNW; ++b) mbar_init(&s_full[b], 1);
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
  // Each sampling request ends in one final draw.  With fewer than two per
  // CTA, the last draws would leave most CTAs idle while a few run two whole
  // draws: split each draw's chunks over two CTAs (their chunk sums meet in
  // the workspace, and the second part to finish walks the draw).  With more
  // draws the split only adds work (measured).
  C.dshift = (C.nsamp < 2 * static_cast<int>(gridDim.x) && p.ncd >= 2) ? 1 : 0;
  C.dper = (p.ncd + (1 << C.dshift) - 1) >> C.dshift;
  C.nw = K1;
  C.U = s_WS[K1];
  C.tab = s_tab;

  Sampler<T, VEC> S{p, C, s_ent, s_seq, s_fin, s_cnt, &s_end, s_inf, s_rec, bufs, s_heavy, s_full,
                    &s_stop, lane, warp, p.V * static_cast<int>(sizeof(T))};
  if (warp < kNW) {
    S.stream();
  } else if (warp == kNW) {
    if (lane == 0) S.schedule();
    // The CTA barrier below is warp-aligned: the scheduler warp reaches it
    // converged.
    __syncwarp();
  } else {
    S.finish_units(warp - kNW - 1);
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
    for (int i = tid; i < bs; i += kThreads) p.st[i] = 0;  // the requests' decision words
    if (ld_acquire(p.ctrl + kCtlStop)) {
      const int pairs = bs * K1;
      for (int q = tid; q < pairs; q += kThreads) p.pc[q] = 0;
      for (int i = tid; i < bs; i += kThreads) {
        p.accepted_len[i] = 0;
        for (int j = 0; j < K1; ++j)
          p.out_tokens[static_cast<size_t>(i) * K1 + j] = j == 0 ? 0 : -1;
      }
      for (int e = tid; e < 2 * bs; e += kThreads) {
        p.dl[e] = 0;
        p.dpc[e] = 0;
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

void sampler_geometry(int V, int elem, int* slice, int* ncr, int* ncd) {
  const long long R = static_cast<long long>(V) * elem;
  const long long sl = ((R + kNW - 1) / kNW + 15) / 16 * 16;
  *slice = static_cast<int>(sl > 0 ? sl : 16);
  *ncr = static_cast<int>((*slice + kChunk - 1) / kChunk);
  *ncd = static_cast<int>((*slice + kHalf - 1) / kHalf);
}

SamplerWs sampler_ws_layout(int bs, int k_max, int V, int elem) {
  auto al = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
  const size_t rows_t = static_cast<size_t>(bs) * (k_max + 1);
  const size_t rows_d = static_cast<size_t>(bs) * k_max;
  int slice, ncr, ncd;
  sampler_geometry(V, elem, &slice, &ncr, &ncd);
  SamplerWs L;
  L.rst = 0;
  L.rs = al(L.rst + (rows_t + rows_d) * sizeof(RowStat));
  L.zero = al(L.rs + 2 * static_cast<size_t>(bs) * kNW * ncd * 8);
  L.pc = L.zero;
  L.st = al(L.pc + rows_t * 4);
  L.dl = al(L.st + static_cast<size_t>(bs) * 4);
  L.dpc = al(L.dl + 2 * static_cast<size_t>(bs) * 4);
  L.ctrl = al(L.dpc + 2 * static_cast<size_t>(bs) * 4);
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
  const size_t need = static_cast<size_t>(kNW) * 2 * kChunk + tables;
  if (need > static_cast<size_t>(lim)) return cudaSuccess;
  // the buffers also hold the request bins while the tables are built
  if (static_cast<size_t>(kNW) * 2 * kChunk < static_cast<size_t>(bs) * 4) return cudaSuccess;
  out->nbuf = 2 * kNW;
  out->threads = kThreads;
  out->blocks = blocks > 0 ? std::min(blocks, sms) : sms;
  out->smem = need;
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
