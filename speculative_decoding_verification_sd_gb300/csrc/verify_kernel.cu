// verify_kernel.cu -- the sampling stage: speculative rejection sampling over
// the whole vocabulary in one persistent kernel.
//
// Rule (the original papers cited by the fosworld blog "추측 디코딩과 vLLM
// 적응형 검증" under "참고 링크 / 논문"; greedy form in "추측 디코딩이란";
// distribution-preserving per "속도, 메모리, 정확도에 주는 영향", row 정확도):
//   tau > 0: accept slot j iff u_j * q_j(x_j) <= p_j(x_j); at the first
//            rejection draw from max(p - q, 0) normalised; after a fully
//            accepted prefix draw a bonus token from p of the next row.
//   tau = 0: accept iff x_j == argmax p_j; the correction/bonus is the argmax.
//
// Design (GB300): one persistent CTA per SM, warp-specialised.  The work is
// a list of rows -- every compacted target row, and the draft row of every
// verified slot of a sampling request -- plus the residual draws, which are
// listed as requests are decided.  In each CTA, NT/32 - 3 streaming warps
// each own a contiguous range of every row and stream it from HBM through a
// private ring of bulk copies (mbarrier completion) into shared memory,
// reducing it to softmax statistics at the request's temperature (kept per
// chunk for target rows) or to the argmax, plus the logit at the draft
// token.  They never wait for one another.  The scheduling warp hands out
// the queue (a row from a global counter, or a slice of a listed residual
// draw), folds each unit once every streaming warp has arrived on the
// unit's barrier, stores the row statistics and counts the row for its
// request; when it counts a request's last row it queues the request's tail
// for one of the CTA's two draw warps, which takes the accept decisions and
// draws the final token: the argmax, a bonus token from p (the chunk
// statistics locate the crossing chunk, which alone is read again), or --
// after a rejection -- lists a residual draw, whose row pair is streamed
// again in slices by whichever CTAs claim them; the CTA that folds the last
// slice finishes the inverse CDF.  Inverse-CDF sums are exact 64-bit fixed
// point, so the crossing chunk does not depend on summation order.  The
// ordering between CTAs rides on the arrival counters (acquire-release
// read-modify-writes), not on GPU-scope fences, which wait for the memory
// traffic in flight.
#include <algorithm>
#include <atomic>
#include <climits>
#include <mutex>
#include <type_traits>

#include "sd_device.cuh"
#include "sd_internal.h"

namespace sdk {

namespace {

template <typename T, bool VEC>
struct VT;

// 16-byte vectors (V * elem % 16 == 0 and 16-byte aligned base pointers).
template <>
struct VT<float, true> {
  using Raw = float4;
  static constexpr int VE = 4;
  __device__ __forceinline__ static void unpack(const Raw& r, float (&f)[VE]) {
    f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w;
  }
};

template <>
struct VT<uint16_t, true> {  // bf16 bit patterns
  using Raw = uint4;
  static constexpr int VE = 8;
  __device__ __forceinline__ static void unpack(const Raw& r, float (&f)[VE]) {
    f[0] = __uint_as_float(r.x << 16); f[1] = __uint_as_float(r.x & 0xFFFF0000u);
    f[2] = __uint_as_float(r.y << 16); f[3] = __uint_as_float(r.y & 0xFFFF0000u);
    f[4] = __uint_as_float(r.z << 16); f[5] = __uint_as_float(r.z & 0xFFFF0000u);
    f[6] = __uint_as_float(r.w << 16); f[7] = __uint_as_float(r.w & 0xFFFF0000u);
  }
};

// Single elements (any V, any alignment).
template <>
struct VT<float, false> {
  using Raw = float;
  static constexpr int VE = 1;
  __device__ __forceinline__ static void unpack(const Raw& r, float (&f)[VE]) { f[0] = r; }
};

template <>
struct VT<uint16_t, false> {
  using Raw = uint16_t;
  static constexpr int VE = 1;
  __device__ __forceinline__ static void unpack(const Raw& r, float (&f)[VE]) {
    f[0] = __uint_as_float(static_cast<uint32_t>(r) << 16);
  }
};

// Element-path loads of the logits through the read-only data path.
template <typename Raw>
__device__ __forceinline__ Raw ld_stream(const Raw* p) {
  return __ldg(p);
}

template <typename Raw>
__device__ __forceinline__ void prefetch_l1(const Raw* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ float from_ordered(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// One thread's values into its running (max, scaled sum) at scale s2:
// z = sum 2^((l - m) * s2) with m the running maximum.  The exponent
// argument is formed as (l - m) * s2 (the rounding of m * s2 in l * s2 - m * s2
// would scale the whole sum; the vector path keeps that form and undoes the
// scale with bias_fix).  The arguments and the sum use packed fp32x2
// arithmetic.
template <int VE>
__device__ __forceinline__ void online_add(const float (&f)[VE], float s2, float& m, float& z) {
  float vm = f[0];
#pragma unroll
  for (int e = 1; e < VE; ++e) vm = fmaxf(vm, f[e]);
  if (vm > m) {
    z = (m == -INFINITY) ? 0.0f : z * exp2_ftz((m - vm) * s2);
    m = vm;
  }
  if (m != -INFINITY) {
    if constexpr (VE % 2 == 0) {
      const float2 s22 = make_float2(s2, s2);
      const float2 nm2 = make_float2(-m, -m);
      float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int e = 0; e < VE; e += 2) {
        const float2 t = __fmul2_rn(__fadd2_rn(make_float2(f[e], f[e + 1]), nm2), s22);
        acc = __fadd2_rn(acc, make_float2(exp2_ftz(t.x), exp2_ftz(t.y)));
      }
      z += acc.x + acc.y;
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e) z += exp2_ftz((f[e] - m) * s2);
    }
  }
}


// Packed bf16x2 maximum (NaN-ignoring / NaN-propagating), fp32 maximum that
// propagates NaN.
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Arrival counters with the ordering on the counter itself: a fence at GPU
// scope waits for the memory traffic in flight and costs microseconds while
// the SM streams, an acquire-release read-modify-write does not.
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void red_add_release(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

constexpr float kLn2 = 0.693147180559945309f;

// The hot loops form each exponent with one fused multiply-add, l * s2 - b
// with b = RN(M * s2).  That shifts every argument by the same amount, the
// rounding error of b: (l - M) * s2 = (l * s2 - b) - fma(M, s2, -b), where
// the fma is exact (the error of a rounded product is representable).  The
// shift is undone once per sum (or folded into a scale) by the factor
// 2^-fma(M, s2, -b) = 1 + c, |c| < 1e-6; this returns c.
__device__ __forceinline__ float bias_fix(float M, float s2, float b) {
  return __fmul_rn(-__fmaf_rn(M, s2, -b), kLn2);
}

// Running softmax statistics of one lane over a chunk: (m, z2) with
// z2.x + z2.y = sum 2^((l - m) * s2); the chunk's maximum is folded in once.
template <typename T>
struct ChunkOps;

template <>
struct ChunkOps<uint16_t> {  // 8 bf16 per 16-byte vector
  static constexpr uint32_t kNegInf2 = 0xFF80FF80u;
  __device__ __forceinline__ static uint4 neg_inf() {
    return make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
  }
  template <int N>
  __device__ __forceinline__ static void softmax(const uint4 (&r)[N], float s2, float& m,
                                                 float2& z2) {
    // per-vector maxima, then a tree over the vectors (short dependency chains)
    uint32_t vm[N];
#pragma unroll
    for (int q = 0; q < N; ++q) vm[q] = bmax2(bmax2(r[q].x, r[q].y), bmax2(r[q].z, r[q].w));
#pragma unroll
    for (int st = 1; st < N; st <<= 1)
#pragma unroll
      for (int q = 0; q + st < N; q += 2 * st) vm[q] = bmax2(vm[q], vm[q + st]);
    const float lm = fmaxf(bf_lo(vm[0]), bf_hi(vm[0]));
    if (lm > m) {
      if (m == -INFINITY) {
        z2 = make_float2(0.0f, 0.0f);
      } else {
        const float sc = exp2_ftz((m - lm) * s2);
        z2 = __fmul2_rn(z2, make_float2(sc, sc));
      }
      m = lm;
    }
    if (m != -INFINITY) {
      const float b = __fmul_rn(m, s2);
      const float2 s22 = make_float2(s2, s2), nb2 = make_float2(-b, -b);
      float2 acc[4];  // four independent partial sums, one per word of the vector
#pragma unroll
      for (int h = 0; h < 4; ++h) acc[h] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const uint32_t w4[4] = {r[q].x, r[q].y, r[q].z, r[q].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 t = __ffma2_rn(make_float2(bf_lo(w4[h]), bf_hi(w4[h])), s22, nb2);
          acc[h] = __fadd2_rn(acc[h], make_float2(exp2_ftz(t.x), exp2_ftz(t.y)));
        }
      }
      const float2 sum = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
      const float c = bias_fix(m, s2, b);
      z2 = __ffma2_rn(sum, make_float2(c, c), __fadd2_rn(z2, sum));
    }
  }
  // Running argmax of one lane: the first vector whose maximum strictly
  // exceeds the best so far is kept whole in registers (bvec, at vector
  // index bv); the element index is resolved once per row by first_of.
  template <int N>
  __device__ __forceinline__ static void argmax(const uint4 (&r)[N], int v0, float& best,
                                                uint4& bvec, int& bv, int& nanf) {
#pragma unroll
    for (int q = 0; q < N; ++q) {
      const uint32_t mx = bmax2_nan(bmax2_nan(r[q].x, r[q].y), bmax2_nan(r[q].z, r[q].w));
      const float lo = bf_lo(mx), hi = bf_hi(mx);
      nanf |= (lo != lo) | (hi != hi);
      const float vm = fmaxf(lo, hi);
      const bool up = vm > best;  // strictly larger: earlier vectors keep ties
      best = up ? vm : best;
      bvec = up ? r[q] : bvec;
      bv = up ? v0 + 32 * q : bv;
    }
  }
  // Lowest element index of `best` inside the kept vector.
  __device__ __forceinline__ static int first_of(const uint4& r, int v, float best) {
    const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
    int e = 7;
#pragma unroll
    for (int h = 3; h >= 0; --h) {
      if (bf_hi(w4[h]) == best) e = 2 * h + 1;
      if (bf_lo(w4[h]) == best) e = 2 * h;
    }
    return v * 8 + e;
  }
};

template <>
struct ChunkOps<float> {  // 4 fp32 per 16-byte vector
  __device__ __forceinline__ static float4 neg_inf() {
    return make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
  template <int N>
  __device__ __forceinline__ static void softmax(const float4 (&r)[N], float s2, float& m,
                                                 float2& z2) {
    float vm[N];
#pragma unroll
    for (int q = 0; q < N; ++q) vm[q] = fmaxf(fmaxf(r[q].x, r[q].y), fmaxf(r[q].z, r[q].w));
#pragma unroll
    for (int st = 1; st < N; st <<= 1)
#pragma unroll
      for (int q = 0; q + st < N; q += 2 * st) vm[q] = fmaxf(vm[q], vm[q + st]);
    const float lm = vm[0];
    if (lm > m) {
      if (m == -INFINITY) {
        z2 = make_float2(0.0f, 0.0f);
      } else {
        const float sc = exp2_ftz((m - lm) * s2);
        z2 = __fmul2_rn(z2, make_float2(sc, sc));
      }
      m = lm;
    }
    if (m != -INFINITY) {
      const float b = __fmul_rn(m, s2);
      const float2 s22 = make_float2(s2, s2), nb2 = make_float2(-b, -b);
      float2 a0 = make_float2(0.0f, 0.0f), a1 = make_float2(0.0f, 0.0f);  // independent sums
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const float2 t0 = __ffma2_rn(make_float2(r[q].x, r[q].y), s22, nb2);
        const float2 t1 = __ffma2_rn(make_float2(r[q].z, r[q].w), s22, nb2);
        a0 = __fadd2_rn(a0, make_float2(exp2_ftz(t0.x), exp2_ftz(t0.y)));
        a1 = __fadd2_rn(a1, make_float2(exp2_ftz(t1.x), exp2_ftz(t1.y)));
      }
      const float2 sum = __fadd2_rn(a0, a1);
      const float c = bias_fix(m, s2, b);
      z2 = __ffma2_rn(sum, make_float2(c, c), __fadd2_rn(z2, sum));
    }
  }
  template <int N>
  __device__ __forceinline__ static void argmax(const float4 (&r)[N], int v0, float& best,
                                                float4& bvec, int& bv, int& nanf) {
#pragma unroll
    for (int q = 0; q < N; ++q) {
      const float vm = fmax_nan(fmax_nan(r[q].x, r[q].y), fmax_nan(r[q].z, r[q].w));
      nanf |= vm != vm;
      const bool up = vm > best;
      best = up ? vm : best;
      bvec = up ? r[q] : bvec;
      bv = up ? v0 + 32 * q : bv;
    }
  }
  __device__ __forceinline__ static int first_of(const float4& r, int v, float best) {
    int e = 3;
    if (r.z == best) e = 2;
    if (r.y == best) e = 1;
    if (r.x == best) e = 0;
    return v * 4 + e;
  }
};

constexpr int kUnroll = 8;                 // element path: loads in flight per lane
constexpr int kSlots = 2;                  // ring slots per streaming warp
constexpr uint32_t kSpinLimit = 1u << 22;  // polls (~100 ns apart) before a wait gives up
// log2(e) split into two floats (hi + lo) for a double-float exponent.
constexpr float kLog2eHi = 1.44269502162933349609375f;
constexpr float kLog2eLo = 1.925963033500011079e-08f;
constexpr float kTwo40 = 1099511627776.0f;            // 2^40
constexpr float kTwo56 = 72057594037927936.0f;        // 2^56
constexpr float kTwo64 = 18446744073709551616.0f;     // 2^64

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// 2^(d * s2) with d = l - M given as (d_hi, d_lo) and s2 = s2_hi + s2_lo: the
// exponent is formed in double-float so its rounding does not depend on |d|
// (the accept test's p(x) and q(x)).  Written with explicitly rounded
// intrinsics so that its value does not depend on how it is compiled.
__device__ __forceinline__ float exp2_df(float d_hi, float d_lo, float s2_hi, float s2_lo) {
  const float t_hi = __fmul_rn(d_hi, s2_hi);
  const float t_lo = __fadd_rn(__fmaf_rn(d_hi, s2_hi, -t_hi),
                               __fmaf_rn(d_hi, s2_lo, __fmul_rn(d_lo, s2_hi)));
  const float e = exp2_ftz(t_hi);
  return __fmaf_rn(__fmul_rn(e, kLn2), t_lo, e);
}

// l - M split exactly into (hi, lo) (Knuth's two-sum).
__device__ __forceinline__ void two_diff(float l, float M, float& hi, float& lo) {
  hi = __fsub_rn(l, M);
  const float bb = __fsub_rn(hi, l);
  lo = __fadd_rn(__fsub_rn(l, __fsub_rn(hi, bb)), __fsub_rn(-M, bb));
}

// ---------------------------------------------------------------------------
// Layout of one row for a launch with NS streaming warps.  The row's units
// (16-byte vectors, or elements on the element path) are cut into nch
// chunks of CU units; streaming warp w owns chunks [w * cpw, (w + 1) * cpw).
// On the vector path a chunk is one bulk copy of at most kSlotBytes.  The
// statistics chunks group g consecutive chunks of one warp (spw per warp,
// NS * spw <= kStatStride).  A residual draw is streamed in S_sl slices:
// slice s takes chunks [s * m_sl, (s + 1) * m_sl) of every warp's range
// (as many slices as make every slice non-empty, at most kMaxSlices).
struct Geom {
  int nvec, cpw, CU, nch, g, spw, S_sl, m_sl;
};

constexpr int kSlotBytes = 4352;  // largest chunk of the vector path (272 vectors)
constexpr int kMaxSlices = 8;     // slices of one residual draw

__device__ __forceinline__ Geom make_geom(int nvec, bool vec, int ns) {
  Geom G;
  G.nvec = nvec;
  if (vec) {
    constexpr int kMaxVec = kSlotBytes / 16;
    G.cpw = max(1, (nvec + ns * kMaxVec - 1) / (ns * kMaxVec));
    G.CU = (nvec + ns * G.cpw - 1) / (ns * G.cpw);
  } else {
    G.cpw = 4;
    G.CU = 32 * ((nvec + ns * G.cpw * 32 - 1) / (ns * G.cpw * 32));
  }
  G.nch = (nvec + G.CU - 1) / G.CU;
  const int spw_max = kStatStride / ns;
  G.g = (G.cpw + spw_max - 1) / spw_max;
  G.spw = (G.cpw + G.g - 1) / G.g;
  G.S_sl = min(kMaxSlices, G.cpw);
  G.m_sl = (G.cpw + G.S_sl - 1) / G.S_sl;
  G.S_sl = (G.cpw + G.m_sl - 1) / G.m_sl;  // no empty slice
  return G;
}

// Units [ub, ue) of statistics chunk sc (empty when past the row's end).
__device__ __forceinline__ void stat_units(const Geom& G, int sc, int& ub, int& ue) {
  const int w = sc / G.spw, j = sc - w * G.spw;
  const int c0 = min(G.nch, w * G.cpw + j * G.g);
  const int c1 = min(G.nch, min(w * G.cpw + (j + 1) * G.g, (w + 1) * G.cpw));
  ub = min(G.nvec, c0 * G.CU);
  ue = min(G.nvec, c1 * G.CU);
  if (c1 <= c0) ue = ub;
}

// Release / acquire on a shared-memory word between the warps of a CTA.
__device__ __forceinline__ void st_release_cta(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.s32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
// Relaxed shared-memory read for polling; the poll ends with an acquire.
__device__ __forceinline__ int ld_volatile_cta(const int* p) {
  return *reinterpret_cast<const volatile int*>(p);
}

__device__ __forceinline__ int ld_acquire_cta(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.s32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Per-CTA state shared by the warps: request tables in shared memory and
// the unit queue.  Position k of the queue is published in q[k % kDepth]
// once pub >= k; the control warp keeps at most kWindow positions published
// ahead of the last one it has folded.
constexpr int kDepth = 4;
constexpr int kWindow = 2;  // a unit streaming, one published behind it

struct Cta {
  const int* cu;     // [bs+1] cu_seqlens
  const float* tau;  // [bs] temperatures (invalid ones as 0)
  const int* order;  // [bs] request order of the work list
  const int* ustart; // [bs+1] first row unit of order[k]
  int* q;            // [kDepth] queue
  int* qx;           // [kDepth] of a slice: its draw's request and slot (i << 4 | a)
  int* pub;          // last published position
  int nsamp;         // sampling requests
  int U_rows;        // row units
};

// Row unit u -> (request, slot, kind, row index).
struct Unit {
  int i, j, n, c0;
  bool draft, greedy;
  size_t row;
};

__device__ __forceinline__ Unit locate(const Cta& C, int bs, int u) {
  int lo = 0, hi = bs;  // ustart[lo] <= u < ustart[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (C.ustart[mid] <= u) lo = mid;
    else hi = mid;
  }
  Unit t;
  t.i = C.order[lo];
  const int r = u - C.ustart[lo];
  t.c0 = C.cu[t.i];
  t.n = C.cu[t.i + 1] - t.c0 - 1;
  t.greedy = !(C.tau[t.i] > 0.0f);
  t.draft = r > t.n;
  t.j = t.draft ? r - (t.n + 1) : r;
  t.row = t.draft ? static_cast<size_t>(t.c0 - t.i + t.j) : static_cast<size_t>(t.c0 + t.j);
  return t;
}

// Queue entries past the rows: slice s of listed residual draw e, as
// kResBase | e << 8 | s (e < 4096, s < 256); the draw's request i and slot a
// travel beside it in the queue's side array, as i << 4 | a.  kEnd closes
// the queue.
constexpr int kResBase = 1 << 30;
constexpr int kEnd = INT_MAX;
constexpr int kWait = INT_MAX - 1;  // scheduler: nothing to hand out yet
__device__ __forceinline__ bool is_slice(int u) { return u >= kResBase && u < kWait; }

// ---------------------------------------------------------------------------
// Weight functions of the final draws.  A draw from p (target row rt, max
// Mt, scale s2 = log2(e)/tau) weighs an element 2^((l - Mt) s2) <= 1 (2^40
// fixed point); a residual draw adds the draft row rd (max Md) and both 1/Z
// and weighs max(p - q, 0) <= 1 (2^56).  All in fp32 with the hardware
// exponent; a unit's weight is the fixed-point value of its fp32 sum (what
// the residual slices add into the chunk sums, so the walk of the crossing
// chunk retraces those sums exactly), an element's weight its own fixed-point
// value.
template <typename Raw>
struct DrawRows {
  const Raw* rt;  // unit u at rt[u - off] (off > 0: a staged copy in shared memory)
  const Raw* rd;
  float Mt, Md, s2;
  float bt, bd;    // RN(Mt * s2), RN(Md * s2): exponent arguments l * s2 - b
  float iZt, iZd;  // 1 / Z, each times the correction of its bias (bias_fix)
  float sp;        // 2^40 times the target bias's correction (draws from p)
  int off;
};

template <typename T, bool VEC>
__device__ __forceinline__ DrawRows<typename VT<T, VEC>::Raw> make_rows(
    const VerifyParams& p, const int* cu, int i, int a, float tau, const float4& ts,
    const float4& ds, bool resid) {
  using Raw = typename VT<T, VEC>::Raw;
  DrawRows<Raw> w;
  const int c0 = cu[i];
  w.rt = reinterpret_cast<const Raw*>(static_cast<const T*>(p.target) +
                                      static_cast<size_t>(c0 + a) * p.V);
  w.rd = resid ? reinterpret_cast<const Raw*>(static_cast<const T*>(p.draft) +
                                              static_cast<size_t>(c0 - i + a) * p.V)
               : w.rt;
  w.Mt = ts.x;
  w.Md = ds.x;
  w.s2 = kLog2e / tau;
  w.bt = __fmul_rn(w.Mt, w.s2);
  w.bd = __fmul_rn(w.Md, w.s2);
  // no correction for a non-finite maximum (the weights are not finite then)
  const float ct = fabsf(w.bt) < INFINITY ? bias_fix(w.Mt, w.s2, w.bt) : 0.0f;
  const float cd = fabsf(w.bd) < INFINITY ? bias_fix(w.Md, w.s2, w.bd) : 0.0f;
  const float izt = 1.0f / ts.y, izd = 1.0f / ds.y;
  w.iZt = __fmaf_rn(izt, ct, izt);
  w.iZd = __fmaf_rn(izd, cd, izd);
  w.sp = __fmaf_rn(kTwo40, ct, kTwo40);
  w.off = 0;
  return w;
}

// max(p - q, 0) of one element (biases bt, bd; iZt, iZd carry their corrections)
__device__ __forceinline__ float res_weight(float f, float g, float s2, float bt, float bd,
                                            float iZt, float iZd) {
  const float et = exp2_ftz(fmaf(f, s2, -bt));
  const float ed = exp2_ftz(fmaf(g, s2, -bd));
  return fmaxf(fmaf(et, iZt, -__fmul_rn(ed, iZd)), 0.0f);
}

template <typename T, bool VEC>
__device__ __forceinline__ float fast_res(const DrawRows<typename VT<T, VEC>::Raw>& w,
                                          const typename VT<T, VEC>::Raw& ra,
                                          const typename VT<T, VEC>::Raw& rb) {
  using Tr = VT<T, VEC>;
  float f[Tr::VE], g[Tr::VE];
  Tr::unpack(ra, f);
  Tr::unpack(rb, g);
  float ws = 0.0f;
#pragma unroll
  for (int e = 0; e < Tr::VE; ++e) ws += res_weight(f[e], g[e], w.s2, w.bt, w.bd, w.iZt, w.iZd);
  return ws;
}

// Residual draw: unit u's weight, and its elements' weights.
template <typename T, bool VEC>
__device__ __forceinline__ unsigned long long unit_res(const DrawRows<typename VT<T, VEC>::Raw>& w,
                                                       int u) {
  return __float2ull_rn(__fmul_rn(fast_res<T, VEC>(w, w.rt[u - w.off], w.rd[u - w.off]), kTwo56));
}
template <typename T, bool VEC>
__device__ __forceinline__ void elem_res(const DrawRows<typename VT<T, VEC>::Raw>& w, int u,
                                         unsigned long long (&wi)[VT<T, VEC>::VE]) {
  using Tr = VT<T, VEC>;
  float f[Tr::VE], g[Tr::VE];
  Tr::unpack(w.rt[u - w.off], f);
  Tr::unpack(w.rd[u - w.off], g);
#pragma unroll
  for (int e = 0; e < Tr::VE; ++e)
    wi[e] = __float2ull_rn(__fmul_rn(res_weight(f[e], g[e], w.s2, w.bt, w.bd, w.iZt, w.iZd), kTwo56));
}

// Draw from p: unit u's weight, and its elements' weights.
template <typename T, bool VEC>
__device__ __forceinline__ unsigned long long unit_p(const DrawRows<typename VT<T, VEC>::Raw>& w,
                                                     int u) {
  using Tr = VT<T, VEC>;
  float f[Tr::VE];
  Tr::unpack(w.rt[u - w.off], f);
  float ws = 0.0f;
#pragma unroll
  for (int e = 0; e < Tr::VE; ++e) ws += exp2_ftz(fmaf(f[e], w.s2, -w.bt));
  return __float2ull_rn(__fmul_rn(ws, w.sp));
}
template <typename T, bool VEC>
__device__ __forceinline__ void elem_p(const DrawRows<typename VT<T, VEC>::Raw>& w, int u,
                                       unsigned long long (&wi)[VT<T, VEC>::VE]) {
  using Tr = VT<T, VEC>;
  float f[Tr::VE];
  Tr::unpack(w.rt[u - w.off], f);
#pragma unroll
  for (int e = 0; e < Tr::VE; ++e) wi[e] = __float2ull_rn(__fmul_rn(exp2_ftz(fmaf(f[e], w.s2, -w.bt)), w.sp));
}

// ---------------------------------------------------------------------------
// A streaming warp: walks the queue, streams its chunk range of every unit
// (through its ring of bulk copies on the vector path), leaves the unit's
// partial results in shared memory and arrives on the unit's barrier.
// Streaming warps never wait for one another.
template <typename T, bool VEC, int NS>
struct Streamer {
  using Tr = VT<T, VEC>;
  using Raw = typename Tr::Raw;
  static constexpr int VE = Tr::VE;

  const VerifyParams& p;
  const Cta& C;
  const Geom& G;
  const int w, lane;
  unsigned char* ring;      // this warp's kSlots slots
  uint64_t* bar;            // this warp's kSlots barriers
  const int cb, ce;         // this warp's chunks
  uint32_t cseq = 0, iseq = 0;   // ring entries consumed / issued
  int fk = 0, fe = 0, f_n = 0, f_c0 = 0, fk_cached = -1;
  bool f_two = false;
  const char* f_base = nullptr;
  const char* f_base2 = nullptr;

  __device__ Streamer(const VerifyParams& p_, const Cta& C_, const Geom& G_, int w_, int lane_,
                      unsigned char* ring_all, uint64_t* bar_all)
      : p(p_), C(C_), G(G_), w(w_), lane(lane_),
        ring(ring_all + static_cast<size_t>(w_) * kSlots * kSlotBytes),
        bar(bar_all + w_ * kSlots),
        cb(min(G_.nch, w_ * G_.cpw)), ce(min(G_.nch, w_ * G_.cpw + G_.cpw)) {}

  __device__ size_t row_bytes() const { return static_cast<size_t>(G.nvec) * 16; }

  // Issues ring entries up to kSlots ahead of consumption, across published
  // positions.  A row position takes one entry per chunk of [cb, ce); a
  // slice takes two (target chunk, then draft chunk) per chunk of its part.
  __device__ void refill() {
    while (iseq - cseq < static_cast<uint32_t>(kSlots)) {
      if (fk_cached != fk) {
        // every lane acquires the counter and all act on the smallest value
        // seen, so the lanes take the same trips through this loop and each
        // has synchronised with the publication it acts on
        if (fk > __reduce_min_sync(kFull, ld_acquire_cta(C.pub))) break;
        const int u = C.q[fk % kDepth];
        if (u == kEnd) break;
        f_two = false;
        f_n = 0;
        if (u < C.U_rows) {
          const Unit t = locate(C, p.bs, u);
          f_base = reinterpret_cast<const char*>(t.draft ? p.draft : p.target) + t.row * row_bytes();
          f_c0 = cb;
          f_n = ce - cb;
        } else if (is_slice(u)) {
          const int ia = C.qx[fk % kDepth];
          const int i = (ia >> 4) & 0xFFF, a = ia & 15, s = u & 0xFF;
          const int c0 = C.cu[i];
          f_base = reinterpret_cast<const char*>(p.target) + static_cast<size_t>(c0 + a) * row_bytes();
          f_base2 = reinterpret_cast<const char*>(p.draft) + static_cast<size_t>(c0 - i + a) * row_bytes();
          f_c0 = min(ce, cb + s * G.m_sl);
          f_n = 2 * (min(ce, f_c0 + G.m_sl) - f_c0);
          f_two = true;
        }
        fk_cached = fk;
        fe = 0;
      }
      if (fe >= f_n) {
        ++fk;
        continue;
      }
      const int c = f_c0 + (f_two ? fe >> 1 : fe);
      const char* base = (f_two && (fe & 1)) ? f_base2 : f_base;
      const int slot = static_cast<int>(iseq % kSlots);
      const size_t off = static_cast<size_t>(c) * G.CU * 16;
      const uint32_t bytes = static_cast<uint32_t>(min(static_cast<size_t>(G.CU) * 16, row_bytes() - off));
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar[slot], bytes);
        // logits are read once: first out of L2, so the small per-call data
        // (statistics, counters, the next call's planner inputs) stays
        bulk_load(ring + slot * kSlotBytes, base + off, bytes, &bar[slot], policy_evict_first());
      }
      ++iseq;
      ++fe;
    }
    __syncwarp();  // lane 0's copies are issued before any lane waits on them
  }

  // Waits for ring entry `seq`; returns its data.
  __device__ const Raw* entry(uint32_t seq, int* err) {
    const int slot = static_cast<int>(seq % kSlots);
    const bool ok = __all_sync(kFull, mbar_wait_bounded(&bar[slot], (seq / kSlots) & 1, 1u << 24));
    if (!ok && lane == 0) raise_error(err, SD_DEV_ERR_TIMEOUT);
    return reinterpret_cast<const Raw*>(ring + slot * kSlotBytes);
  }

  // Statistics chunk of chunk c of this warp.
  __device__ int stat_of(int c) const { return w * G.spw + (c - w * G.cpw) / G.g; }
  __device__ bool stat_ends(int c) const {
    return c + 1 == ce || (c + 1 - w * G.cpw) % G.g == 0;
  }

  // Running (max, scaled sum) at scale s2 with one more (mc, zc) folded in.
  __device__ static void combine(float& M, float& Z, float mc, float zc, float s2) {
    if (mc == -INFINITY) return;
    if (M == -INFINITY) {
      M = mc;
      Z = zc;
    } else if (mc > M) {
      Z = fmaf(Z, exp2_ftz((M - mc) * s2), zc);
      M = mc;
    } else {
      Z = fmaf(zc, exp2_ftz((mc - M) * s2), Z);
    }
  }

  // The warp's (max, scaled sum) of one chunk from the lanes' values.
  __device__ static void chunk_reduce(float m, float z, float s2, float& mc, float& zc) {
    mc = warp_max(m);
    zc = warp_sum((m == -INFINITY || mc == -INFINITY) ? 0.0f : z * exp2_ftz((m - mc) * s2));
  }

  __device__ static float element_of(const Raw* d, int idx) {
    if constexpr (sizeof(T) == 2)
      return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(d)[idx]) << 16);
    else
      return reinterpret_cast<const float*>(d)[idx];
  }

  // Row unit u at queue position k: softmax statistics at the request's
  // temperature (per chunk, kept for target rows of sampling requests) or
  // the argmax, and the logit at the slot's draft token.
  __device__ void row(int k, int u, float (*red_m)[NS], float (*red_z)[NS],
                      unsigned long long (*red_k)[NS], int (*red_n)[NS], float* s_lx,
                      unsigned long long* sbuf) {
    const Unit t = locate(C, p.bs, u);
    const int x = t.j < t.n ? p.draft_ids[t.c0 - t.i + t.j] : -1;
    const bool x_ok = x >= 0 && x < p.V;
    const float tau = C.tau[t.i];
    const float s2 = t.greedy ? 0.0f : kLog2e / tau;
    const bool keep = !t.greedy && !t.draft;
    const Raw* rowp = reinterpret_cast<const Raw*>(
        reinterpret_cast<const char*>(t.draft ? p.draft : p.target) + t.row * (static_cast<size_t>(p.V) * sizeof(T)));
    float best = -INFINITY;  // greedy
    int bv = -1, nanf = 0, bidx = INT_MAX;
    Raw bvec{};
    float Mw = -INFINITY, Zw = 0.0f, Ms = -INFINITY, Zs = 0.0f;  // sampling: range, stat chunk
    for (int c = cb; c < ce; ++c) {
      const int u0 = c * G.CU, nv = min(G.CU, G.nvec - u0);
      float mc = -INFINITY, zc = 0.0f;
      if constexpr (VEC) {
        const Raw* d = entry(cseq, p.err);
        if (x_ok && lane == 0 && x / VE >= u0 && x / VE < u0 + nv) s_lx[k % kDepth] = element_of(d, x - u0 * VE);
        constexpr int VPL = (kSlotBytes / 16 + 31) / 32;  // vectors per lane and chunk
        Raw rv[VPL];
#pragma unroll
        for (int q = 0; q < VPL; ++q) rv[q] = lane + 32 * q < nv ? d[lane + 32 * q] : ChunkOps<T>::neg_inf();
        if (t.greedy) {
          ChunkOps<T>::argmax(rv, u0 + lane, best, bvec, bv, nanf);
        } else {
          float m = -INFINITY;
          float2 z2 = make_float2(0.0f, 0.0f);
          ChunkOps<T>::softmax(rv, s2, m, z2);
          chunk_reduce(m, z2.x + z2.y, s2, mc, zc);
        }
        __syncwarp();
        ++cseq;
        refill();
      } else {
        float m = -INFINITY, z = 0.0f;
        for (int v0 = u0 + lane; v0 < u0 + nv; v0 += 32 * kUnroll) {
          Raw rv[kUnroll];
#pragma unroll
          for (int q = 0; q < kUnroll; ++q)
            if (v0 + 32 * q < u0 + nv) rv[q] = ld_stream(rowp + v0 + 32 * q);
#pragma unroll
          for (int q = 0; q < kUnroll; ++q) {
            const int v = v0 + 32 * q;
            if (v < u0 + nv) {
              float f[VE];
              Tr::unpack(rv[q], f);
              if (v == x) s_lx[k % kDepth] = f[0];
              if (t.greedy) {
                nanf |= (f[0] != f[0]);
                if (f[0] > best) { best = f[0]; bidx = v; }
              } else {
                online_add<VE>(f, s2, m, z);
              }
            }
          }
        }
        if (!t.greedy) chunk_reduce(m, z, s2, mc, zc);
      }
      if (!t.greedy) {
        combine(Ms, Zs, mc, zc, s2);
        combine(Mw, Zw, mc, zc, s2);
        if (stat_ends(c)) {
          if (keep && lane == 0)
            sbuf[stat_of(c)] = static_cast<unsigned long long>(__float_as_uint(Ms)) |
                               (static_cast<unsigned long long>(__float_as_uint(Zs)) << 32);
          Ms = -INFINITY;
          Zs = 0.0f;
        }
      }
    }
    if (t.greedy) {
      if constexpr (VEC) bidx = bv >= 0 ? ChunkOps<T>::first_of(bvec, bv, best) : INT_MAX;
      unsigned long long key = bidx == INT_MAX ? 0ull
          : (static_cast<unsigned long long>(ordered_bits(best)) << 32) |
                static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(bidx));
      key = warp_max_u64(key);
      nanf = __any_sync(kFull, nanf);
      if (lane == 0) {
        red_k[k % kDepth][w] = key;
        red_n[k % kDepth][w] = nanf;
      }
    } else if (lane == 0) {
      red_m[k % kDepth][w] = Mw;
      red_z[k % kDepth][w] = Zw;
    }
  }

  // Slice unit u: this warp's part of a listed residual draw, summed per
  // statistics chunk in 2^56 fixed point into the draw's chunk sums.
  __device__ void slice(int u, int ia, unsigned long long* sbuf) {
    const int s = u & 0xFF, i = (ia >> 4) & 0xFFF, a = ia & 15;
    const int c0 = C.cu[i];
    const float4 ts = __ldcg(reinterpret_cast<const float4*>(p.st_t + c0 + a));
    const float4 ds = __ldcg(reinterpret_cast<const float4*>(p.st_d + c0 - i + a));
    const DrawRows<Raw> wr = make_rows<T, VEC>(p, C.cu, i, a, C.tau[i], ts, ds, true);
    if (lane == 0)
      for (int j = 0; j < G.spw; ++j) sbuf[w * G.spw + j] = 0;  // chunks this slice misses
    const int c_lo = min(ce, cb + s * G.m_sl), c_hi = min(ce, c_lo + G.m_sl);
    unsigned long long acc = 0;
    for (int c = c_lo; c < c_hi; ++c) {
      const int u0 = c * G.CU, nv = min(G.CU, G.nvec - u0);
      if constexpr (VEC) {
        const Raw* dt = entry(cseq, p.err);
        const Raw* dd = entry(cseq + 1, p.err);
        constexpr int VPL = (kSlotBytes / 16 + 31) / 32;
#pragma unroll 2
        for (int q = 0; q < VPL; ++q) {
          const int v = lane + 32 * q;
          if (v < nv) acc += __float2ull_rn(__fmul_rn(fast_res<T, VEC>(wr, dt[v], dd[v]), kTwo56));
        }
        __syncwarp();
        cseq += 2;
        refill();
      } else {
        for (int v0 = u0 + lane; v0 < u0 + nv; v0 += 32 * kUnroll) {
          Raw at[kUnroll], ad[kUnroll];
#pragma unroll
          for (int q = 0; q < kUnroll; ++q)
            if (v0 + 32 * q < u0 + nv) {
              at[q] = ld_stream(wr.rt + v0 + 32 * q);
              ad[q] = ld_stream(wr.rd + v0 + 32 * q);
            }
#pragma unroll
          for (int q = 0; q < kUnroll; ++q)
            if (v0 + 32 * q < u0 + nv)
              acc += __float2ull_rn(__fmul_rn(fast_res<T, VEC>(wr, at[q], ad[q]), kTwo56));
        }
      }
      if (stat_ends(c) || c + 1 == c_hi) {
        const unsigned long long sum = warp_sum_u64(acc);
        if (lane == 0) sbuf[stat_of(c)] = sum;
        acc = 0;
      }
    }
  }

  __device__ void run(uint64_t* pbar, float (*red_m)[NS], float (*red_z)[NS],
                      unsigned long long (*red_k)[NS], int (*red_n)[NS], float* s_lx,
                      unsigned long long (*s_stat)[kStatStride]) {
    for (int k = 0;; ++k) {
      bool ok = false;
      for (uint32_t it = 0; it < kSpinLimit; ++it) {
        if (ld_volatile_cta(C.pub) >= k) {
          ok = ld_acquire_cta(C.pub) >= k;
          break;
        }
        __nanosleep(64);
      }
      ok = __all_sync(kFull, ok);  // the same verdict in every lane
      if (!ok) {
        if (lane == 0) raise_error(p.err, SD_DEV_ERR_TIMEOUT);
        break;
      }
      const int u = C.q[k % kDepth];
      if (u == kEnd) break;
      if constexpr (VEC) refill();
      if (u < C.U_rows) row(k, u, red_m, red_z, red_k, red_n, s_lx, s_stat[k % kDepth]);
      else if (is_slice(u)) slice(u, C.qx[k % kDepth], s_stat[k % kDepth]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&pbar[k % kDepth]);
    }
    // entries issued but never consumed exist only after a time-out
    if constexpr (VEC) {
      while (cseq != iseq) {
        entry(cseq, p.err);
        ++cseq;
      }
    }
  }
};

// ---------------------------------------------------------------------------
// The control warps.  The scheduling warp hands out the queue, folds each
// finished unit, and queues the tail of every request whose last row it
// folds and the finish of every residual draw whose last slice it folds; the
// two draw warps take those jobs.  Scheduling is lane 0's; folds, tails and
// draws use the whole warp.
template <typename T, bool VEC, int NS>
struct Control {
  using Tr = VT<T, VEC>;
  using Raw = typename Tr::Raw;
  static constexpr int VE = Tr::VE;
  static constexpr int kCpl = (kStatStride + 31) / 32;  // statistics chunks per lane
  static constexpr int kWalk = 12;                       // units per lane in one walk round
  static constexpr int kJobs = 64;                       // job ring capacity
  static constexpr int kScratch = 40;                    // per-lane values of a warp-wide search

  const VerifyParams& p;
  const Cta& C;
  const Geom& G;
  const int lane;
  uint64_t* pbar;
  float (*red_m)[NS];
  float (*red_z)[NS];
  unsigned long long (*red_k)[NS];
  int (*red_n)[NS];
  float* s_lx;
  unsigned long long* s_walk;  // [32][kWalk] unit sums of the walk in hand, then [kScratch] (per draw warp)
  int* jobs;                   // [kJobs] job ring
  int* jtail;                  // jobs appended
  int* jhead;                  // jobs taken
  int* jdone;                  // jobs read
  unsigned long long (*s_stat)[kStatStride];  // per-chunk results of the units in flight
  unsigned char* cbuf;         // [2][kSlotBytes] staged chunk of the walk in hand (draw warps)
  uint64_t* cbar;              // its barrier
  mutable uint32_t cphase = 0;
  // lane 0's scheduler state: rows ran out; the next row id, fetched one
  // schedule ahead; a slice slot taken before its draw was listed
  bool rows_done = false;
  bool dealt = false;  // every row was dealt at the start
  int stash = 0, held = -1;
  mutable int last_ia = 0;  // request and slot of the last slice handed out

  __device__ Control(const VerifyParams& p_, const Cta& C_, const Geom& G_, int lane_,
                     uint64_t* pbar_, float (*rm)[NS], float (*rz)[NS],
                     unsigned long long (*rk)[NS], int (*rn)[NS], float* lx,
                     unsigned long long* walk_buf, int* jobs_, int* jtail_, int* jhead_,
                     int* jdone_, unsigned long long (*stat_)[kStatStride], unsigned char* cbuf_,
                     uint64_t* cbar_)
      : p(p_), C(C_), G(G_), lane(lane_), pbar(pbar_), red_m(rm), red_z(rz), red_k(rk),
        red_n(rn), s_lx(lx), s_walk(walk_buf), jobs(jobs_), jtail(jtail_), jhead(jhead_),
        jdone(jdone_), s_stat(stat_), cbuf(cbuf_), cbar(cbar_) {}

  // Copies units [ub, ue) of the draw's row (and draft row) into this warp's
  // buffer with bulk copies (vector path, one chunk at most) and points w at
  // the copy; false when the range does not qualify.
  __device__ bool stage(DrawRows<Raw>& w, bool two, int ub, int ue) const {
    if constexpr (!VEC) {
      return false;
    } else {
      const uint32_t bytes = static_cast<uint32_t>(ue - ub) * 16u;
      if (ue <= ub || bytes > static_cast<uint32_t>(kSlotBytes)) return false;
      if (lane == 0) {
        fence_proxy_async();  // earlier reads of the buffer before the copies
        mbar_arrive_expect_tx(cbar, two ? 2 * bytes : bytes);
        bulk_load_nohint(cbuf, w.rt + ub, bytes, cbar);
        if (two) bulk_load_nohint(cbuf + kSlotBytes, w.rd + ub, bytes, cbar);
      }
      // The copies are issued before any lane starts waiting for them: lanes
      // left to spin ahead of lane 0 could hold the warp until their wait
      // gives up and then read the buffer before it has landed.
      __syncwarp();
      const bool ok = __all_sync(kFull, mbar_wait_bounded(cbar, cphase & 1, 1u << 24));
      if (!ok && lane == 0) raise_error(p.err, SD_DEV_ERR_TIMEOUT);
      ++cphase;
      w.rt = reinterpret_cast<const Raw*>(cbuf);
      w.rd = two ? reinterpret_cast<const Raw*>(cbuf + kSlotBytes) : w.rt;
      w.off = ub;
      return true;
    }
  }

  // ---- scheduling (lane 0) ------------------------------------------------
  // ctrl[0] rows handed out, ctrl[2] draws listed, ctrl[3] slice slots
  // taken, ctrl[4] sampling requests decided.  Slot h is slice h % S_sl of
  // the (h / S_sl)-th listed draw.
  __device__ unsigned long long load_lc() const {
    return ld_relaxed_u64(reinterpret_cast<const unsigned long long*>(p.ctrl + 2));
  }
  __device__ bool decided() const { return ld_acquire(&p.ctrl[4]) >= C.nsamp; }
  __device__ int slot_unit(int h) const {
    const int e = h / G.S_sl, s = h - e * G.S_sl;
    int v = 0;  // the draw is listed; its publisher may still be storing the entry
    for (uint32_t it = 0; it < kSpinLimit; ++it) {
      v = *reinterpret_cast<const volatile int*>(&p.res_list[e]);
      if (v != 0) {
        v = ld_acquire(&p.res_list[e]);
        break;
      }
      __nanosleep(32);
    }
    if (v == 0) {
      raise_error(p.err, SD_DEV_ERR_TIMEOUT);
      return kWait;
    }
    last_ia = v - 1;  // published beside the unit
    return kResBase | (e << 8) | s;
  }
  // Next unit for this CTA: a listed slice first, else a row; kEnd once
  // nothing is left anywhere; kWait when a draw may still be listed.
  // `depth` is the number of units published behind the one being folded
  // (-1: none in flight).  Once the rows have run out, a CTA takes a slice
  // only when it has no unit in flight, so that a late draw's slices go to
  // idle CTAs and start at once instead of waiting behind a row.
  __device__ int schedule(int depth) {
    const unsigned long long lc = load_lc();
    const int avail = static_cast<int>(lc & 0xFFFFFFFFull) * G.S_sl;
    const bool deep = rows_done && depth >= 0;
    if (!deep && held < 0 && static_cast<int>(lc >> 32) < avail) held = atomicAdd(&p.ctrl[3], 1);
    if (held >= 0 && held < avail) {
      const int h = held;
      held = -1;
      return slot_unit(h);
    }
    if (!rows_done) {
      const int u = stash;
      if (u < C.U_rows) {
        stash = dealt ? C.U_rows : atomicAdd(&p.ctrl[0], 1);  // used by the next schedule
        return u;
      }
      rows_done = true;
      if (depth >= 0) return kWait;  // as above: slices only with nothing in flight
    }
    if (deep || !decided()) return kWait;
    const unsigned long long f = load_lc();  // the final list
    const int fin = static_cast<int>(f & 0xFFFFFFFFull) * G.S_sl;
    if (held < 0) {
      if (static_cast<int>(f >> 32) >= fin) return kEnd;
      held = atomicAdd(&p.ctrl[3], 1);
    }
    const int h = held;
    held = -1;
    return h < fin ? slot_unit(h) : kEnd;  // a slot past the final list is void
  }

  // ---- warp-wide draw helpers ---------------------------------------------
  // The searches below share their per-lane values through the warp's
  // scratch in shared memory (one barrier per exchange) rather than through
  // chains of shuffles: every lane reads all 32 values and computes the sums
  // and the search result itself.
  __device__ unsigned long long* scratch() const { return s_walk + 32 * kWalk; }

  // Sum of the 32 values in sc[0..32) (read by every lane).
  __device__ static unsigned long long sum32(const unsigned long long* sc) {
    unsigned long long t = 0;
#pragma unroll 8
    for (int l = 0; l < 32; ++l) t += sc[l];
    return t;
  }
  // The first l whose running sum of sc[0..l] exceeds th (th < the total), and
  // the running sum before it.
  __device__ static int first_past(const unsigned long long* sc, unsigned long long th,
                                   unsigned long long& before) {
    int ln = 31;
    unsigned long long run = 0;
    before = 0;
    bool found = false;
#pragma unroll 8
    for (int l = 0; l < 32; ++l) {
      const unsigned long long nx = run + sc[l];
      if (!found && nx > th) {
        ln = l;
        before = run;
        found = true;
      }
      run = nx;
    }
    return ln;
  }

  // The first of n weights (vocabulary order) whose running sum exceeds the
  // threshold: floor(u * S) when use_u, else th_in clamped below S.  Each
  // lane sums a contiguous block exactly in 64 bits.  Returns false when
  // S = 0; else sets c (the index) and th (the threshold within it).
  // Lane l holds the weights of entries [l * cpl, (l + 1) * cpl) in wv.
  __device__ bool crossing(int n, const unsigned long long (&wv)[kCpl], bool use_u, float ufin,
                           unsigned long long th_in, int& c_out, unsigned long long& th_out) const {
    const int cpl = (n + 31) / 32;
    const int b0 = min(n, lane * cpl), b1 = min(n, b0 + cpl);
    unsigned long long ls = 0;
#pragma unroll
    for (int q = 0; q < kCpl; ++q) ls += wv[q];
    unsigned long long* sc = scratch();
    sc[lane] = ls;
    __syncwarp();
    const unsigned long long S = sum32(sc);
    if (S == 0) {
      __syncwarp();  // the scratch is read before it is reused
      return false;
    }
    const unsigned long long thr =
        use_u ? __umul64hi(__float2ull_rn(ufin * kTwo64), S) : (th_in < S ? th_in : S - 1);
    unsigned long long before;
    const int ln = first_past(sc, thr, before);
    __syncwarp();  // every lane has read the lane sums
    if (lane == ln) {
      unsigned long long run = before;
      int c = b1 - 1;
      for (int q = 0; q < kCpl; ++q) {
        if (q < cpl && b0 + q < b1) {
          if (run + wv[q] > thr) {
            c = b0 + q;
            break;
          }
          run += wv[q];
        }
      }
      sc[32] = static_cast<unsigned long long>(c);
      sc[33] = thr - run;
    }
    __syncwarp();
    c_out = static_cast<int>(sc[32]);
    th_out = sc[33];
    __syncwarp();  // read before the scratch is reused
    return true;
  }

  // The element of units [ub, ue) where the running weight passes th:
  // usum(u) is unit u's weight, elem(u, wi) its elements' weights.  Each lane
  // takes a block of at most kWalk units: it first prefetches the block into
  // L1, then sums each unit, keeping the sums in shared memory, so the lane
  // holding the crossing recomputes one unit only.  Longer ranges go in
  // rounds.  When the threshold lies past the units or past the crossing
  // unit's elements (their fixed-point values need not add up to the unit's
  // exactly), the last positive weight is taken.
  template <typename UF, typename EF, typename FF>
  __device__ int walk(UF usum, EF elem, FF pref, int ub, int ue, unsigned long long th) const {
    unsigned long long* us = s_walk + lane * kWalk;
    // the element of unit u where the running weight from 0 passes r, else its last positive one
    auto pick_in = [&](int u, unsigned long long r) {
      unsigned long long wi[VE];
      elem(u, wi);
      unsigned long long acc = 0;
      int last = u * VE + VE - 1, hit = -1;
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        if (wi[e] > 0) last = u * VE + e;
        if (hit < 0 && acc + wi[e] > r) hit = u * VE + e;
        acc += wi[e];
      }
      return hit >= 0 ? hit : last;
    };
    int lastu = -1;
    for (int rb = ub; rb < ue; rb += 32 * kWalk) {
      const int re = min(ue, rb + 32 * kWalk);
      const int upl = (re - rb + 31) / 32;
      const int b0 = min(re, rb + lane * upl), b1 = min(re, b0 + upl);
      for (int u = b0; u < b1; ++u) pref(u);
      unsigned long long sv = 0;
#pragma unroll 1
      for (int u = b0; u < b1; ++u) {
        const unsigned long long su = usum(u);
        if (su > 0) lastu = u;
        us[u - b0] = su;
        sv += su;
      }
      unsigned long long* sc = scratch();
      sc[lane] = sv;
      __syncwarp();
      const unsigned long long tot = sum32(sc);
      if (th < tot) {
        unsigned long long acc;
        const int ln = first_past(sc, th, acc);
        __syncwarp();  // every lane has read the block sums
        if (lane == ln) {
          int u = b1 - 1;
          for (int v = b0; v < b1; ++v) {
            if (acc + us[v - b0] > th) {
              u = v;
              break;
            }
            acc += us[v - b0];
          }
          sc[32] = static_cast<unsigned long long>(pick_in(u, th - acc));
        }
        __syncwarp();
        const int pk = static_cast<int>(sc[32]);
        __syncwarp();  // read before the scratch is reused
        return pk;
      }
      th -= tot;
      __syncwarp();  // read before the next round rewrites the scratch
    }
    unsigned long long* sc = scratch();
    sc[lane] = static_cast<unsigned long long>(lastu + 1);
    __syncwarp();
    unsigned long long mx = 0;
#pragma unroll 8
    for (int l = 0; l < 32; ++l) mx = sc[l] > mx ? sc[l] : mx;
    __syncwarp();  // read before the scratch is reused
    const int lu = static_cast<int>(mx) - 1;
    if (lu < 0) return ub * VE;
    return pick_in(lu, ~0ull);  // every lane: the same unit, the same answer
  }

  // Draw from p of target row c0 + a (its per-chunk statistics give the
  // chunk weights; only the crossing chunk is read again).
  // This lane's block of the chunk statistics of target row trow (all
  // requested before any is used).
  __device__ void load_stats(size_t trow, float2 (&st)[kCpl]) const {
    const float2* stc = p.st_c + trow * kStatStride;
    const int nst = NS * G.spw;
    const int cpl = (nst + 31) / 32, b0 = min(nst, lane * cpl), b1 = min(nst, b0 + cpl);
#pragma unroll
    for (int q = 0; q < kCpl; ++q) {
      int ub = 0, ue = 0;
      if (q < cpl && b0 + q < b1) stat_units(G, b0 + q, ub, ue);
      st[q] = ub < ue ? __ldcg(stc + b0 + q) : make_float2(-INFINITY, 0.0f);
    }
  }

  __device__ int bonus(size_t trow, const DrawRows<Raw>& w, float ufin) const {
    float2 st[kCpl];
    load_stats(trow, st);
    return bonus(st, w, ufin);
  }

  // Draw from p with the row's chunk statistics already in hand.
  __device__ int bonus(const float2 (&st)[kCpl], const DrawRows<Raw>& w, float ufin) const {
    const int nst = NS * G.spw;
    unsigned long long wv[kCpl];
#pragma unroll
    for (int q = 0; q < kCpl; ++q)
      wv[q] = (st[q].x != -INFINITY && st[q].y > 0.0f)
                  ? __float2ull_rn(__fmul_rn(st[q].y * exp2_ftz((st[q].x - w.Mt) * w.s2), kTwo40))
                  : 0ull;
    int c;
    unsigned long long th;
    if (!crossing(nst, wv, true, ufin, 0ull, c, th)) {
      if (lane == 0) raise_error(p.err, SD_DEV_ERR_LOGITS);
      return 0;
    }
    int ub, ue;
    stat_units(G, c, ub, ue);
    DrawRows<Raw> ws = w;
    const bool staged = stage(ws, false, ub, ue);
    return walk([&](int u) { return unit_p<T, VEC>(ws, u); },
                [&](int u, unsigned long long (&wi)[VE]) { elem_p<T, VEC>(ws, u, wi); },
                [&](int u) {
                  if (!staged) prefetch_l1(ws.rt + u);
                },
                ub, ue, th);
  }

  // ---- per-request work (warp) --------------------------------------------
  // Accept tests of request i (lane j tests slot j), then its final token:
  // the argmax (greedy), a bonus draw from p (whole prefix accepted), or --
  // at a rejection -- a residual draw, listed for the slices.
  __device__ void tail(int i) const {
    const int c0 = C.cu[i];
    const int n = C.cu[i + 1] - c0 - 1;
    const int d0 = c0 - i;
    const float tau = C.tau[i];
    const bool greedy = !(tau > 0.0f);
    float s2h = 0.0f, s2l = 0.0f;
    if (!greedy) {
      s2h = kLog2eHi / tau;
      s2l = (fmaf(-s2h, tau, kLog2eHi) + kLog2eLo) / tau;
    }
    const float* urow = p.uniforms + static_cast<size_t>(i) * (p.k_max + 1);
    // lane j holds the statistics of slot j's rows (lane n: the bonus row)
    float4 ts_l = make_float4(0.0f, 1.0f, 0.0f, 0.0f), ds_l = make_float4(0.0f, 1.0f, 0.0f, 0.0f);
    if (lane <= n) ts_l = __ldcg(reinterpret_cast<const float4*>(p.st_t + c0 + lane));
    if (lane < n && !greedy) ds_l = __ldcg(reinterpret_cast<const float4*>(p.st_d + d0 + lane));
    // Every lane runs the accept test (lanes past the slots repeat the last
    // slot and discard the result), so the warp does not split here.
    bool acc = true;
    if (n > 0) {
      const bool slot = lane < n;
      const int j = slot ? lane : n - 1;
      const int x = p.draft_ids[d0 + j];
      const bool x_ok = x >= 0 && x < p.V;
      if (slot && !x_ok) raise_error(p.err, SD_DEV_ERR_DRAFT_ID);
      const float4 ts = ts_l;
      if (greedy) {
        const int amax = __float_as_int(ts.w);
        if (slot && amax < 0) raise_error(p.err, SD_DEV_ERR_LOGITS);
        acc = !slot || (x_ok && amax >= 0 && x == amax);
      } else {
        const float4 ds = ds_l;
        const bool ok = isfinite(ts.x) && isfinite(ts.y) && ts.y > 0.0f && isfinite(ds.x) &&
                        isfinite(ds.y) && ds.y > 0.0f;
        float px = 0.0f, qx = 0.0f;
        if (ok && x_ok) {
          float h, l;
          two_diff(ts.z, ts.x, h, l);
          px = exp2_df(h, l, s2h, s2l) / ts.y;
          two_diff(ds.z, ds.x, h, l);
          qx = exp2_df(h, l, s2h, s2l) / ds.y;
        }
        const float u = urow[j];
        if (slot && !ok) raise_error(p.err, SD_DEV_ERR_LOGITS);
        if (slot && !(u >= 0.0f && u < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
        acc = !slot || (ok && x_ok && (u * qx) <= px);
        if (slot && p.probs_out) {
          p.probs_out[2 * static_cast<size_t>(d0 + j)] = px;
          p.probs_out[2 * static_cast<size_t>(d0 + j) + 1] = qx;
        }
      }
    }
    const unsigned rej = __ballot_sync(kFull, !acc);
    const int a = rej ? __ffs(rej) - 1 : n;
    float4 ts;
    ts.x = __shfl_sync(kFull, ts_l.x, a);
    ts.y = __shfl_sync(kFull, ts_l.y, a);
    ts.z = __shfl_sync(kFull, ts_l.z, a);
    ts.w = __shfl_sync(kFull, ts_l.w, a);
    int pick = 0;
    bool residual = false;
    if (greedy) {
      const int amax = __float_as_int(ts.w);
      if (amax < 0 && lane == 0) raise_error(p.err, SD_DEV_ERR_LOGITS);
      pick = amax >= 0 ? amax : 0;
    } else {
      const bool reject = a < n;
      float4 ds;
      ds.x = __shfl_sync(kFull, ds_l.x, a);
      ds.y = __shfl_sync(kFull, ds_l.y, a);
      ds.z = __shfl_sync(kFull, ds_l.z, a);
      ds.w = __shfl_sync(kFull, ds_l.w, a);
      const bool ok = isfinite(ts.x) && isfinite(ts.y) && ts.y > 0.0f &&
                      (!reject || (isfinite(ds.x) && isfinite(ds.y) && ds.y > 0.0f));
      const float ufin = urow[p.k_max];
      if (lane == 0 && !(ufin >= 0.0f && ufin < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
      if (!ok) {
        if (lane == 0) raise_error(p.err, SD_DEV_ERR_LOGITS);
      } else if (reject) {
        residual = true;
      } else {
        // every slot accepted: a bonus draw from the next row (its chunk
        // statistics are read only here; most sampling requests reject)
        pick = bonus(static_cast<size_t>(c0 + n), make_rows<T, VEC>(p, C.cu, i, a, tau, ts, ds, false),
                     ufin);
      }
    }
    // outputs: the accepted draft tokens, the final token (a residual one is
    // written by its draw's last slice), -1 after it
    int* o = p.out_tokens + static_cast<size_t>(i) * (p.k_max + 1);
    if (lane <= p.k_max)
      o[lane] = lane < a ? p.draft_ids[d0 + lane] : (lane == a ? (residual ? -1 : pick) : -1);
    __syncwarp();
    if (lane == 0) {
      p.accepted_len[i] = a;
      p.req_cnt[i] = 0;  // leave the workspace ready for the next call
      if (!greedy) {
        if (residual) {
          const int pos = atomicAdd(&p.ctrl[2], 1);
          st_release(&p.res_list[pos], 1 + ((i << 4) | a));  // publishes the outputs too
        }
        // one more sampling request decided; releases the warp's outputs (the
        // lanes' writes are ordered before it by the warp barrier above)
        red_add_release(&p.ctrl[4], 1);
      }
    }
    __syncwarp();
  }

  // Last slice of listed draw e folded: the residual's chunk sums are
  // complete; find the crossing chunk and walk it.
  __device__ void finish(int e, int i, int a, const float4& ts, const float4& ds, float ufin) const {
    const int c0 = C.cu[i];
    unsigned long long* rs = p.rs + static_cast<size_t>(e) * kStatStride;
    const int nst = NS * G.spw;
    const int cpl = (nst + 31) / 32, b0 = min(nst, lane * cpl), b1 = min(nst, b0 + cpl);
    unsigned long long wv[kCpl];
#pragma unroll
    for (int q = 0; q < kCpl; ++q) {
      int ub = 0, ue = 0;
      if (q < cpl && b0 + q < b1) stat_units(G, b0 + q, ub, ue);
      wv[q] = ub < ue ? __ldcg(rs + b0 + q) : 0ull;
    }
    const DrawRows<Raw> w = make_rows<T, VEC>(p, C.cu, i, a, C.tau[i], ts, ds, true);
    int c;
    unsigned long long th;
    int pick;
    if (crossing(nst, wv, true, ufin, 0ull, c, th)) {
      int ub, ue;
      stat_units(G, c, ub, ue);
      DrawRows<Raw> ws = w;
      const bool staged = stage(ws, true, ub, ue);
      pick = walk([&](int u) { return unit_res<T, VEC>(ws, u); },
                  [&](int u, unsigned long long (&wi)[VE]) { elem_res<T, VEC>(ws, u, wi); },
                  [&](int u) {
                    if (!staged) {
                      prefetch_l1(ws.rt + u);
                      prefetch_l1(ws.rd + u);
                    }
                  },
                  ub, ue, th);
    } else {
      pick = bonus(static_cast<size_t>(c0 + a), w, ufin);  // no residual mass in fp32: draw from p
    }
    for (int q = lane; q < nst; q += 32) rs[q] = 0;  // zero for the next call
    __syncwarp();
    if (lane == 0) {
      p.out_tokens[static_cast<size_t>(i) * (p.k_max + 1) + a] = pick;
      p.slice_cnt[e] = 0;
      p.res_list[e] = 0;
    }
    __syncwarp();
  }

  // Unit u at position k is done in every streaming warp: fold it.
  __device__ void fold(int k, int u) const {
    const int sl = k % kDepth;
    if (u < C.U_rows) {
      const Unit t = locate(C, p.bs, u);
      float4 stat;
      if (t.greedy) {
        const unsigned long long kk = warp_max_u64(lane < NS ? red_k[sl][lane] : 0ull);
        const int nn = __any_sync(kFull, lane < NS ? red_n[sl][lane] : 0);
        const float bv = from_ordered(static_cast<uint32_t>(kk >> 32));
        const bool rowbad = nn || kk == 0ull || !isfinite(bv);
        const int amax = rowbad ? -1 : static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(kk));
        stat = make_float4(bv, 0.0f, s_lx[sl], __int_as_float(amax));
      } else {
        const float s2 = kLog2e / C.tau[t.i];
        const float mw = lane < NS ? red_m[sl][lane] : -INFINITY;
        const float M = warp_max(mw);
        const float zr = (lane < NS && mw != -INFINITY && M != -INFINITY)
                             ? red_z[sl][lane] * exp2_ftz((mw - M) * s2)
                             : 0.0f;
        stat = make_float4(M, warp_sum(zr), s_lx[sl], __int_as_float(0));
      }
      if (!t.greedy && !t.draft) {  // the chunk statistics of a sampling request's target row
        float2* stc = p.st_c + t.row * kStatStride;
        for (int c = lane; c < NS * G.spw; c += 32) {
          int ub, ue;
          stat_units(G, c, ub, ue);
          const unsigned long long v = s_stat[sl][c];
          if (ub < ue)
            __stcg(stc + c, make_float2(__uint_as_float(static_cast<uint32_t>(v)),
                                        __uint_as_float(static_cast<uint32_t>(v >> 32))));
        }
      }
      __syncwarp();  // every lane's writes of the row before lane 0's count
      int old = 0;
      if (lane == 0) {
        __stcg(reinterpret_cast<float4*>(t.draft ? p.st_d + t.row : p.st_t + t.row), stat);
        // releases this row's statistics, acquires those of the rows counted before
        old = atom_add_acq_rel(&p.req_cnt[t.i], 1);
      }
      old = __shfl_sync(kFull, old, 0);
      if (old == (t.n + 1) + (t.greedy ? 0 : t.n) - 1) push_job(t.i);  // the request's last row: its tail
    } else if (is_slice(u)) {
      const int e = (u >> 8) & 0xFFF;
      unsigned long long* rs = p.rs + static_cast<size_t>(e) * kStatStride;
      for (int c = lane; c < NS * G.spw; c += 32) {
        const unsigned long long v = s_stat[sl][c];
        if (v != 0) atomicAdd(rs + c, v);
      }
      __syncwarp();  // every lane's sums before lane 0's count
      int old = 0;
      // releases this slice's sums, acquires those of the slices counted before
      if (lane == 0) old = atom_add_acq_rel(&p.slice_cnt[e], 1);
      old = __shfl_sync(kFull, old, 0);
      if (old == G.S_sl - 1) push_job(kFinishJob | (e << 16) | C.qx[sl]);  // the draw's last slice: its finish
    }
  }

  // ---- jobs: tails and draw finishes, run by the draw warps ---------------
  // The scheduling warp appends; each draw warp takes the next job.
  static constexpr int kFinishJob = 1 << 30;
  static constexpr int kStopJob = -1;
  __device__ void push_job(int code) const {
    if (lane == 0) {
      const int t = *jtail;
      uint32_t it = 0;
      for (; it < kSpinLimit && t - ld_volatile_cta(jdone) >= kJobs; ++it) __nanosleep(64);
      if (it >= kSpinLimit) raise_error(p.err, SD_DEV_ERR_TIMEOUT);  // the ring is full
      jobs[t % kJobs] = code;
      st_release_cta(jtail, t + 1);
    }
    __syncwarp();
  }
  __device__ void run_draw() {
    for (;;) {
      int code = kStopJob;
      if (lane == 0) {
        const int j = atomicAdd(jhead, 1);
        bool ok = false;
        for (uint32_t it = 0; it < kSpinLimit; ++it) {
          if (ld_volatile_cta(jtail) > j) {
            ok = ld_acquire_cta(jtail) > j;
            break;
          }
          __nanosleep(64);
        }
        if (ok) {
          code = jobs[j % kJobs];
          atomicAdd(jdone, 1);
        } else {
          raise_error(p.err, SD_DEV_ERR_TIMEOUT);
        }
      }
      code = __shfl_sync(kFull, code, 0);
      if (code == kStopJob) break;
      // lane 0 acquired the job, which the scheduling warp released after its
      // counter had acquired the statistics and sums; the warp barrier orders
      // the other lanes' reads after that acquire
      __syncwarp();
      if (code & kFinishJob) {
        const int e = (code >> 16) & 0xFFF, i = (code >> 4) & 0xFFF, a = code & 15;
        const int c0 = C.cu[i];
        const float4 ts = __ldcg(reinterpret_cast<const float4*>(p.st_t + c0 + a));
        const float4 ds = __ldcg(reinterpret_cast<const float4*>(p.st_d + c0 - i + a));
        const float ufin = p.uniforms[static_cast<size_t>(i) * (p.k_max + 1) + p.k_max];
        finish(e, i, a, ts, ds, ufin);
      } else {
        tail(code);
      }
    }
  }

  __device__ void run_sched(int k_pub) {
    int k_done = 0;
    bool end_pub = false;
    uint32_t idle = 0;
    for (;;) {
      bool progress = false;
      if (!end_pub && k_pub < k_done + kWindow - 1) {
        int e = kWait;
        if (lane == 0) e = schedule(k_pub - k_done);
        e = __shfl_sync(kFull, e, 0);
        if (e != kWait) {
          if (lane == 0) {
            C.q[(k_pub + 1) % kDepth] = e;
            if (is_slice(e)) C.qx[(k_pub + 1) % kDepth] = last_ia;
            st_release_cta(C.pub, k_pub + 1);
          }
          ++k_pub;
          end_pub = e == kEnd;
          progress = true;
        }
      }
      if (k_done <= k_pub) {
        const int u = C.q[k_done % kDepth];
        if (u == kEnd) break;
        // one lane tests the barrier and the warp follows its verdict, so
        // every lane takes the same path through the fold's shuffles
        bool done = lane == 0 && mbar_try_wait(&pbar[k_done % kDepth], (k_done / kDepth) & 1);
        done = __shfl_sync(kFull, done, 0);
        if (done) {
          __syncwarp();  // lane 0's acquire covers the whole warp
          fold(k_done, u);
          ++k_done;
          progress = true;
        }
      }
      if (progress) {
        idle = 0;
      } else if (++idle > kSpinLimit) {
        if (lane == 0) raise_error(p.err, SD_DEV_ERR_TIMEOUT);
        if (lane == 0 && !end_pub) {  // let the streaming warps finish
          C.q[(k_pub + 1) % kDepth] = kEnd;
          st_release_cta(C.pub, k_pub + 1);
        }
        break;
      } else {
        __nanosleep(64);
      }
    }
    push_job(kStopJob);  // one per draw warp, after every job of the call
    push_job(kStopJob);
  }
};

// ---------------------------------------------------------------------------
// The kernel: NT / 32 - 3 streaming warps, a scheduling warp and two draw
// warps per CTA, one CTA per SM, persistent over the whole work list.
template <typename T, int NT, bool VEC>
__global__ void __launch_bounds__(NT, 1) verify_kernel(const __grid_constant__ VerifyParams p) {
  using Raw = typename VT<T, VEC>::Raw;
  constexpr int VE = VT<T, VEC>::VE;
  constexpr int NW = NT / 32;
  constexpr int NS = NW - 3;  // streaming warps; warp NS schedules, NS + 1 and NS + 2 draw
  static_assert(NS <= 32, "one lane of the control warp per streaming warp");
  constexpr size_t kRing = VEC ? static_cast<size_t>(NS) * kSlots * kSlotBytes : 0;
  constexpr int kBars = VEC ? NS * kSlots : 0;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;                                   // [NS][kSlots][kSlotBytes]
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + kRing);   // [NS][kSlots]
  int* cu_s = reinterpret_cast<int*>(mbar + kBars);             // [bs+1]
  float* tau_s = reinterpret_cast<float*>(cu_s + p.bs + 1);     // [bs]
  int* order = reinterpret_cast<int*>(tau_s + p.bs);            // [bs] request order
  int* ustart = order + p.bs;                                   // [bs+1] first unit of order[k]

  __shared__ uint64_t pbar[kDepth];  // position k done by every streaming warp
  __shared__ int s_q[kDepth];        // the unit of position k at s_q[k % kDepth]
  __shared__ int s_qx[kDepth];       // beside a slice unit: its draw's request and slot
  __shared__ int s_pub;              // positions 0..s_pub are published
  __shared__ float red_m[kDepth][NS], red_z[kDepth][NS];
  __shared__ unsigned long long red_k[kDepth][NS];
  __shared__ int red_n[kDepth][NS];
  __shared__ float s_lx[kDepth];
  __shared__ unsigned long long s_stat[kDepth][kStatStride];
  __shared__ int red_i[NW];
  __shared__ int s_count, s_nsamp;
  __shared__ unsigned long long s_walk[2][32 * Control<T, VEC, NS>::kWalk + Control<T, VEC, NS>::kScratch];
  __shared__ int s_jobs[Control<T, VEC, NS>::kJobs];
  __shared__ int s_jtail, s_jhead, s_jdone;
  __shared__ __align__(128) unsigned char s_chunk[2][2 * kSlotBytes];  // draw warps' staging
  __shared__ uint64_t s_cbar[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = (p.V + VE - 1) / VE;  // VE divides V on the vector path

  // ---- per-call checks of the compaction (identical verdict in every CTA)
  for (int i = tid; i <= p.bs; i += NT) cu_s[i] = p.cu[i];
  __syncthreads();
  int bad = (tid == 0 && cu_s[0] != 0) ? 1 : 0;
  for (int i = tid; i < p.bs; i += NT) {
    const int d = cu_s[i + 1] - cu_s[i];
    if (d < 1 || d > p.k_max + 1) bad = 1;
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0) {
      if (tid == 0) raise_error(p.err, SD_DEV_ERR_CU_SEQLENS);
      for (int i = tid; i < p.bs; i += NT) {
        p.accepted_len[i] = 0;
        for (int j = 0; j <= p.k_max; ++j)
          p.out_tokens[static_cast<size_t>(i) * (p.k_max + 1) + j] = -1;
      }
    }
    return;  // nothing read, no counter touched
  }
  int badt = 0;
  for (int i = tid; i < p.bs; i += NT) {
    float t = p.temps[i];
    if (!(t >= 0.0f) || !isfinite(t)) { badt |= SD_DEV_ERR_TEMP; t = 0.0f; }
    if (t > 0.0f && p.draft == nullptr) { badt |= SD_DEV_ERR_LOGITS; t = 0.0f; }
    tau_s[i] = t;
  }
  if (badt && blockIdx.x == 0) raise_error(p.err, badt);
  __syncthreads();

  // The small per-request inputs that only the final draws read (uniforms,
  // draft ids) are brought into L2 and kept there, so that those draws do
  // not wait behind the row traffic queued at the memory controllers.  Every
  // address prefetched lies inside its array.
  {
    const size_t bu = static_cast<size_t>(p.bs) * (p.k_max + 1) * sizeof(float);
    const size_t bd = p.draft_ids ? static_cast<size_t>(cu_s[p.bs] - p.bs) * sizeof(int) : 0;
    const size_t lu = (bu + 127) / 128, ld = (bd + 127) / 128;
    for (size_t l = static_cast<size_t>(blockIdx.x) * NT + tid; l < lu + ld;
         l += static_cast<size_t>(gridDim.x) * NT) {
      const char* a = l < lu ? reinterpret_cast<const char*>(p.uniforms) + l * 128
                             : reinterpret_cast<const char*>(p.draft_ids) + (l - lu) * 128;
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(a));
    }
  }

  // Exclusive prefix of one value per thread (thread order); *total = sum.
  auto block_scan = [&](int v, int* total) {
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) red_i[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      const int w = lane < NW ? red_i[lane] : 0;
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, wi, o);
        if (lane >= o) wi += t;
      }
      if (lane < NW) red_i[lane] = wi - w;
      if (lane == 31) s_count = wi;
    }
    __syncthreads();
    const int r = red_i[warp] + inc - v;
    *total = s_count;
    __syncthreads();
    return r;
  };

  // ---- work list: every request's n_i + 1 target rows, then its n_i draft
  // rows when tau > 0; sampling requests first (their final draws then
  // overlap the greedy requests' rows), each group in index order.
  {
    const int chunk = (p.bs + NT - 1) / NT;
    const int beg = min(p.bs, tid * chunk), end = min(p.bs, beg + chunk);
    int npos = 0;
    for (int i = beg; i < end; ++i) npos += tau_s[i] > 0.0f;
    int n_samp;
    int pos_s = block_scan(npos, &n_samp);
    if (tid == 0) s_nsamp = n_samp;
    int pos_g = n_samp + (beg - pos_s);
    for (int i = beg; i < end; ++i) {
      if (tau_s[i] > 0.0f) order[pos_s++] = i;
      else order[pos_g++] = i;
    }
    __syncthreads();
    int units = 0;
    for (int k = beg; k < end; ++k) {
      const int i = order[k];
      const int n = cu_s[i + 1] - cu_s[i] - 1;
      units += (n + 1) + (tau_s[i] > 0.0f ? n : 0);
    }
    int total;
    int run = block_scan(units, &total);
    for (int k = beg; k < end; ++k) {
      ustart[k] = run;
      const int i = order[k];
      const int n = cu_s[i + 1] - cu_s[i] - 1;
      run += (n + 1) + (tau_s[i] > 0.0f ? n : 0);
    }
    if (tid == 0) ustart[p.bs] = total;
  }
  if (tid == 0) {
    s_jtail = 0;
    s_jhead = 0;
    s_jdone = 0;
    for (int b = 0; b < kBars; ++b) mbar_init(&mbar[b], 1);
    for (int b = 0; b < kDepth; ++b) mbar_init(&pbar[b], NS);
    mbar_init(&s_cbar[0], 1);
    mbar_init(&s_cbar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  const Geom G = make_geom(nvec, VEC, NS);
  const Cta C{cu_s, tau_s, order, ustart, s_q, s_qx, &s_pub, s_nsamp, ustart[p.bs]};
  // The first kWindow positions: rows (no draw is listed yet); the row
  // after them is the control warp's first stash.  Each CTA claims these
  // kWindow + 1 rows at once.  When that covers every row of the call, the
  // rows are dealt position-major instead (CTA b's q-th is unit
  // q * gridDim.x + b): consecutive claims would give a request's rows to one
  // CTA, one after another, and every request would finish last.
  int k_pub = -1;
  int stash = 0;
  bool dealt = false;
  if (warp == NS && lane == 0) {
    const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
    dealt = C.U_rows <= (kWindow + 1) * G;
    const int u0 = dealt ? 0 : atomicAdd(&p.ctrl[0], kWindow + 1);
    for (int q = 0; q < kWindow; ++q) {
      const int u = dealt ? q * G + b : u0 + q;
      if (u >= C.U_rows) break;
      s_q[q] = u;
      k_pub = q;
    }
    stash = dealt ? kWindow * G + b : u0 + kWindow;
    s_pub = k_pub;
  }
  __syncthreads();

  if (warp < NS) {
    Streamer<T, VEC, NS> S(p, C, G, warp, lane, ring, mbar);
    S.run(pbar, red_m, red_z, red_k, red_n, s_lx, s_stat);
  } else {
    Control<T, VEC, NS> K(p, C, G, lane, pbar, red_m, red_z, red_k, red_n, s_lx,
                          s_walk[warp == NS ? 0 : warp - NS - 1], s_jobs, &s_jtail, &s_jhead,
                          &s_jdone, s_stat, s_chunk[warp == NS ? 0 : warp - NS - 1],
                          &s_cbar[warp == NS ? 0 : warp - NS - 1]);
    if (warp == NS) {
      K.stash = stash;
      K.dealt = dealt;
      K.run_sched(__shfl_sync(kFull, k_pub, 0));
    } else {
      K.run_draw();
    }
  }
  (void)sizeof(Raw);

  // The last CTA out resets the work counters for the next call.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&p.ctrl[1], 1) == static_cast<int>(gridDim.x) - 1) {
      p.ctrl[0] = 0;
      p.ctrl[1] = 0;
      p.ctrl[2] = 0;
      p.ctrl[3] = 0;
      p.ctrl[4] = 0;
      __threadfence();
    }
  }
}

template <typename T, int NT, bool VEC>
void* kfn() {
  return reinterpret_cast<void*>(&verify_kernel<T, NT, VEC>);
}

// All instantiations: (fp32, bf16) x (vector, scalar) x (256, 512 threads).
void* const* kernel_table() {
  static void* const t[8] = {kfn<float, 256, true>(),    kfn<float, 256, false>(),
                             kfn<uint16_t, 256, true>(), kfn<uint16_t, 256, false>(),
                             kfn<float, 512, true>(),    kfn<float, 512, false>(),
                             kfn<uint16_t, 512, true>(), kfn<uint16_t, 512, false>()};
  return t;
}

void* pick_kernel(int elem, bool vec, int threads) {
  const int idx = (threads == 512 ? 4 : 0) + (elem == 4 ? 0 : 2) + (vec ? 0 : 1);
  return kernel_table()[idx];
}

// Raises the kernel's dynamic shared-memory limit to the device maximum once
// per (kernel, device); later calls are lock-free reads.
cudaError_t prepare(void* fn, size_t smem) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> limit_of[8][kMaxDev];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int slot = -1;
  for (int k = 0; k < 8; ++k)
    if (fn == kernel_table()[k]) slot = k;
  if (slot < 0 || dev < 0 || dev >= kMaxDev) return cudaErrorInvalidValue;
  int lim = limit_of[slot][dev].load(std::memory_order_acquire);
  if (lim == 0) {
    std::lock_guard<std::mutex> lk(mu);
    lim = limit_of[slot][dev].load(std::memory_order_relaxed);
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
      limit_of[slot][dev].store(lim, std::memory_order_release);
    }
  }
  return smem <= static_cast<size_t>(lim) ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

size_t verify_smem_bytes(int bs, int V, int elem, bool vec, int threads) {
  (void)V;
  (void)elem;
  const int ns = threads / 32 - 3;  // streaming warps
  const size_t ring = vec ? static_cast<size_t>(ns) * kSlots * (kSlotBytes + 8) : 0;
  return ring + static_cast<size_t>(4) * (4 * static_cast<size_t>(bs) + 2) + 16;
}

cudaError_t choose_verify_shape(int V, int elem, int bs, const sd_launch_cfg* req, bool vec,
                                VerifyShape* out, bool* fits) {
  *fits = false;
  const int treq = req ? req->threads : 0;
  if (treq && treq != 256 && treq != 512) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // 512 threads (13 streaming warps, a 113 KB ring) unless the shared
  // memory does not fit (large batches), then 256 threads (5 warps, 44 KB).
  const int cands[2] = {512, 256};
  for (int ci = 0; ci < 2; ++ci) {
    const int threads = treq ? treq : cands[ci];
    if (treq && ci > 0) break;
    void* fn = pick_kernel(elem, vec, threads);
    const size_t smem = verify_smem_bytes(bs, V, elem, vec, threads);
    e = prepare(fn, 0);
    if (e != cudaSuccess) return e;
    if (prepare(fn, smem) != cudaSuccess) continue;  // does not fit
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) continue;
    const int want = (req && req->blocks_per_sm) ? req->blocks_per_sm : 2;
    per_sm = std::min(per_sm, want);
    out->threads = threads;
    out->blocks = sms * per_sm;
    if (req && req->blocks > 0) out->blocks = std::min(req->blocks, out->blocks);
    out->smem = smem;
    out->vec = vec;
    *fits = true;
    return cudaSuccess;
  }
  return cudaSuccess;
}

cudaError_t launch_verify(const VerifyParams& p, int elem, const VerifyShape& shape,
                          cudaStream_t s) {
  void* fn = pick_kernel(elem, shape.vec, shape.threads);
  cudaError_t e = prepare(fn, shape.smem);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<VerifyParams*>(&p)};
  e = cudaLaunchKernel(fn, dim3(shape.blocks), dim3(shape.threads), args, shape.smem, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace sdk
