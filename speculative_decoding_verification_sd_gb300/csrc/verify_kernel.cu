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
// Design (GB300): the work is a list of rows -- every compacted target row,
// and the draft row of every verified slot of a sampling request -- handed
// out to persistent CTAs by an atomic counter.  A CTA streams one whole row
// from HBM with 16-byte loads and reduces it to its statistics (running max
// and scaled sum at the request's temperature, or the argmax when greedy,
// plus the logit at the draft token), which it stores in the workspace.  The
// CTA that completes the last row of a request (a per-request arrival count)
// takes the request's accept decisions from those statistics and, for a
// sampling request, re-reads the one row pair that ends the accepted prefix
// -- from L2, where it was streamed moments before -- to draw the residual or
// bonus token by inverse CDF; it writes the request's outputs directly.
// Sampling requests' rows are scheduled before greedy ones so the final draws
// overlap the remaining streaming.  No CTA ever waits on another.
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

// Streaming loads: read once, keep out of L1 (L2 keeps them for the final draw).
template <typename Raw>
__device__ __forceinline__ Raw ld_stream(const Raw* p) {
  return __ldg(p);
}

template <>
__device__ __forceinline__ uint4 ld_stream<uint4>(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <>
__device__ __forceinline__ float4 ld_stream<float4>(const float4* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float from_ordered(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// One thread's values into its running (max, scaled sum) at scale s2:
// z = sum 2^((l - m) * s2) with m the running maximum.  The exponent
// arguments and the sum use packed fp32x2 arithmetic.
template <int VE>
__device__ __forceinline__ void online_add(const float (&f)[VE], float s2, float& m, float& z,
                                           float& b) {
  float vm = f[0];
#pragma unroll
  for (int e = 1; e < VE; ++e) vm = fmaxf(vm, f[e]);
  if (vm > m) {
    z = (m == -INFINITY) ? 0.0f : z * exp2_ftz((m - vm) * s2);
    m = vm;
    b = m * s2;
  }
  if (m != -INFINITY) {
    if constexpr (VE % 2 == 0) {
      const float2 s22 = make_float2(s2, s2);
      const float2 nb2 = make_float2(-b, -b);
      float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int e = 0; e < VE; e += 2) {
        const float2 t = __ffma2_rn(make_float2(f[e], f[e + 1]), s22, nb2);
        acc = __fadd2_rn(acc, make_float2(exp2_ftz(t.x), exp2_ftz(t.y)));
      }
      z += acc.x + acc.y;
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e) z += exp2_ftz(fmaf(f[e], s2, -b));
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

// Counter increment that publishes this thread's earlier writes (release)
// and sees everything published before earlier increments (acquire).
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
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
                                                 float2& z2, float& nb) {
    uint32_t mx = kNegInf2;
#pragma unroll
    for (int q = 0; q < N; ++q) mx = bmax2(mx, bmax2(bmax2(r[q].x, r[q].y), bmax2(r[q].z, r[q].w)));
    const float lm = fmaxf(bf_lo(mx), bf_hi(mx));
    if (lm > m) {
      if (m == -INFINITY) {
        z2 = make_float2(0.0f, 0.0f);
      } else {
        const float sc = exp2_ftz((m - lm) * s2);
        z2 = __fmul2_rn(z2, make_float2(sc, sc));
      }
      m = lm;
      nb = -m * s2;
    }
    if (m != -INFINITY) {
      const float2 s22 = make_float2(s2, s2), nb2 = make_float2(nb, nb);
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const uint32_t w4[4] = {r[q].x, r[q].y, r[q].z, r[q].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 t = __ffma2_rn(make_float2(bf_lo(w4[h]), bf_hi(w4[h])), s22, nb2);
          z2 = __fadd2_rn(z2, make_float2(exp2_ftz(t.x), exp2_ftz(t.y)));
        }
      }
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
                                                 float2& z2, float& nb) {
    float lm = -INFINITY;
#pragma unroll
    for (int q = 0; q < N; ++q) lm = fmaxf(fmaxf(lm, fmaxf(r[q].x, r[q].y)), fmaxf(r[q].z, r[q].w));
    if (lm > m) {
      if (m == -INFINITY) {
        z2 = make_float2(0.0f, 0.0f);
      } else {
        const float sc = exp2_ftz((m - lm) * s2);
        z2 = __fmul2_rn(z2, make_float2(sc, sc));
      }
      m = lm;
      nb = -m * s2;
    }
    if (m != -INFINITY) {
      const float2 s22 = make_float2(s2, s2), nb2 = make_float2(nb, nb);
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const float2 t0 = __ffma2_rn(make_float2(r[q].x, r[q].y), s22, nb2);
        const float2 t1 = __ffma2_rn(make_float2(r[q].z, r[q].w), s22, nb2);
        z2 = __fadd2_rn(z2, make_float2(exp2_ftz(t0.x), exp2_ftz(t0.y)));
        z2 = __fadd2_rn(z2, make_float2(exp2_ftz(t1.x), exp2_ftz(t1.y)));
      }
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

constexpr int kUnroll = 8;          // element path: loads in flight per thread
constexpr int kChunkBytes = 4096;       // vector path: one bulk copy
constexpr int kSlots = 3;               // ring slots per warp
constexpr uint32_t kSpinLimit = 1u << 22;  // polls (~100 ns apart) before a wait gives up
// Queue entries past the rows: slice s of listed residual draw e, the draw
// of request i at slot a, as kResBase | e << 18 | s << 16 | i << 4 | a
// (e, i < 4096, s < 4, a < 16), and three tokens.
constexpr int kResBase = 1 << 30;
constexpr int kNoop = INT_MAX - 2;
constexpr int kPoll = INT_MAX - 1;
constexpr int kEnd = INT_MAX;
constexpr float kLn2 = 0.693147180559945309f;
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

__device__ __forceinline__ unsigned long long warp_scan_u64(unsigned long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// 2^(d * s2) with d = l - M given as (d_hi, d_lo) and s2 = s2_hi + s2_lo: the
// exponent is formed in double-float so its rounding does not depend on |d|.
// Written with explicitly rounded intrinsics so that every call site computes
// bit-identical values (the final draw recomputes weights it summed before).
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

template <typename T, int NT, bool VEC>
__global__ void __launch_bounds__(NT, NT <= 256 ? 2 : 1) verify_kernel(const VerifyParams p) {
  using Tr = VT<T, VEC>;
  using Raw = typename Tr::Raw;
  constexpr int VE = Tr::VE;
  constexpr int NW = NT / 32;
  constexpr int CB = kChunkBytes;  // bytes per ring slot (one chunk)
  constexpr int VPC = CB / 16;     // 16-byte vectors per chunk
  constexpr int VPL = VPC / 32;    // vectors per lane per chunk
  constexpr int EPC = CB / static_cast<int>(sizeof(T));  // elements per chunk
  constexpr int BW = NW - 1;       // the warp that keeps the per-row books
  static_assert(NW <= 32, "one lane per warp in the cross-warp reductions");
  static_assert(VPL * 32 * 16 == CB, "chunk is a whole number of warp-wide vectors");
  constexpr size_t kRing = VEC ? static_cast<size_t>(NW) * kSlots * CB : 0;
  constexpr int kBars = VEC ? NW * kSlots : 0;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;                                   // [NW][kSlots][CB]
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + kRing);   // [NW][kSlots]
  int* cu_s = reinterpret_cast<int*>(mbar + kBars);             // [bs+1]
  float* tau_s = reinterpret_cast<float*>(cu_s + p.bs + 1);     // [bs]
  int* order = reinterpret_cast<int*>(tau_s + p.bs);            // [bs] request order
  int* ustart = order + p.bs;                                   // [bs+1] first unit of order[k]

  // per-warp partial row statistics, double-buffered by unit parity
  __shared__ float red_m[2][NW], red_z[2][NW];
  __shared__ unsigned long long red_k[2][NW];
  __shared__ int red_n[2][NW];
  __shared__ int red_i[NW];
  __shared__ float s_lx[2];
  __shared__ int s_q[4];        // unit queue of this CTA: the k-th unit at s_q[k & 3]
  __shared__ int s_pending[2];  // request whose last row ended unit k-1 (or -1)
  __shared__ int s_a, s_pick, s_count, s_found, s_ch, s_lastpos, s_hit, s_nsamp, s_last;
  __shared__ unsigned long long s_th;
  __shared__ unsigned long long red_u[NW];
  __shared__ unsigned long long s_R[kMaxDrawChunks];  // chunk sums of the draw in hand
  __shared__ unsigned long long s_Rr[kMaxRanges];     // range sums of a bonus draw

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V;
  const int nvec = (V + VE - 1) / VE;  // VE divides V on the vector path
  const size_t row_bytes = static_cast<size_t>(V) * sizeof(T);

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

  // ---- request order (sampling requests first, each group in index order)
  // and each request's first unit: its n_i + 1 target rows, then its n_i
  // draft rows when tau > 0.
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
  if (VEC && tid == 0) {
    for (int b = 0; b < kBars; ++b) mbar_init(&mbar[b], 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Geometry of the final draws: chunks of CUd = 32 * Ld units (Ld units per
  // lane, at most kMaxDrawChunks chunks per row).
  const int Ld = 4 * ((((nvec + 32 * kMaxDrawChunks - 1) / (32 * kMaxDrawChunks)) + 3) / 4);
  const int CUd = 32 * Ld;
  // Warp ranges of a row: warp w streams units [w * RU, (w + 1) * RU).
  const int nch_row = static_cast<int>((row_bytes + CB - 1) / CB);
  const int cpw = (nch_row + NW - 1) / NW;  // vector path: ring chunks per warp
  const int RU = VEC ? cpw * VPC : 32 * ((nvec + 32 * NW - 1) / (32 * NW));
  // The work list's rows; residual draws are added as requests are decided,
  // each as S_sl slices: slice s takes the s-th part of every warp's range
  // (m_sl ring chunks, or mu_sl elements, per warp).
  const int U_stream = ustart[p.bs];
  const int S_sl = VEC ? min(4, max(1, cpw)) : (RU >= 128 ? 4 : 1);
  const int m_sl = (cpw + S_sl - 1) / S_sl;
  const int mu_sl = 32 * ((RU + 32 * S_sl - 1) / (32 * S_sl));

  // Unit -> (request, row kind, slot, row index).
  struct Unit {
    int i, j, n, c0;
    bool draft, greedy;
    size_t row;
  };
  auto locate = [&](int u) {
    int lo = 0, hi = p.bs;  // ustart[lo] <= u < ustart[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ustart[mid] <= u) lo = mid;
      else hi = mid;
    }
    Unit t;
    t.i = order[lo];
    const int r = u - ustart[lo];
    t.c0 = cu_s[t.i];
    t.n = cu_s[t.i + 1] - t.c0 - 1;
    t.greedy = !(tau_s[t.i] > 0.0f);
    t.draft = r > t.n;
    t.j = t.draft ? r - (t.n + 1) : r;
    t.row = t.draft ? static_cast<size_t>(t.c0 - t.i + t.j) : static_cast<size_t>(t.c0 + t.j);
    return t;
  };
  auto row_base = [&](const Unit& t) {
    return reinterpret_cast<const char*>(t.draft ? p.draft : p.target) + t.row * row_bytes;
  };

  // ---- per-warp bulk-copy ring (vector path): this warp's chunks of every
  // row are the contiguous range [cb_w, ce_w).  A row position takes one
  // ring entry per chunk; a residual draw takes two (target chunk c, then
  // draft chunk c).  The fetch cursor runs up to kSlots entries ahead of
  // consumption, across positions, but stops at a position whose entry is
  // not yet a unit.
  const int cb_w = min(nch_row, warp * cpw), ce_w = min(nch_row, cb_w + cpw);
  uint32_t cseq = 0, iseq = 0;  // entries consumed / issued by this warp
  int fk = 0, fe = 0;           // fetch cursor: queue position, entry within it
  int fk_cached = -1, f_n = 0;  // position whose bases are cached, its entries
  int f_c0 = 0;                 // first chunk of the cached position
  bool f_two = false;           // two entries (target, draft) per chunk
  const char* f_base = nullptr;
  const char* f_base2 = nullptr;
  auto refill = [&](int k_limit) {
    while (iseq - cseq < static_cast<uint32_t>(kSlots) && fk <= k_limit) {
      if (fk_cached != fk) {
        const int u = s_q[fk & 3];
        if (u == kPoll || u == kEnd) break;  // not known yet / nothing follows
        f_n = 0;
        f_two = false;
        if (u < U_stream) {
          f_base = row_base(locate(u));
          f_c0 = cb_w;
          f_n = ce_w - cb_w;
        } else if (u >= kResBase && u < kNoop) {
          const int i = (u >> 4) & 0xFFF, a = u & 15, sl = (u >> 16) & 3;
          f_base = reinterpret_cast<const char*>(p.target) +
                   static_cast<size_t>(cu_s[i] + a) * row_bytes;
          f_base2 = reinterpret_cast<const char*>(p.draft) +
                    static_cast<size_t>(cu_s[i] - i + a) * row_bytes;
          f_c0 = min(ce_w, cb_w + sl * m_sl);
          f_n = 2 * (min(ce_w, f_c0 + m_sl) - f_c0);
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
      const uint32_t bytes = static_cast<uint32_t>(
          min(static_cast<size_t>(CB), row_bytes - static_cast<size_t>(c) * CB));
      if (lane == 0) {
        uint64_t* bar = &mbar[warp * kSlots + slot];
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load_nohint(ring + (warp * kSlots + slot) * CB, base + static_cast<size_t>(c) * CB,
                         bytes, bar);
      }
      ++iseq;
      ++fe;
    }
  };

  // ------------------------------------------------------------------------
  // Final draws by inverse CDF: the first element (vocabulary order) whose
  // running weight sum exceeds a threshold.  Weights are summed in 64-bit
  // fixed point (residual max(p - q, 0) <= 1 at 2^56, unnormalised
  // 2^((l - M) s2) <= 1 at 2^40), so every prefix over chunks is exact and
  // the chunk holding the crossing is found without rounding.  That chunk is
  // then recomputed with the precise weight function (double-float exponent)
  // and walked block-wide; where the two weight functions disagree by
  // rounding and the threshold passes the recomputed chunk, the chunk's last
  // positive weight stands in.
  //
  // chunk_sums: fast fixed-point sums of the chunks c0 <= c < c1 of CUd
  // units starting at unit ub (clipped at ue) -> out[c]; warp w sums chunks
  // c0 + w, c0 + w + NW, ...; each lane issues QB loads per row before using
  // any (the rows come from L2 or HBM, latency-bound otherwise).
  auto chunk_sums = [&](auto resid_tag, const Raw* rt, const Raw* rd, auto fast, float scale,
                        int ub, int ue, int c0, int c1, unsigned long long* out) {
    constexpr bool resid = decltype(resid_tag)::value;
    constexpr int QB = 2;  // loads ahead per lane and row (register budget)
    for (int c = c0 + warp; c < c1; c += NW) {
      const int cb = ub + c * CUd;
      const int ce = min(cb + CUd, ue);
      unsigned long long ls = 0;
      for (int q0 = 0; q0 < Ld; q0 += QB) {
        Raw a[QB], b[QB];
#pragma unroll
        for (int q = 0; q < QB; ++q) {
          const int u = cb + (q0 + q) * 32 + lane;
          if (u < ce) {
            a[q] = ld_stream(rt + u);
            if constexpr (resid) b[q] = ld_stream(rd + u);
          }
        }
#pragma unroll
        for (int q = 0; q < QB; ++q) {
          const int u = cb + (q0 + q) * 32 + lane;
          if (u < ce) ls += __float2ull_rn(__fmul_rn(fast(a[q], b[q]), scale));
        }
      }
      ls = warp_sum_u64(ls);
      if (lane == 0) out[c] = ls;
    }
  };

  // crossing: over the n sums R[0..n) (shared memory), with threshold
  // floor(u * S) when use_u, else th_in clamped below the total.  Sets
  // s_found (total > 0), s_ch (the chunk) and s_th (threshold within it).
  auto crossing = [&](const unsigned long long* R, int n, bool use_u, float ufin,
                      unsigned long long th_in) {
    __syncthreads();
    if (warp == 0) {
      const int epl = (n + 31) / 32;
      const int eb = min(n, lane * epl), ee = min(n, eb + epl);
      unsigned long long lsum = 0;
      for (int e = eb; e < ee; ++e) lsum += R[e];
      const unsigned long long inc = warp_scan_u64(lsum, lane);
      const unsigned long long S = __shfl_sync(kFull, inc, 31);
      if (S > 0) {
        // thr < S, so some prefix exceeds it
        const unsigned long long thr =
            use_u ? __umul64hi(__float2ull_rn(ufin * kTwo64), S) : (th_in < S ? th_in : S - 1);
        const unsigned cm = __ballot_sync(kFull, inc > thr);
        const int ln = __ffs(cm) - 1;
        const unsigned long long up = __shfl_up_sync(kFull, inc, 1);
        const unsigned long long excl = ln == 0 ? 0ull : __shfl_sync(kFull, up, ln);
        if (lane == ln) {
          unsigned long long run = excl;
          int ch = ee - 1;
          for (int e = eb; e < ee; ++e) {
            if (run + R[e] > thr) { ch = e; break; }
            run += R[e];
          }
          s_ch = ch;
          s_th = thr - run;
        }
      }
      if (lane == 0) s_found = S > 0;
    }
    __syncthreads();
  };

  // pick_in: the precise walk over units [cb, ce) for threshold th (relative
  // to cb): each thread takes a contiguous run of units, an exact 64-bit
  // block prefix finds the run that holds the crossing, and that thread
  // recomputes its run to find the element.  Sets s_pick.
  auto pick_in = [&](auto precise, int cb, int ce, unsigned long long th) {
    if (tid == 0) { s_hit = 0; s_lastpos = -1; }
    __syncthreads();
    const int upt = (ce - cb + NT - 1) / NT;
    const int tb = min(ce, cb + tid * upt), te = min(ce, tb + upt);
    unsigned long long sv = 0;
    int lastpos = -1;
    for (int u = tb; u < te; ++u) {
      unsigned long long wi[VE];
      precise(u, wi);
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        sv += wi[e];
        if (wi[e] > 0) lastpos = u * VE + e;
      }
    }
    const unsigned long long winc = warp_scan_u64(sv, lane);
    if (lane == 31) red_u[warp] = winc;
    if (lastpos >= 0) atomicMax(&s_lastpos, lastpos);
    __syncthreads();
    if (warp == 0) {
      const unsigned long long wt = lane < NW ? red_u[lane] : 0ull;
      const unsigned long long wti = warp_scan_u64(wt, lane);
      if (lane < NW) red_u[lane] = wti - wt;  // exclusive warp offsets
    }
    __syncthreads();
    const unsigned long long before = red_u[warp] + winc - sv;  // exclusive prefix
    if (sv > 0 && before <= th && th < before + sv) {
      unsigned long long acc = before;
      int pk = -1;
      for (int u = tb; u < te && pk < 0; ++u) {
        unsigned long long wi[VE];
        precise(u, wi);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          acc += wi[e];
          if (pk < 0 && acc > th) pk = u * VE + e;
        }
      }
      s_pick = pk;
      s_hit = 1;
    }
    __syncthreads();
    if (tid == 0 && !s_hit) s_pick = s_lastpos >= 0 ? s_lastpos : cb * VE;
    __syncthreads();
  };

  // Weight functions of a draw from p (target row rt, max Mt, temperature
  // scale s2 = log2(e)/tau, also as the double-float s2h + s2l) and of a
  // residual max(p - q, 0) (adds the draft row rd, max Md, and 1/Z of both).
  struct DrawRows {
    const Raw* rt;
    const Raw* rd;
    float Mt, Md, iZt, iZd, s2, s2h, s2l;
  };
  __shared__ DrawRows s_dr;  // the residual draw in hand
  auto fast_p = [](const DrawRows& w) {
    const float bt = w.Mt * w.s2, s2 = w.s2;
    return [=](const Raw& ra, const Raw&) {
      float f[VE];
      Tr::unpack(ra, f);
      float ws = 0.0f;
#pragma unroll
      for (int e = 0; e < VE; ++e) ws += exp2_ftz(fmaf(f[e], s2, -bt));
      return ws;
    };
  };
  auto precise_p = [](const DrawRows& w) {
    return [=](int u, unsigned long long (&wi)[VE]) {
      float f[VE];
      Tr::unpack(w.rt[u], f);
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        float h, l;
        two_diff(f[e], w.Mt, h, l);
        wi[e] = __float2ull_rn(__fmul_rn(exp2_df(h, l, w.s2h, w.s2l), kTwo40));
      }
    };
  };
  auto fast_res = [](const DrawRows& w) {
    const float bt = w.Mt * w.s2, bd = w.Md * w.s2, s2 = w.s2, iZt = w.iZt, iZd = w.iZd;
    return [=](const Raw& ra, const Raw& rb) {
      float f[VE], g[VE];
      Tr::unpack(ra, f);
      Tr::unpack(rb, g);
      float ws = 0.0f;
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        const float et = exp2_ftz(fmaf(f[e], s2, -bt));
        const float ed = exp2_ftz(fmaf(g[e], s2, -bd));
        ws += fmaxf(fmaf(et, iZt, -(ed * iZd)), 0.0f);
      }
      return ws;
    };
  };
  auto precise_res = [](const DrawRows& w) {
    return [=](int u, unsigned long long (&wi)[VE]) {
      float f[VE], g[VE];
      Tr::unpack(w.rt[u], f);
      Tr::unpack(w.rd[u], g);
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        float h, l;
        two_diff(f[e], w.Mt, h, l);
        const float et = exp2_df(h, l, w.s2h, w.s2l);
        two_diff(g[e], w.Md, h, l);
        const float ed = exp2_df(h, l, w.s2h, w.s2l);
        const float x = fmaxf(__fmaf_rn(et, w.iZt, -__fmul_rn(ed, w.iZd)), 0.0f);
        wi[e] = __float2ull_rn(__fmul_rn(x, kTwo56));
      }
    };
  };

  auto make_rows = [&](int i, int a, const float4& ts, const float4& ds, bool resid) {
    const float tau = tau_s[i];
    DrawRows w;
    const int c0 = cu_s[i];
    w.rt = reinterpret_cast<const Raw*>(static_cast<const T*>(p.target) +
                                        static_cast<size_t>(c0 + a) * V);
    w.rd = resid ? reinterpret_cast<const Raw*>(static_cast<const T*>(p.draft) +
                                                static_cast<size_t>(c0 - i + a) * V)
                 : w.rt;
    w.Mt = ts.x;
    w.Md = ds.x;
    w.iZt = 1.0f / ts.y;
    w.iZd = 1.0f / ds.y;
    w.s2 = kLog2e / tau;
    // s2 = log2(e) / tau as a double-float
    w.s2h = kLog2eHi / tau;
    w.s2l = (fmaf(-w.s2h, tau, kLog2eHi) + kLog2eLo) / tau;
    return w;
  };

  // Draw from p of target row trow: the row's per-range statistics give the
  // range sums, so only the crossing range is read again.
  auto bonus_draw = [&](size_t trow, const DrawRows& w, float ufin) {
    if (tid < kMaxRanges) {
      unsigned long long r = 0;
      if (tid < NW) {
        const float2 st = __ldcg(p.st_r + trow * kMaxRanges + tid);
        if (st.x != -INFINITY && st.y > 0.0f)
          r = __float2ull_rn(__fmul_rn(st.y * exp2_ftz((st.x - w.Mt) * w.s2), kTwo40));
      }
      s_Rr[tid] = r;
    }
    crossing(s_Rr, NW, true, ufin, 0ull);
    if (!s_found) {  // no mass: only a row that failed its checks gets here
      if (tid == 0) {
        raise_error(p.err, SD_DEV_ERR_LOGITS);
        s_pick = 0;
      }
      __syncthreads();
      return;
    }
    const int ub = min(nvec, s_ch * RU), ue = min(nvec, ub + RU);
    const unsigned long long th_r = s_th;
    const int nc = (ue - ub + CUd - 1) / CUd;
    chunk_sums(std::false_type{}, w.rt, w.rt, fast_p(w), kTwo40, ub, ue, 0, nc, s_R);
    crossing(s_R, nc, false, 0.0f, th_r);
    if (!s_found) {
      pick_in(precise_p(w), ub, ue, 0ull);
      return;
    }
    const int cb = ub + s_ch * CUd;
    pick_in(precise_p(w), cb, min(cb + CUd, ue), s_th);
  };


  // ------------------------------------------------------------------------
  // Tail of request i: decisions from the row statistics, then the final
  // token: the argmax (greedy), a bonus draw from p (whole prefix accepted),
  // or -- at a rejection -- a residual draw, which is listed for the slice
  // phase at the end of the work list.
  auto tail = [&](int i) {
    const int c0 = cu_s[i];
    const int n = cu_s[i + 1] - c0 - 1;
    const int d0 = c0 - i;
    const float tau = tau_s[i];
    const bool greedy = !(tau > 0.0f);
    // s2 = log2(e) / tau as a double-float
    float s2h = 0.0f, s2l = 0.0f;
    if (!greedy) {
      s2h = kLog2eHi / tau;
      s2l = (fmaf(-s2h, tau, kLog2eHi) + kLog2eLo) / tau;
    }
    const float* urow = p.uniforms + static_cast<size_t>(i) * (p.k_max + 1);
    // accept tests of all slots in parallel (thread j tests slot j)
    if (tid == 0) { s_a = n; s_pick = 0; }
    __syncthreads();
    if (tid < n) {
      const int j = tid;
      const int x = p.draft_ids[d0 + j];
      const bool x_ok = x >= 0 && x < V;
      if (!x_ok) raise_error(p.err, SD_DEV_ERR_DRAFT_ID);
      const float4 ts = __ldcg(reinterpret_cast<const float4*>(p.st_t + c0 + j));
      bool acc;
      if (greedy) {
        const int amax = __float_as_int(ts.w);
        if (amax < 0) raise_error(p.err, SD_DEV_ERR_LOGITS);
        acc = x_ok && amax >= 0 && x == amax;
      } else {
        const float4 ds = __ldcg(reinterpret_cast<const float4*>(p.st_d + d0 + j));
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
        if (!ok) raise_error(p.err, SD_DEV_ERR_LOGITS);
        const float u = urow[j];
        if (!(u >= 0.0f && u < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
        acc = ok && x_ok && (u * qx) <= px;
        if (p.probs_out) {
          p.probs_out[2 * static_cast<size_t>(d0 + j)] = px;
          p.probs_out[2 * static_cast<size_t>(d0 + j) + 1] = qx;
        }
      }
      if (!acc) atomicMin(&s_a, j);
    }
    __syncthreads();
    const int a = s_a;
    const float4 ts = __ldcg(reinterpret_cast<const float4*>(p.st_t + c0 + a));
    bool residual = false;
    if (greedy) {
      const int amax = __float_as_int(ts.w);
      if (tid == 0) {
        if (amax < 0) raise_error(p.err, SD_DEV_ERR_LOGITS);
        s_pick = amax >= 0 ? amax : 0;
      }
    } else {
      const bool reject = a < n;
      float4 ds = make_float4(0.0f, 1.0f, 0.0f, 0.0f);
      if (reject) ds = __ldcg(reinterpret_cast<const float4*>(p.st_d + d0 + a));
      const bool ok = isfinite(ts.x) && isfinite(ts.y) && ts.y > 0.0f &&
                      (!reject || (isfinite(ds.x) && isfinite(ds.y) && ds.y > 0.0f));
      const float ufin = urow[p.k_max];
      if (tid == 0 && !(ufin >= 0.0f && ufin < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
      if (!ok) {
        if (tid == 0) raise_error(p.err, SD_DEV_ERR_LOGITS);
      } else if (reject) {
        residual = true;
      } else {
        bonus_draw(static_cast<size_t>(c0 + a), make_rows(i, a, ts, ds, false), ufin);
      }
    }
    __syncthreads();
    if (tid == 0) {
      int* o = p.out_tokens + static_cast<size_t>(i) * (p.k_max + 1);
      p.accepted_len[i] = a;
      for (int j = 0; j < a; ++j) o[j] = p.draft_ids[d0 + j];
      o[a] = residual ? -1 : s_pick;  // a residual token is written by its last slice
      for (int j = a + 1; j <= p.k_max; ++j) o[j] = -1;
      p.req_cnt[i] = 0;  // leave the workspace ready for the next call
      if (!greedy) {
        if (residual) {
          const int pos = atomicAdd(&p.ctrl[2], 1);
          st_release(&p.res_list[pos], 1 + ((i << 4) | a));  // publishes the outputs too
        }
        atom_add_acq_rel(&p.ctrl[4], 1);  // one more sampling request decided
      }
    }
    __syncthreads();
  };

  // ------------------------------------------------------------------------
  // Work loop.  Position k of this CTA's queue (s_q[k & 3]) holds a row
  // unit, a residual draw, or a token (kPoll, kNoop, kEnd).  Warp BW lane 0
  // schedules position k + 3 right after the barrier that ends position k:
  // a listed residual draw is claimed first, else the next row of the work
  // list; once the rows are exhausted it yields kPoll (a draw may still be
  // listed) or, when every sampling request is decided and every listed
  // draw claimed, kEnd.  After that barrier warp BW also folds the warps'
  // partials into the row statistics and counts the row for its request
  // with an acquire-release increment whose result is read at the end of
  // the next position: the CTA that saw the last row of a request runs the
  // request's tail.
  // Scheduler (warp BW lane 0).  Slices are handed out in order by an
  // atomic counter (ctrl[3]); slot h is slice h % S_sl of the (h / S_sl)-th
  // listed draw.  A slot taken before its draw is listed is held and
  // scheduled once listed, or dropped once every sampling request is decided
  // without it being listed.  The next row id is fetched one schedule ahead
  // so that its atomic's latency is hidden.
  bool rows_done = false;
  int stash = 0;   // next row id
  int held = -1;   // a slot taken but not yet listed
  // (listed draws, slots taken): ctrl[2] and ctrl[3] in one 8-byte read
  auto load_lc = [&]() {
    return ld_relaxed_u64(reinterpret_cast<const unsigned long long*>(p.ctrl + 2));
  };
  // The queue entry of listed slot h.
  auto slot_entry = [&](int h) -> int {
    const int e = h / S_sl, sl = h - e * S_sl;
    int v = 0;  // the draw is listed; its publisher may be finishing the store
    for (uint32_t it = 0; it < kSpinLimit; ++it) {
      v = ld_acquire(&p.res_list[e]);
      if (v != 0) break;
      __nanosleep(32);
    }
    if (v == 0) {
      raise_error(p.err, SD_DEV_ERR_TIMEOUT);
      return kNoop;
    }
    return kResBase | (e << 18) | (sl << 16) | (v - 1);
  };
  // A listed slice for this CTA (held, or newly taken when lc shows one
  // untaken), else -1.
  auto claim_residual = [&](unsigned long long lc) -> int {
    const int avail = static_cast<int>(lc & 0xFFFFFFFFull) * S_sl;
    if (held < 0 && static_cast<int>(lc >> 32) < avail) held = atomicAdd(&p.ctrl[3], 1);
    if (held >= 0 && held < avail) {
      const int h = held;
      held = -1;
      return slot_entry(h);
    }
    return -1;
  };
  auto decided = [&]() { return ld_acquire(&p.ctrl[4]) >= s_nsamp; };
  auto schedule = [&](unsigned long long lc) -> int {
    const int r = claim_residual(lc);
    if (r != -1) return r;
    if (!rows_done) {
      const int u = stash;
      if (u < U_stream) {
        stash = atomicAdd(&p.ctrl[0], 1);  // used by the next schedule
        return u;
      }
      rows_done = true;
    }
    if (held < 0 && decided()) {
      const unsigned long long f = load_lc();  // final list
      if (static_cast<int>(f >> 32) >= static_cast<int>(f & 0xFFFFFFFFull) * S_sl) return kEnd;
      held = atomicAdd(&p.ctrl[3], 1);
      if (held < static_cast<int>(f & 0xFFFFFFFFull) * S_sl) {
        const int h = held;
        held = -1;
        return slot_entry(h);
      }
      held = -1;  // past the final list
      return kEnd;
    }
    return kPoll;
  };
  // kPoll: settle the held slot if its draw is listed (or never will be).
  auto poll = [&]() -> int {
    const unsigned long long f = load_lc();
    const int r = claim_residual(f);
    if (r != -1) return r;
    if (held >= 0 && decided()) {
      const int avail = static_cast<int>(load_lc() & 0xFFFFFFFFull) * S_sl;
      if (held < avail) {
        const int h = held;
        held = -1;
        return slot_entry(h);
      }
      held = -1;  // past the final list
    }
    return kNoop;
  };
  if (warp == BW && lane == 0) {  // the first three positions: rows (no draw is listed yet)
    const int u0 = atomicAdd(&p.ctrl[0], 4);
    for (int q = 0; q < 3; ++q) {
      if (u0 + q < U_stream) {
        s_q[q] = u0 + q;
      } else {
        rows_done = true;
        s_q[q] = decided() ? kEnd : kPoll;
      }
    }
    stash = u0 + 3;
  }
  __syncthreads();
  if constexpr (VEC) refill(1);

  int pend_i = -1, pend_old = 0, pend_rows = 0;  // warp BW lane 0: outstanding count
  uint32_t polls = 0;                            // warp BW lane 0: fruitless polls
  for (int k = 0;; ++k) {
    int cur = s_q[k & 3];
    if (cur == kEnd) break;
    const int par = k & 1;
    unsigned long long lc = 0;
    if (warp == BW && lane == 0) lc = load_lc();  // consumed by this position's schedule
    if (cur == kPoll) {
      // Settle this CTA's own outstanding row count first: a tail it owes
      // may be what the others wait for.
      if (warp == BW && lane == 0) {
        s_pending[par] = (pend_i >= 0 && pend_old == pend_rows - 1) ? pend_i : -1;
        pend_i = -1;
      }
      __syncthreads();
      if (s_pending[par] >= 0) {
        __threadfence();
        tail(s_pending[par]);
      }
      // One attempt: later positions may already hold this CTA's slices, so
      // a poll never blocks; the scheduler keeps adding kPoll until the call
      // is over (kEnd), bounded by kSpinLimit polls.
      if (warp == BW && lane == 0) {
        int r = poll();
        if (r == kNoop) {
          if (++polls > kSpinLimit) {
            raise_error(p.err, SD_DEV_ERR_TIMEOUT);
            r = kEnd;
          } else {
            __nanosleep(200);
          }
        }
        s_q[k & 3] = r;
      }
      __syncthreads();
      cur = s_q[k & 3];
      if (cur == kEnd) break;
    }
    const bool is_row = cur < U_stream;
    const bool is_res = cur >= kResBase && cur < kNoop;
    Unit t{};
    float s2 = 0.0f;
    int ri = 0, ra = 0, re = 0;
    if (is_row) {
      t = locate(cur);
      const int x = t.j < t.n ? p.draft_ids[t.c0 - t.i + t.j] : -1;
      const bool x_ok = x >= 0 && x < V;
      const float tau = tau_s[t.i];
      s2 = t.greedy ? 0.0f : kLog2e / tau;

      float best = -INFINITY;  // greedy
      int bidx = INT_MAX, nanf = 0, bv = -1;
      Raw bvec;
      float m = -INFINITY, nb = 0.0f;  // sampling
      float2 z2 = make_float2(0.0f, 0.0f);
      if constexpr (VEC) {
        const int cx = x_ok ? x / EPC : -1;
        refill(k + 1);
        for (int c = cb_w; c < ce_w; ++c) {
          const int slot = static_cast<int>(cseq % kSlots);
          uint64_t* bar = &mbar[warp * kSlots + slot];
          if (!mbar_wait_bounded(bar, (cseq / kSlots) & 1, 1u << 24))
            raise_error(p.err, SD_DEV_ERR_TIMEOUT);
          const unsigned char* chunk = ring + (warp * kSlots + slot) * CB;
          const int nv = min(VPC, nvec - c * VPC);
          if (c == cx && lane == 0) {
            float v;
            if (sizeof(T) == 2)
              v = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(chunk)[x - c * EPC]) << 16);
            else
              v = reinterpret_cast<const float*>(chunk)[x - c * EPC];
            s_lx[par] = v;
          }
          Raw rv[VPL];
  #pragma unroll
          for (int q = 0; q < VPL; ++q)
            rv[q] = lane + 32 * q < nv ? reinterpret_cast<const Raw*>(chunk)[lane + 32 * q]
                                       : ChunkOps<T>::neg_inf();
          if (t.greedy) ChunkOps<T>::argmax(rv, c * VPC + lane, best, bvec, bv, nanf);
          else ChunkOps<T>::softmax(rv, s2, m, z2, nb);
          __syncwarp();
          ++cseq;
          refill(k + 1);
        }
        if (t.greedy && bv >= 0) bidx = ChunkOps<T>::first_of(bvec, bv, best);
      } else {
        const Raw* rowp = reinterpret_cast<const Raw*>(row_base(t));
        float b = 0.0f, z = 0.0f;
        const int eb = min(nvec, warp * RU), ee = min(nvec, eb + RU);  // this warp's range
        for (int v0 = eb + lane; v0 < ee; v0 += 32 * kUnroll) {
          Raw rv[kUnroll];
  #pragma unroll
          for (int q = 0; q < kUnroll; ++q) {
            const int v = v0 + q * 32;
            if (v < ee) rv[q] = ld_stream(rowp + v);
          }
  #pragma unroll
          for (int q = 0; q < kUnroll; ++q) {
            const int v = v0 + q * 32;
            if (v < ee) {
              float f[VE];
              Tr::unpack(rv[q], f);
              if (v == x) s_lx[par] = f[0];
              if (t.greedy) {
                nanf |= (f[0] != f[0]);
                if (f[0] > best) { best = f[0]; bidx = v; }
              } else {
                online_add<VE>(f, s2, m, z, b);
              }
            }
          }
        }
        z2 = make_float2(z, 0.0f);
      }

      // warp partials
      if (t.greedy) {
        unsigned long long key = bidx == INT_MAX ? 0ull
            : (static_cast<unsigned long long>(ordered_bits(best)) << 32) |
                  static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(bidx));
        key = warp_max_u64(key);
        nanf = __any_sync(kFull, nanf);
        if (lane == 0) { red_k[par][warp] = key; red_n[par][warp] = nanf; }
      } else {
        const float mw = warp_max(m);
        const float zr = (m == -INFINITY || mw == -INFINITY) ? 0.0f
                                                            : (z2.x + z2.y) * exp2_ftz((m - mw) * s2);
        const float zw = warp_sum(zr);
        if (lane == 0) {
          red_m[par][warp] = mw;
          red_z[par][warp] = zw;
          if (!t.draft) __stcg(p.st_r + t.row * kMaxRanges + warp, make_float2(mw, zw));
        }
      }
    } else if (is_res) {
      // Slice sl of listed residual draw re (request ri, first rejected slot
      // ra): the sl-th part of each warp's range of the row pair streams
      // through the ring like a row (target and draft chunk c in consecutive
      // entries); each warp adds its sum of max(p - q, 0), in 2^56 fixed
      // point, to the draw's range sum.
      ri = (cur >> 4) & 0xFFF;
      ra = cur & 15;
      re = (cur >> 18) & 0xFFF;
      const int sl = (cur >> 16) & 3;
      const int c0r = cu_s[ri];
      const float4 ts = __ldcg(reinterpret_cast<const float4*>(p.st_t + c0r + ra));
      const float4 ds = __ldcg(reinterpret_cast<const float4*>(p.st_d + c0r - ri + ra));
      const DrawRows w = make_rows(ri, ra, ts, ds, true);
      if (tid == 0) s_dr = w;  // for the finish after the barrier
      const auto fr = fast_res(w);
      unsigned long long acc = 0;
      if constexpr (VEC) {
        refill(k + 1);
        const int c_lo = min(ce_w, cb_w + sl * m_sl), c_hi = min(ce_w, c_lo + m_sl);
        for (int c = c_lo; c < c_hi; ++c) {
          const int s0 = static_cast<int>(cseq % kSlots), s1 = static_cast<int>((cseq + 1) % kSlots);
          if (!mbar_wait_bounded(&mbar[warp * kSlots + s0], (cseq / kSlots) & 1, 1u << 24) ||
              !mbar_wait_bounded(&mbar[warp * kSlots + s1], ((cseq + 1) / kSlots) & 1, 1u << 24))
            raise_error(p.err, SD_DEV_ERR_TIMEOUT);
          const Raw* ct = reinterpret_cast<const Raw*>(ring + (warp * kSlots + s0) * CB);
          const Raw* cd = reinterpret_cast<const Raw*>(ring + (warp * kSlots + s1) * CB);
          const int nv = min(VPC, nvec - c * VPC);
#pragma unroll 2
          for (int q = 0; q < VPL; ++q) {
            const int v = lane + 32 * q;
            if (v < nv) acc += __float2ull_rn(__fmul_rn(fr(ct[v], cd[v]), kTwo56));
          }
          __syncwarp();
          cseq += 2;
          refill(k + 1);
        }
      } else {
        const int we = min(nvec, warp * RU + RU);  // end of this warp's range
        const int eb = min(we, warp * RU + sl * mu_sl), ee = min(we, eb + mu_sl);
        for (int v0 = eb + lane; v0 < ee; v0 += 32 * kUnroll) {
          Raw at[kUnroll], ad[kUnroll];
#pragma unroll
          for (int q = 0; q < kUnroll; ++q) {
            const int v = v0 + q * 32;
            if (v < ee) {
              at[q] = ld_stream(w.rt + v);
              ad[q] = ld_stream(w.rd + v);
            }
          }
#pragma unroll
          for (int q = 0; q < kUnroll; ++q)
            if (v0 + q * 32 < ee) acc += __float2ull_rn(__fmul_rn(fr(at[q], ad[q]), kTwo56));
        }
      }
      acc = warp_sum_u64(acc);
      if (lane == 0 && acc != 0) atomicAdd(p.rs + static_cast<size_t>(re) * kMaxRanges + warp, acc);
    }
    if (warp == BW && lane == 0) {
      s_pending[par] = (pend_i >= 0 && pend_old == pend_rows - 1) ? pend_i : -1;
      pend_i = -1;
    }
    __syncthreads();
    if (is_row && warp == BW) {
        float4 stat;
        if (t.greedy) {
          const unsigned long long kk = warp_max_u64(lane < NW ? red_k[par][lane] : 0ull);
          const int nn = __any_sync(kFull, lane < NW ? red_n[par][lane] : 0);
          const float bv = from_ordered(static_cast<uint32_t>(kk >> 32));
          const bool rowbad = nn || kk == 0ull || !isfinite(bv);
          const int amax = rowbad ? -1 : static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(kk));
          stat = make_float4(bv, 0.0f, s_lx[par], __int_as_float(amax));
        } else {
          const float mw = lane < NW ? red_m[par][lane] : -INFINITY;
          const float M = warp_max(mw);
          const float zr = (lane < NW && mw != -INFINITY && M != -INFINITY)
                               ? red_z[par][lane] * exp2_ftz((mw - M) * s2)
                               : 0.0f;
          stat = make_float4(M, warp_sum(zr), s_lx[par], __int_as_float(0));
        }
        if (lane == 0) {
          RowStat* dst = t.draft ? p.st_d + t.row : p.st_t + t.row;
          __stcg(reinterpret_cast<float4*>(dst), stat);
          pend_rows = (t.n + 1) + (t.greedy ? 0 : t.n);
          pend_i = t.i;
          __threadfence();  // the statistics are visible before the count
        pend_old = atomicAdd(&p.req_cnt[t.i], 1);  // read one position later
        }
    }
    if constexpr (VEC) refill(k + 2);  // position k + 2 is known since the last barrier
    if (is_res) {
      if (tid == 0) s_last = atom_add_acq_rel(&p.slice_cnt[re], 1) == S_sl - 1;
      __syncthreads();
    }
    if (is_res && s_last) {
      // The last slice finishes the draw: the crossing range from the range
      // sums, then its crossing chunk (read again), then the precise walk of
      // that chunk.  The draw's entries go back to zero for the next call.
      __threadfence();
      if (tid < NW) {
        s_Rr[tid] = __ldcg(p.rs + static_cast<size_t>(re) * kMaxRanges + tid);
        p.rs[static_cast<size_t>(re) * kMaxRanges + tid] = 0;
      }
      if (tid == 0) {
        p.slice_cnt[re] = 0;
        p.res_list[re] = 0;
      }
      const float ufin = p.uniforms[static_cast<size_t>(ri) * (p.k_max + 1) + p.k_max];
      const DrawRows w = s_dr;
      crossing(s_Rr, NW, true, ufin, 0ull);
      if (s_found) {
        const int ub = min(nvec, s_ch * RU), ue = min(nvec, ub + RU);
        const unsigned long long th_r = s_th;
        const int nc = (ue - ub + CUd - 1) / CUd;
        chunk_sums(std::true_type{}, w.rt, w.rd, fast_res(w), kTwo56, ub, ue, 0, nc, s_R);
        crossing(s_R, nc, false, 0.0f, th_r);
        if (s_found) {
          const int cb = ub + s_ch * CUd;
          pick_in(precise_res(w), cb, min(cb + CUd, ue), s_th);
        } else {
          pick_in(precise_res(w), ub, ue, 0ull);
        }
      } else {
        bonus_draw(static_cast<size_t>(cu_s[ri] + ra), w, ufin);  // no residual mass in fp32
      }
      if (tid == 0) p.out_tokens[static_cast<size_t>(ri) * (p.k_max + 1) + ra] = s_pick;
    }
    const int tail_i = s_pending[par];
    if (tail_i >= 0) {
      __threadfence();
      tail(tail_i);
    }
    if (warp == BW && lane == 0) s_q[(k + 3) & 3] = schedule(lc);
  }
  // the count of the last unit
  __syncthreads();
  if (warp == BW && lane == 0)
    s_pending[0] = (pend_i >= 0 && pend_old == pend_rows - 1) ? pend_i : -1;
  __syncthreads();
  if (s_pending[0] >= 0) {
    __threadfence();
    tail(s_pending[0]);
  }

  // The last CTA out resets the work counters for the next call.
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
  const int nw = threads / 32;
  const size_t ring = vec ? static_cast<size_t>(nw) * kSlots * (kChunkBytes + 8) : 0;
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
  // 512 threads (16 warps, 192 KB ring) unless the shared memory does not
  // fit (large batches), then 256 threads (96 KB ring).
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
