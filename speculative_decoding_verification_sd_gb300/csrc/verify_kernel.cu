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
// z = sum 2^((l - m) * s2) with m the running maximum.
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
#pragma unroll
    for (int e = 0; e < VE; ++e) z += exp2_ftz(fmaf(f[e], s2, -b));
  }
}

constexpr int kUnroll = 8;

template <typename T, int NT, bool VEC>
__global__ void __launch_bounds__(NT, NT <= 256 ? 2 : 1) verify_kernel(const VerifyParams p) {
  using Tr = VT<T, VEC>;
  using Raw = typename Tr::Raw;
  constexpr int VE = Tr::VE;
  constexpr int NW = NT / 32;
  static_assert(NW <= 32, "one lane per warp in the cross-warp reductions");

  extern __shared__ __align__(16) unsigned char smem[];
  int* cu_s = reinterpret_cast<int*>(smem);                  // [bs+1]
  float* tau_s = reinterpret_cast<float*>(cu_s + p.bs + 1);  // [bs]
  int* order = reinterpret_cast<int*>(tau_s + p.bs);         // [bs] request order
  int* ustart = order + p.bs;                                // [bs+1] first unit of order[k]
  float* R = reinterpret_cast<float*>(ustart + p.bs + 1);    // [rounds * NW] final-draw sums

  __shared__ float red_f[NW];
  __shared__ float red_g[NW];
  __shared__ unsigned long long red_k[NW];
  __shared__ int red_i[NW];
  __shared__ float s_lx;
  __shared__ int s_unit[2];
  __shared__ int s_last, s_a, s_pick, s_entry, s_count;
  __shared__ float s_S, s_th;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V;
  const int nvec = (V + VE - 1) / VE;  // VE divides V on the vector path
  const int rounds = (nvec + NT - 1) / NT;

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
    __syncthreads();
  }
  const int U_total = ustart[p.bs];

  // ------------------------------------------------------------------------
  // Final draw over one row (pair): the first element whose running weight
  // sum exceeds u * S.  Weights are summed per (round, warp) in vocabulary
  // order; warp 0 finds the entry holding the crossing and recomputes its 32
  // vectors to pick the element.  Rounding disagreements between levels fall
  // back to the last positive weight of the chosen range.  Returns S.
  auto draw = [&](auto weights, float ufin) -> float {
    for (int r = 0; r < rounds; ++r) {
      const int v = r * NT + tid;
      float s = 0.0f;
      if (v < nvec) {
        float w[VE];
        weights(v, w);
#pragma unroll
        for (int e = 0; e < VE; ++e) s += w[e];
      }
      s = warp_sum(s);
      if (lane == 0) R[r * NW + warp] = s;
    }
    __syncthreads();
    if (warp == 0) {
      const int E = rounds * NW;
      const int epl = (E + 31) / 32;
      const int eb = min(E, lane * epl), ee = min(E, eb + epl);
      float ls = 0.0f;
      for (int e = eb; e < ee; ++e) ls += R[e];
      const float inc = warp_inclusive_scan(ls, lane);
      const float S = __shfl_sync(kFull, inc, 31);
      if (lane == 0) s_S = S;
      if (S > 0.0f && isfinite(S)) {
        const float theta = ufin * S;
        const unsigned cm = __ballot_sync(kFull, inc > theta);
        int ln;
        if (cm) {
          ln = __ffs(cm) - 1;
        } else {
          const unsigned pm = __ballot_sync(kFull, ls > 0.0f);
          ln = pm ? 31 - __clz(pm) : 0;
        }
        const float up = __shfl_up_sync(kFull, inc, 1);
        const float excl = ln == 0 ? 0.0f : __shfl_sync(kFull, up, ln);
        if (lane == ln) {
          float run = excl;
          int ent = -1, lastpos = -1;
          for (int e = eb; e < ee; ++e) {
            if (R[e] > 0.0f) lastpos = e;
            if (run + R[e] > theta) { ent = e; break; }
            run += R[e];
          }
          if (ent < 0) {
            ent = lastpos >= 0 ? lastpos : eb;
            run = excl;
            for (int e = eb; e < ent; ++e) run += R[e];
          }
          s_entry = ent;
          s_th = fmaxf(theta - run, 0.0f);
        }
        __syncwarp();
        const int ent = s_entry;
        const float th = s_th;
        const int v = (ent / NW) * NT + (ent % NW) * 32 + lane;
        float w[VE];
        float sv = 0.0f;
        int lane_last = -1;
        if (v < nvec) {
          weights(v, w);
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            sv += w[e];
            if (w[e] > 0.0f) lane_last = v * VE + e;
          }
        } else {
#pragma unroll
          for (int e = 0; e < VE; ++e) w[e] = 0.0f;
        }
        const float vinc = warp_inclusive_scan(sv, lane);
        const float vup = __shfl_up_sync(kFull, vinc, 1);
        const float vex = lane == 0 ? 0.0f : vup;
        const unsigned m = __ballot_sync(kFull, vinc > th);
        int lp = lane_last;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(kFull, lp, o));
        if (m) {
          const int lsel = __ffs(m) - 1;
          if (lane == lsel) {
            float rr = vex;
            int pick = lane_last >= 0 ? lane_last : v * VE;
#pragma unroll
            for (int e = 0; e < VE; ++e) {
              rr += w[e];
              if (rr > th) { pick = v * VE + e; break; }
            }
            s_pick = pick;
          }
        } else if (lane == 0) {
          s_pick = lp >= 0 ? lp : 0;
        }
      }
    }
    __syncthreads();
    return s_S;
  };

  // ------------------------------------------------------------------------
  // Tail of request i: decisions from the row statistics, final draw, outputs.
  auto tail = [&](int i) {
    const int c0 = cu_s[i];
    const int n = cu_s[i + 1] - c0 - 1;
    const int d0 = c0 - i;
    const float tau = tau_s[i];
    const bool greedy = !(tau > 0.0f);
    const float s2 = greedy ? 0.0f : kLog2e / tau;
    const float* urow = p.uniforms + static_cast<size_t>(i) * (p.k_max + 1);
    if (tid == 0) {
      int a = n;
      for (int j = 0; j < n; ++j) {
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
            px = exp2_full(fmaf(ts.z, s2, -ts.x * s2)) / ts.y;
            qx = exp2_full(fmaf(ds.z, s2, -ds.x * s2)) / ds.y;
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
        if (!acc) { a = j; break; }
      }
      s_a = a;
      s_pick = 0;
    }
    __syncthreads();
    const int a = s_a;
    const float4 ts = __ldcg(reinterpret_cast<const float4*>(p.st_t + c0 + a));
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
      } else {
        const Raw* rt = reinterpret_cast<const Raw*>(static_cast<const T*>(p.target) +
                                                     static_cast<size_t>(c0 + a) * V);
        const Raw* rd = reinterpret_cast<const Raw*>(
            static_cast<const T*>(p.draft) + static_cast<size_t>(reject ? d0 + a : 0) * V);
        const float bt = ts.x * s2, bd = ds.x * s2;
        const float iZt = 1.0f / ts.y, iZd = 1.0f / ds.y;
        float S = 0.0f;
        if (reject) {
          S = draw(
              [&](int v, float (&w)[VE]) {
                float f[VE], g[VE];
                Tr::unpack(rt[v], f);
                Tr::unpack(rd[v], g);
#pragma unroll
                for (int e = 0; e < VE; ++e) {
                  const float et = exp2_ftz(fmaf(f[e], s2, -bt));
                  const float ed = exp2_ftz(fmaf(g[e], s2, -bd));
                  w[e] = fmaxf(fmaf(et, iZt, -(ed * iZd)), 0.0f);
                }
              },
              ufin);
        }
        // bonus token, or a residual with no mass in fp32: draw from p
        if (!reject || !(S > 0.0f && isfinite(S))) {
          draw(
              [&](int v, float (&w)[VE]) {
                float f[VE];
                Tr::unpack(rt[v], f);
#pragma unroll
                for (int e = 0; e < VE; ++e) w[e] = exp2_ftz(fmaf(f[e], s2, -bt));
              },
              ufin);
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      int* o = p.out_tokens + static_cast<size_t>(i) * (p.k_max + 1);
      p.accepted_len[i] = a;
      for (int j = 0; j < a; ++j) o[j] = p.draft_ids[d0 + j];
      o[a] = s_pick;
      for (int j = a + 1; j <= p.k_max; ++j) o[j] = -1;
      p.req_cnt[i] = 0;  // leave the workspace ready for the next call
    }
    __syncthreads();
  };

  // ------------------------------------------------------------------------
  // Work loop: one row per unit.
  if (tid == 0) s_unit[0] = atomicAdd(&p.ctrl[0], 1);
  __syncthreads();
  int buf = 0;
  int cur = s_unit[0];
  while (cur < U_total) {
    int nxt = 0;
    if (tid == 0) nxt = atomicAdd(&p.ctrl[0], 1);  // next unit, consumed after this one
    int lo = 0, hi = p.bs;  // ustart[lo] <= cur < ustart[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ustart[mid] <= cur) lo = mid;
      else hi = mid;
    }
    const int i = order[lo];
    const int r = cur - ustart[lo];
    const int c0 = cu_s[i];
    const int n = cu_s[i + 1] - c0 - 1;
    const float tau = tau_s[i];
    const bool greedy = !(tau > 0.0f);
    const bool is_draft = r > n;
    const int j = is_draft ? r - (n + 1) : r;
    const size_t row = is_draft ? static_cast<size_t>(c0 - i + j) : static_cast<size_t>(c0 + j);
    const Raw* rowp = reinterpret_cast<const Raw*>(
        static_cast<const T*>(is_draft ? p.draft : p.target) + row * V);
    const int x = j < n ? p.draft_ids[c0 - i + j] : -1;
    const int vx = (x >= 0 && x < V) ? x / VE : -1;
    if (tid == 0) s_lx = 0.0f;
    __syncthreads();

    float4 stat = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (greedy) {
      float best = -INFINITY;
      int bidx = INT_MAX, nanf = 0;
      for (int v0 = tid; v0 < nvec; v0 += NT * kUnroll) {
        Raw rv[kUnroll];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
          const int v = v0 + q * NT;
          if (v < nvec) rv[q] = ld_stream(rowp + v);
        }
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
          const int v = v0 + q * NT;
          if (v < nvec) {
            float f[VE];
            Tr::unpack(rv[q], f);
            if (v == vx) {
#pragma unroll
              for (int e = 0; e < VE; ++e)
                if (v * VE + e == x) s_lx = f[e];
            }
#pragma unroll
            for (int e = 0; e < VE; ++e) {
              nanf |= (f[e] != f[e]);
              if (f[e] > best) { best = f[e]; bidx = v * VE + e; }
            }
          }
        }
      }
      // Lowest index among the maxima: a thread meets its elements in
      // increasing index order, so its first maximum is its lowest.
      unsigned long long key = bidx == INT_MAX ? 0ull
          : (static_cast<unsigned long long>(ordered_bits(best)) << 32) |
                static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(bidx));
      key = warp_max_u64(key);
      nanf = __any_sync(kFull, nanf);
      if (lane == 0) { red_k[warp] = key; red_i[warp] = nanf; }
      __syncthreads();
      if (tid == 0) {
        unsigned long long kk = 0ull;
        int nn = 0;
        for (int w = 0; w < NW; ++w) {
          kk = red_k[w] > kk ? red_k[w] : kk;
          nn |= red_i[w];
        }
        const float bv = from_ordered(static_cast<uint32_t>(kk >> 32));
        const bool rowbad = nn || kk == 0ull || !isfinite(bv);
        const int amax = rowbad ? -1 : static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(kk));
        stat = make_float4(bv, 0.0f, s_lx, __int_as_float(amax));
      }
    } else {
      const float s2 = kLog2e / tau;
      float m = -INFINITY, z = 0.0f, b = 0.0f;
      for (int v0 = tid; v0 < nvec; v0 += NT * kUnroll) {
        Raw rv[kUnroll];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
          const int v = v0 + q * NT;
          if (v < nvec) rv[q] = ld_stream(rowp + v);
        }
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
          const int v = v0 + q * NT;
          if (v < nvec) {
            float f[VE];
            Tr::unpack(rv[q], f);
            if (v == vx) {
#pragma unroll
              for (int e = 0; e < VE; ++e)
                if (v * VE + e == x) s_lx = f[e];
            }
            online_add<VE>(f, s2, m, z, b);
          }
        }
      }
      // block max, then every thread rescales its sum to the block max
      const float mw = warp_max(m);
      if (lane == 0) red_f[warp] = mw;
      __syncthreads();
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, red_f[w]);
      const float zr = (m == -INFINITY || M == -INFINITY) ? 0.0f : z * exp2_ftz((m - M) * s2);
      const float zw = warp_sum(zr);
      if (lane == 0) red_g[warp] = zw;
      __syncthreads();
      if (tid == 0) {
        float Z = 0.0f;
        for (int w = 0; w < NW; ++w) Z += red_g[w];
        stat = make_float4(M, Z, s_lx, __int_as_float(0));
      }
    }
    if (tid == 0) {
      RowStat* dst = is_draft ? p.st_d + row : p.st_t + row;
      __stcg(reinterpret_cast<float4*>(dst), stat);
      __threadfence();
      const int rows_i = (n + 1) + (greedy ? 0 : n);
      s_last = atomicAdd(&p.req_cnt[i], 1) == rows_i - 1;
      s_unit[buf ^ 1] = nxt;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      tail(i);
    }
    buf ^= 1;
    cur = s_unit[buf];
  }
  // The last CTA out resets the work counters for the next call.
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&p.ctrl[1], 1) == static_cast<int>(gridDim.x) - 1) {
      p.ctrl[0] = 0;
      p.ctrl[1] = 0;
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
  const int VE = vec ? 16 / elem : 1;
  const int nvec = (V + VE - 1) / VE;
  const int rounds = (nvec + threads - 1) / threads;
  return static_cast<size_t>(4) * (4 * static_cast<size_t>(bs) + 2) +
         static_cast<size_t>(rounds) * (threads / 32) * 4 + 16;
}

cudaError_t choose_verify_shape(int V, int elem, int bs, const sd_launch_cfg* req, bool vec,
                                VerifyShape* out, bool* fits) {
  *fits = false;
  const int threads = (req && req->threads) ? req->threads : 512;
  if (threads != 256 && threads != 512) return cudaSuccess;
  void* fn = pick_kernel(elem, vec, threads);
  const size_t smem = verify_smem_bytes(bs, V, elem, vec, threads);
  cudaError_t e = prepare(fn, 0);
  if (e != cudaSuccess) return e;
  if (prepare(fn, smem) != cudaSuccess) return cudaSuccess;  // beyond this build's limits
  int dev = 0, sms = 0, per_sm = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaSuccess;
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
