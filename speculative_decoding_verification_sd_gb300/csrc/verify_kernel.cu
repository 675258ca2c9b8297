// verify_kernel.cu -- K2 (rows) and K3 (finalize): speculative rejection
// sampling over the whole vocabulary, one HBM pass over every compacted row.
//
// Rule (the original papers cited by the fosworld blog "추측 디코딩과 vLLM
// 적응형 검증" under "참고 링크 / 논문"; greedy form in "추측 디코딩이란";
// distribution-preserving per "속도, 메모리, 정확도에 주는 영향", row 정확도):
//   tau > 0: accept slot j iff u_j * q_j(x_j) <= p_j(x_j); at the first
//            rejection draw from max(p - q, 0) normalised; after a fully
//            accepted prefix draw a bonus token from p of the next row.
//   tau = 0: accept iff x_j == argmax p_j; the correction/bonus is the argmax.
//
// Design (GB300): a persistent grid of thread-block clusters.  Each cluster
// owns one compacted row at a time (target row, plus the draft row of the
// same slot when tau > 0); each of its C CTAs holds a 1/C vocabulary slice of
// both rows in shared memory, staged by 1-D bulk copies (cp.async.bulk, one
// per slice, completion on an mbarrier) S items ahead.  Row statistics are
// combined across the cluster through distributed shared memory, so the
// accept test, the residual mass and the inverse-CDF search all run on the
// resident slices: every logit is read from HBM exactly once.  Because the
// row that ends a request's accepted prefix is only known once all its rows
// are decided, every row that could end it (a rejecting row, or the bonus
// row) draws its candidate token speculatively; K3 keeps the right one.
#include <atomic>
#include <algorithm>
#include <climits>
#include <mutex>
#include <utility>

#include "sd_device.cuh"
#include "sd_internal.h"

namespace sdk {

namespace {

constexpr uint32_t kWaitLimit = 1u << 22;

template <typename T>
struct VT;

template <>
struct VT<float> {
  using Raw = float4;
  static constexpr int VE = 4;
  static constexpr int ELEM = 4;
  __device__ __forceinline__ static void unpack(const Raw& r, float (&f)[VE]) {
    f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w;
  }
  __device__ __forceinline__ static float at(const void* base, size_t idx) {
    return static_cast<const float*>(base)[idx];
  }
  __device__ __forceinline__ static void put_neg_inf(void* base, int idx) {
    static_cast<float*>(base)[idx] = -INFINITY;
  }
  __device__ __forceinline__ static void copy(void* dst, int di, const void* src, size_t si) {
    static_cast<float*>(dst)[di] = static_cast<const float*>(src)[si];
  }
};

template <>
struct VT<uint16_t> {  // bf16 bit patterns
  using Raw = uint4;
  static constexpr int VE = 8;
  static constexpr int ELEM = 2;
  __device__ __forceinline__ static void unpack(const Raw& r, float (&f)[VE]) {
    f[0] = __uint_as_float(r.x << 16); f[1] = __uint_as_float(r.x & 0xFFFF0000u);
    f[2] = __uint_as_float(r.y << 16); f[3] = __uint_as_float(r.y & 0xFFFF0000u);
    f[4] = __uint_as_float(r.z << 16); f[5] = __uint_as_float(r.z & 0xFFFF0000u);
    f[6] = __uint_as_float(r.w << 16); f[7] = __uint_as_float(r.w & 0xFFFF0000u);
  }
  __device__ __forceinline__ static float at(const void* base, size_t idx) {
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(base)[idx]) << 16);
  }
  __device__ __forceinline__ static void put_neg_inf(void* base, int idx) {
    static_cast<uint16_t*>(base)[idx] = 0xFF80u;
  }
  __device__ __forceinline__ static void copy(void* dst, int di, const void* src, size_t si) {
    static_cast<uint16_t*>(dst)[di] = static_cast<const uint16_t*>(src)[si];
  }
};

// Per-CTA partials pushed into every peer's shared memory (one entry per
// source CTA), then read locally after the cluster barrier.
struct __align__(16) Slot {
  float mt, zt;  // target: local max and sum of 2^((l - mt) * s2); residual pass: sum
  float md, zd;  // draft: local max and sum
  float lt, ld;  // target / draft logit at the draft token (owner CTA only)
  int flag;      // owns the draft token; greedy: row holds NaN
  int pad;
  unsigned long long key;  // greedy: packed (value, -index) maximum
  unsigned long long pad2;
};

constexpr int kMaxCluster = 16;
constexpr int kMaxRounds = 32;

__device__ __forceinline__ float from_ordered(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// Residual weight max(p - q, 0) of one element pair, with p = 2^(lt*s2 - bt)/Z_t
// and q = 2^(ld*s2 - bd)/Z_d; the same expression serves the sum and the search.
__device__ __forceinline__ float residual_w(float lt, float ld, float s2, float bt, float bd,
                                            float iZt, float iZd) {
  const float et = exp2_ftz(fmaf(lt, s2, -bt));
  const float ed = exp2_ftz(fmaf(ld, s2, -bd));
  return fmaxf(fmaf(et, iZt, -(ed * iZd)), 0.0f);
}

// Merge two (max, scaled sum) pairs of the online softmax.
__device__ __forceinline__ void merge_ms(float& m, float& z, float m2, float z2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) {
    z = 0.0f;
  } else {
    z = z * exp2_ftz((m - M) * s2) + z2 * exp2_ftz((m2 - M) * s2);
  }
  m = M;
}

__device__ __forceinline__ void warp_merge_ms(float& m, float& z, float s2) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(kFull, m, o);
    const float z2 = __shfl_xor_sync(kFull, z, o);
    merge_ms(m, z, m2, z2, s2);
  }
}

// One thread's vector of VE logits into its running (max, sum).
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

template <typename T, int NT, bool BULK>
__global__ void __launch_bounds__(NT, 1) rows_kernel(const VerifyParams p) {
  using Tr = VT<T>;
  using Raw = typename Tr::Raw;
  constexpr int VE = Tr::VE;
  constexpr int ELEM = Tr::ELEM;
  constexpr int NW = NT / 32;
  static_assert(NW <= 32, "one lane per warp in the cross-warp passes");

  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Slot slots[2][2][kMaxCluster];
  __shared__ float Wm_t[NW], Wz_t[NW], Wm_d[NW], Wz_d[NW], Wr[NW];
  __shared__ float Rr[NW][kMaxRounds];
  __shared__ unsigned long long Wk[NW];
  __shared__ int Wn[NW];

  cg::cluster_group cluster = cg::this_cluster();
  const int C = p.C;
  const int rank = static_cast<int>(cluster.block_rank());
  const int cid = blockIdx.x / C;
  const int G = gridDim.x / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V;
  const int SL = p.SL;

  // dynamic shared memory: stages | stage meta (x, u, ufin) | mbarriers | cu | tau
  unsigned char* meta_base = smem + static_cast<size_t>(p.S) * p.stage_bytes;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(meta_base + 16 * 4);
  int* cu_s = reinterpret_cast<int*>(mbar + 4);
  float* tau_s = reinterpret_cast<float*>(cu_s + p.bs + 1);

  // ---- per-call checks of the compaction (identical verdict in every CTA)
  for (int i = tid; i <= p.bs; i += NT) cu_s[i] = p.cu[i];
  __syncthreads();
  int bad = (tid == 0 && cu_s[0] != 0) ? 1 : 0;
  for (int i = tid; i < p.bs; i += NT) {
    const int d = cu_s[i + 1] - cu_s[i];
    if (d < 1 || d > p.k_max + 1) bad = 1;
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && tid == 0) {
      raise_error(p.err, SD_DEV_ERR_CU_SEQLENS);
      *p.ws_status = 1;
    }
    return;  // no cluster barrier entered yet, no copy issued
  }
  if (blockIdx.x == 0 && tid == 0) *p.ws_status = 0;
  int badt = 0;
  for (int i = tid; i < p.bs; i += NT) {
    float t = p.temps[i];
    if (!(t >= 0.0f) || !isfinite(t)) { badt |= SD_DEV_ERR_TEMP; t = 0.0f; }
    if (t > 0.0f && p.draft == nullptr) { badt |= SD_DEV_ERR_LOGITS; t = 0.0f; }
    tau_s[i] = t;
  }
  if (badt && blockIdx.x == 0) raise_error(p.err, badt);
  if (BULK && tid == 0) {
    // one arrival from the bulk-copy issue, one when the metadata copies land
    for (int s = 0; s < p.S; ++s) mbar_init(&mbar[s], 2);
    fence_mbar_init();
  }
  __syncthreads();

  const int lo_e = rank * SL;
  const int len = max(0, min(SL, V - lo_e));
  const int nvec = (len + VE - 1) / VE;
  const int vpw = (nvec + NW - 1) / NW;
  const int vb = min(nvec, warp * vpw);
  const int ve = min(nvec, vb + vpw);
  const int R_total = cu_s[p.bs];
  const int nitems = cid < R_total ? (R_total - cid + G - 1) / G : 0;
  const uint64_t pol = policy_evict_first();

  auto stage_t = [&](int s) { return smem + static_cast<size_t>(s) * p.stage_bytes; };
  auto stage_d = [&](int s) { return stage_t(s) + static_cast<size_t>(SL) * ELEM; };
  auto meta_x = [&](int s) { return reinterpret_cast<int*>(meta_base + 16 * s); };
  auto meta_u = [&](int s) { return reinterpret_cast<float*>(meta_base + 16 * s + 4); };
  auto meta_uf = [&](int s) { return reinterpret_cast<float*>(meta_base + 16 * s + 8); };
  auto locate = [&](int q, int& i, int& j, int& n) {
    int lo = 0, hi = p.bs;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu_s[mid] <= q) lo = mid;
      else hi = mid;
    }
    i = lo;
    j = q - cu_s[i];
    n = cu_s[i + 1] - cu_s[i] - 1;
  };
  auto meta_src = [&](int q, int i, int j, int n, const int*& xs, const float*& us,
                      const float*& ufs) {
    const float* urow = p.uniforms + static_cast<size_t>(i) * (p.k_max + 1);
    us = urow + j;  // j <= n <= k_max
    ufs = urow + p.k_max;
    xs = j < n ? p.draft_ids + (q - i) : reinterpret_cast<const int*>(ufs);
  };
  // Producer (thread 0): stage item q into stage s -- logit slices by bulk
  // copy, the draft token and uniforms by 4-byte asynchronous copies.
  auto issue = [&](int q, int s) {
    int i, j, n;
    locate(q, i, j, n);
    const bool hd = tau_s[i] > 0.0f && j < n;
    const int* xs;
    const float *us, *ufs;
    meta_src(q, i, j, n, xs, us, ufs);
    cp_async4(meta_x(s), xs);
    cp_async4(meta_u(s), us);
    cp_async4(meta_uf(s), ufs);
    cp_async_arrive_noinc(&mbar[s]);
    const uint32_t bytes = static_cast<uint32_t>(len) * ELEM;
    mbar_arrive_expect_tx(&mbar[s], hd ? 2 * bytes : bytes);
    if (len > 0) {
      const char* tg = static_cast<const char*>(p.target) +
                       (static_cast<size_t>(q) * V + lo_e) * ELEM;
      bulk_load(stage_t(s), tg, bytes, &mbar[s], pol);
      if (hd) {
        const char* dg = static_cast<const char*>(p.draft) +
                         (static_cast<size_t>(q - i) * V + lo_e) * ELEM;
        bulk_load(stage_d(s), dg, bytes, &mbar[s], pol);
      }
    }
  };
  // Staged path for layouts the bulk copy cannot take (V*elem or a base
  // pointer not 16-byte aligned): plain loads, tail padded with -inf.
  auto load_plain = [&](int q, int s) {
    int i, j, n;
    locate(q, i, j, n);
    const bool hd = tau_s[i] > 0.0f && j < n;
    const size_t tb = static_cast<size_t>(q) * V + lo_e;
    const size_t db = static_cast<size_t>(q - i) * V + lo_e;
    for (int e = tid; e < nvec * VE; e += NT) {
      if (e < len) Tr::copy(stage_t(s), e, p.target, tb + e);
      else Tr::put_neg_inf(stage_t(s), e);
      if (hd) {
        if (e < len) Tr::copy(stage_d(s), e, p.draft, db + e);
        else Tr::put_neg_inf(stage_d(s), e);
      }
    }
    if (tid == 0) {
      const int* xs;
      const float *us, *ufs;
      meta_src(q, i, j, n, xs, us, ufs);
      *meta_x(s) = *xs;
      *meta_u(s) = *us;
      *meta_uf(s) = *ufs;
    }
    __syncthreads();
  };
  // Pushes warp 0's value `v` (valid in lanes < C) into slot [par][ph][rank]
  // of every CTA of the cluster, then waits for all peers' pushes.
  auto exchange = [&](int par, int ph, const Slot& v) {
    if (warp == 0 && lane < C) *cluster.map_shared_rank(&slots[par][ph][rank], lane) = v;
    cluster.sync();
  };

  // Element search over this CTA's slice: the first element at which the
  // running sum of weights exceeds theta.  `y_c` (lane c < C) holds the CTA
  // totals, `y_w` (lane w < NW) this CTA's per-warp totals, `rsum` (nullable)
  // the warp's per-round totals; `wfun(v, w)` fills the VE weights of vector
  // v.  Only the CTA, warp and round holding the crossing go down a level;
  // rounding disagreements between levels fall back to the last positive
  // weight of the chosen range.
  auto owner_search = [&](float theta, float y_c, float y_w, const float* rsum_base, int q,
                          auto wfun) {
    const float c_inc = warp_inclusive_scan(lane < C ? y_c : 0.0f, lane);
    const unsigned cross = __ballot_sync(kFull, lane < C && c_inc > theta);
    int cstar;
    if (cross) {
      cstar = __ffs(cross) - 1;
    } else {
      const unsigned pos = __ballot_sync(kFull, lane < C && y_c > 0.0f);
      cstar = pos ? 31 - __clz(pos) : 0;
    }
    const float up_c = __shfl_up_sync(kFull, c_inc, 1);
    const float excl_c = cstar == 0 ? 0.0f : __shfl_sync(kFull, up_c, cstar);
    if (rank != cstar) return;
    const float th_c = fmaxf(theta - excl_c, 0.0f);
    const float ww = lane < NW ? y_w : 0.0f;
    const float winc = warp_inclusive_scan(ww, lane);
    const unsigned cw = __ballot_sync(kFull, lane < NW && winc > th_c);
    int wstar;
    if (cw) {
      wstar = __ffs(cw) - 1;
    } else {
      const unsigned pos = __ballot_sync(kFull, lane < NW && ww > 0.0f);
      wstar = pos ? 31 - __clz(pos) : 0;
    }
    const float up_w = __shfl_up_sync(kFull, winc, 1);
    const float excl_w = wstar == 0 ? 0.0f : __shfl_sync(kFull, up_w, wstar);
    if (warp != wstar) return;
    const float th = fmaxf(th_c - excl_w, 0.0f);
    const int wb = min(nvec, wstar * vpw);
    const int we = min(nvec, wb + vpw);
    const int nr = (we - wb + 31) / 32;
    const float* rsum = rsum_base ? rsum_base + wstar * kMaxRounds : nullptr;
    for (int attempt = 0; attempt < 2; ++attempt) {
      float run = 0.0f;
      int r0 = 0;
      if (rsum && attempt == 0 && nr <= kMaxRounds) {
        while (r0 < nr - 1 && run + rsum[r0] <= th) run += rsum[r0++];
      }
      int last_pos = -1;
      for (int base = wb + 32 * r0; base < we; base += 32) {
        const int v = base + lane;
        float w[VE];
        float sv = 0.0f;
        int lane_last = -1;
        if (v < we) {
          wfun(v, w);
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            sv += w[e];
            if (w[e] > 0.0f) lane_last = lo_e + v * VE + e;
          }
        } else {
#pragma unroll
          for (int e = 0; e < VE; ++e) w[e] = 0.0f;
        }
        const float inc = warp_inclusive_scan(sv, lane);
        const float up = __shfl_up_sync(kFull, inc, 1);
        const float excl = lane == 0 ? 0.0f : up;
        const unsigned m = __ballot_sync(kFull, run + inc > th);
        int lp = lane_last;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(kFull, lp, o));
        last_pos = max(last_pos, lp);
        if (m) {
          const int ls = __ffs(m) - 1;
          if (lane == ls) {
            float r = run + excl;
            int pick = lane_last >= 0 ? lane_last : lo_e + v * VE;
#pragma unroll
            for (int e = 0; e < VE; ++e) {
              r += w[e];
              if (r > th) { pick = lo_e + v * VE + e; break; }
            }
            p.ws_cand[q] = pick;
          }
          return;
        }
        run += __shfl_sync(kFull, inc, 31);
      }
      if (r0 == 0 || attempt == 1) {
        if (lane == 0) p.ws_cand[q] = last_pos >= 0 ? last_pos : lo_e + wb * VE;
        return;
      }
      // the stored round totals skipped past the crossing: rescan from the start
    }
  };

  if (BULK && tid == 0)
    for (int k = 0; k < min(p.S, nitems); ++k) issue(cid + k * G, k);

  for (int k = 0; k < nitems; ++k) {
    const int q = cid + k * G;
    const int st = k % p.S;
    const int par = k & 1;
    if (BULK) {
      if (!mbar_wait_bounded(&mbar[st], static_cast<uint32_t>((k / p.S) & 1), kWaitLimit))
        raise_error(p.err, SD_DEV_ERR_TIMEOUT);
    } else {
      load_plain(q, st);
    }
    int i, j, n;
    locate(q, i, j, n);
    const float tau = tau_s[i];
    const bool greedy = !(tau > 0.0f);
    const bool has_draft = !greedy && j < n;
    const bool bonus = (j == n);
    const Raw* vt = reinterpret_cast<const Raw*>(stage_t(st));
    const Raw* vd = reinterpret_cast<const Raw*>(stage_d(st));
    const int x = *meta_x(st);
    const float u = *meta_u(st);
    const float ufin = *meta_uf(st);
    const bool x_ok = !bonus && x >= 0 && x < V;
    const bool lead = (rank == 0 && tid == 0);

    if (greedy) {
      // ---------------- argmax (lowest index on ties), one exchange
      float best = -INFINITY;
      int bidx = INT_MAX;
      int nanf = 0;
      for (int v = vb + lane; v < ve; v += 32) {
        float f[VE];
        Tr::unpack(vt[v], f);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          nanf |= (f[e] != f[e]);
          if (f[e] > best) { best = f[e]; bidx = lo_e + v * VE + e; }
        }
      }
      unsigned long long key = bidx == INT_MAX ? 0ull
          : (static_cast<unsigned long long>(ordered_bits(best)) << 32) |
                static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(bidx));
      key = warp_max_u64(key);
      nanf = __any_sync(kFull, nanf);
      if (lane == 0) { Wk[warp] = key; Wn[warp] = nanf; }
      __syncthreads();
      if (warp == 0) {
        Slot sv;
        sv.key = warp_max_u64(lane < NW ? Wk[lane] : 0ull);
        sv.flag = __any_sync(kFull, lane < NW ? Wn[lane] : 0);
        exchange(par, 0, sv);
      } else {
        cluster.sync();
      }
      const Slot& pc = slots[par][0][lane < C ? lane : 0];
      const unsigned long long kk = warp_max_u64(lane < C ? pc.key : 0ull);
      const int nn = __any_sync(kFull, lane < C ? pc.flag : 0);
      const float bv = from_ordered(static_cast<uint32_t>(kk >> 32));
      const bool rowbad = nn || kk == 0ull || !isfinite(bv);
      const int amax = rowbad ? 0 : static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(kk));
      if (lead) {
        if (rowbad) raise_error(p.err, SD_DEV_ERR_LOGITS);
        if (!bonus && !x_ok) raise_error(p.err, SD_DEV_ERR_DRAFT_ID);
        p.ws_accept[q] = bonus ? 1 : static_cast<uint8_t>(x_ok && !rowbad && x == amax);
        p.ws_cand[q] = amax;
      }
    } else {
      const float s2 = kLog2e / tau;
      // ---------------- fused max + sum (online softmax), one exchange
      float mt = -INFINITY, zt = 0.0f, bt_run = 0.0f;
      float md = -INFINITY, zd = 0.0f, bd_run = 0.0f;
      for (int v = vb + lane; v < ve; v += 32) {
        float f[VE];
        Tr::unpack(vt[v], f);
        online_add<VE>(f, s2, mt, zt, bt_run);
        if (has_draft) {
          Tr::unpack(vd[v], f);
          online_add<VE>(f, s2, md, zd, bd_run);
        }
      }
      warp_merge_ms(mt, zt, s2);
      if (has_draft) warp_merge_ms(md, zd, s2);
      if (lane == 0) { Wm_t[warp] = mt; Wz_t[warp] = zt; Wm_d[warp] = md; Wz_d[warp] = zd; }
      __syncthreads();
      if (warp == 0) {
        float m1 = lane < NW ? Wm_t[lane] : -INFINITY, z1 = lane < NW ? Wz_t[lane] : 0.0f;
        float m2 = lane < NW ? Wm_d[lane] : -INFINITY, z2 = lane < NW ? Wz_d[lane] : 0.0f;
        warp_merge_ms(m1, z1, s2);
        if (has_draft) warp_merge_ms(m2, z2, s2);
        Slot sv;
        sv.mt = m1; sv.zt = z1; sv.md = m2; sv.zd = z2;
        sv.flag = 0;
        sv.lt = 0.0f; sv.ld = 0.0f;
        if (x_ok && x >= lo_e && x < lo_e + len) {
          sv.lt = Tr::at(stage_t(st), x - lo_e);
          sv.ld = has_draft ? Tr::at(stage_d(st), x - lo_e) : 0.0f;
          sv.flag = 1;
        }
        exchange(par, 0, sv);
      } else {
        cluster.sync();
      }
      // Global statistics, identical in every CTA and warp.
      const Slot& pc = slots[par][0][lane < C ? lane : 0];
      const float mt_c = lane < C ? pc.mt : -INFINITY, zt_c = lane < C ? pc.zt : 0.0f;
      const float md_c = lane < C ? pc.md : -INFINITY, zd_c = lane < C ? pc.zd : 0.0f;
      const float Mt = warp_max(mt_c);
      const float Md = warp_max(md_c);
      const float bt = Mt * s2, bd = Md * s2;
      const float yt_c = (lane < C && mt_c != -INFINITY) ? zt_c * exp2_ftz(fmaf(mt_c, s2, -bt)) : 0.0f;
      const float yd_c = (lane < C && md_c != -INFINITY) ? zd_c * exp2_ftz(fmaf(md_c, s2, -bd)) : 0.0f;
      const float Zt = __shfl_sync(kFull, warp_inclusive_scan(yt_c, lane), 31);
      const float Zd = __shfl_sync(kFull, warp_inclusive_scan(yd_c, lane), 31);
      const int cx = x_ok ? min(x / SL, C - 1) : 0;
      const float ltx = slots[par][0][cx].lt;
      const float ldx = slots[par][0][cx].ld;
      const bool rowbad = !isfinite(Mt) || !(isfinite(Zt) && Zt > 0.0f) ||
                          (has_draft && (!isfinite(Md) || !(isfinite(Zd) && Zd > 0.0f)));
      auto p_weight = [&](int v, float (&w)[VE]) {
        float f[VE];
        Tr::unpack(vt[v], f);
#pragma unroll
        for (int e = 0; e < VE; ++e) w[e] = exp2_ftz(fmaf(f[e], s2, -bt));
      };
      bool need_residual = false, need_p = false;
      if (bonus) {
        need_p = !rowbad;
        if (lead) {
          if (rowbad) raise_error(p.err, SD_DEV_ERR_LOGITS);
          if (!(ufin >= 0.0f && ufin < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
          p.ws_accept[q] = 1;
          if (rowbad) p.ws_cand[q] = 0;
        }
      } else {
        float px = 0.0f, qx = 0.0f;
        bool acc = false;
        if (x_ok && !rowbad) {
          px = exp2_full(fmaf(ltx, s2, -bt)) / Zt;
          qx = exp2_full(fmaf(ldx, s2, -bd)) / Zd;
          acc = (u * qx) <= px;
        }
        need_residual = !acc && !rowbad;
        if (lead) {
          if (rowbad) raise_error(p.err, SD_DEV_ERR_LOGITS);
          if (!x_ok) raise_error(p.err, SD_DEV_ERR_DRAFT_ID);
          if (!(u >= 0.0f && u < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
          if (!acc && !(ufin >= 0.0f && ufin < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
          p.ws_accept[q] = static_cast<uint8_t>(acc);
          if (rowbad) p.ws_cand[q] = 0;
          if (p.probs_out) {
            p.probs_out[2 * static_cast<size_t>(q - i)] = px;
            p.probs_out[2 * static_cast<size_t>(q - i) + 1] = qx;
          }
        }
      }
      if (need_residual) {
        // ---------------- residual mass max(p - q, 0), per-round totals kept
        const float iZt = 1.0f / Zt, iZd = 1.0f / Zd;
        float wsum = 0.0f;
        int r = 0;
        for (int base = vb; base < ve; base += 32, ++r) {
          const int v = base + lane;
          float sv = 0.0f;
          if (v < ve) {
            float f[VE], g[VE];
            Tr::unpack(vt[v], f);
            Tr::unpack(vd[v], g);
#pragma unroll
            for (int e = 0; e < VE; ++e) sv += residual_w(f[e], g[e], s2, bt, bd, iZt, iZd);
          }
          const float rs = warp_sum(sv);
          if (lane == 0 && r < kMaxRounds) Rr[warp][r] = rs;
          wsum += rs;
        }
        if (lane == 0) Wr[warp] = wsum;
        __syncthreads();
        if (warp == 0) {
          Slot sv;
          sv.zt = __shfl_sync(kFull, warp_inclusive_scan(lane < NW ? Wr[lane] : 0.0f, lane), 31);
          exchange(par, 1, sv);
        } else {
          cluster.sync();
        }
        const float sr_c = lane < C ? slots[par][1][lane].zt : 0.0f;
        const float S = __shfl_sync(kFull, warp_inclusive_scan(sr_c, lane), 31);
        if (S > 0.0f && isfinite(S)) {
          owner_search(ufin * S, sr_c, lane < NW ? Wr[lane] : 0.0f, &Rr[0][0], q,
                       [&](int v, float (&w)[VE]) {
                         float f[VE], g[VE];
                         Tr::unpack(vt[v], f);
                         Tr::unpack(vd[v], g);
#pragma unroll
                         for (int e = 0; e < VE; ++e)
                           w[e] = residual_w(f[e], g[e], s2, bt, bd, iZt, iZd);
                       });
        } else {
          need_p = true;  // no residual mass in fp32: draw from p instead
        }
      }
      if (need_p) {
        float yw = 0.0f;
        if (lane < NW && Wm_t[lane] != -INFINITY)
          yw = Wz_t[lane] * exp2_ftz(fmaf(Wm_t[lane], s2, -bt));
        owner_search(ufin * Zt, yt_c, yw, nullptr, q, p_weight);
      }
    }
    __syncthreads();  // stage st and the per-warp arrays are free again
    if (BULK && tid == 0 && k + p.S < nitems) issue(cid + (k + p.S) * G, st);
  }
  cluster.sync();  // peers may still push into this CTA's slots
}

__global__ void finalize_kernel(const int* __restrict__ draft_ids, const int* __restrict__ cu,
                                int bs, int k_max, int* __restrict__ accepted_len,
                                int* __restrict__ out_tokens, int* err,
                                const uint8_t* __restrict__ ws_accept,
                                const int* __restrict__ ws_cand, const int* __restrict__ ws_status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= bs) return;
  int* o = out_tokens + static_cast<size_t>(i) * (k_max + 1);
  const int c0 = cu[i], c1 = cu[i + 1];
  const int n = c1 - c0 - 1;
  const bool ok = *ws_status == 0 && c0 >= 0 && n >= 0 && n <= k_max &&
                  c1 <= bs * (k_max + 1);
  if (!ok) {
    if (*ws_status == 0) raise_error(err, SD_DEV_ERR_CU_SEQLENS);
    accepted_len[i] = 0;
    for (int j = 0; j <= k_max; ++j) o[j] = -1;
    return;
  }
  int a = n;
  for (int j = 0; j < n; ++j)
    if (!ws_accept[c0 + j]) { a = j; break; }
  accepted_len[i] = a;
  for (int j = 0; j < a; ++j) o[j] = draft_ids[c0 - i + j];
  o[a] = ws_cand[c0 + a];
  for (int j = a + 1; j <= k_max; ++j) o[j] = -1;
}

template <typename T, int NT, bool BULK>
void* rows_fn() {
  return reinterpret_cast<void*>(&rows_kernel<T, NT, BULK>);
}

// All instantiations: (fp32, bf16) x (bulk, staged) x (256, 512 threads).
void* const* kernel_table() {
  static void* const t[8] = {rows_fn<float, 256, true>(),    rows_fn<float, 256, false>(),
                             rows_fn<uint16_t, 256, true>(), rows_fn<uint16_t, 256, false>(),
                             rows_fn<float, 512, true>(),    rows_fn<float, 512, false>(),
                             rows_fn<uint16_t, 512, true>(), rows_fn<uint16_t, 512, false>()};
  return t;
}

void* pick_rows_kernel(int elem, bool bulk, int threads) {
  const int idx = (threads == 512 ? 4 : 0) + (elem == 4 ? 0 : 2) + (bulk ? 0 : 1);
  return kernel_table()[idx];
}

// stage meta (4 x 16 B) + mbarriers (4 x 8 B) + cu_seqlens + temperatures
size_t meta_bytes(int bs) {
  return 64 + 32 + static_cast<size_t>(bs + 1) * 4 + static_cast<size_t>(bs) * 4;
}

// Dynamic shared memory a kernel may use on the current device: the opt-in
// per-block maximum minus the kernel's static shared memory.
cudaError_t kernel_smem(void* fn, int* dyn_limit, int* static_bytes) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  *static_bytes = static_cast<int>(fa.sharedSizeBytes);
  *dyn_limit = optin - *static_bytes;
  return cudaSuccess;
}

// Raises the kernel's dynamic shared-memory limit to the device maximum and
// allows 16-CTA clusters, once per (kernel, device); later calls are
// lock-free reads, so launches stay cheap and capturable.
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
      int st = 0;
      e = kernel_smem(fn, &lim, &st);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      limit_of[slot][dev].store(lim, std::memory_order_release);
    }
  }
  return smem <= static_cast<size_t>(lim) ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t choose_verify_shape(int V, int elem, int bs, const sd_launch_cfg* req, bool bulk,
                                VerifyShape* out, bool* fits) {
  *fits = false;
  int dev = 0, sm_smem = 0, reserved = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  if (e != cudaSuccess) return e;
  const int creq = req ? req->cluster : 0;
  const int sreq = req ? req->stages : 0;
  const int treq = req ? req->threads : 0;
  if (creq && creq != 1 && creq != 2 && creq != 4 && creq != 8 && creq != 16) return cudaSuccess;
  if (sreq < 0 || sreq > 4) return cudaSuccess;
  if (treq && treq != 256 && treq != 512) return cudaSuccess;
  const size_t meta = meta_bytes(bs);
  // Preference: two 256-thread CTAs per SM with three stages each (barrier
  // waits of one CTA hidden by the other), then one 512-thread CTA per SM.
  struct Cand { int threads, stages, per_sm; };
  const Cand cands[] = {{256, 3, 2}, {512, 3, 1}, {512, 2, 1}, {256, 2, 2}, {512, 1, 1}};
  for (const Cand& c : cands) {
    const int threads = treq ? treq : c.threads;
    const int S = bulk ? (sreq ? sreq : c.stages) : 1;
    const int per_sm = treq || sreq ? 1 : c.per_sm;
    void* fn = pick_rows_kernel(elem, bulk, threads);
    e = prepare(fn, 0);
    if (e != cudaSuccess) return e;
    int dyn_limit = 0, st = 0;
    e = kernel_smem(fn, &dyn_limit, &st);
    if (e != cudaSuccess) return e;
    long long budget = per_sm == 1 ? dyn_limit
                                   : std::min<long long>(dyn_limit, sm_smem / per_sm - reserved - st);
    for (int C = 1; C <= 16; C <<= 1) {
      if (creq && C != creq) continue;
      int SL = (V + C - 1) / C;
      SL = (SL + 63) / 64 * 64;
      const size_t stage = 2 * static_cast<size_t>(SL) * elem;
      const size_t smem = static_cast<size_t>(S) * stage + meta;
      if (static_cast<long long>(smem) <= budget) {
        out->C = C;
        out->S = S;
        out->SL = SL;
        out->threads = threads;
        out->smem = smem;
        out->bulk = bulk;
        out->clusters = req ? req->clusters : 0;
        *fits = true;
        return cudaSuccess;
      }
    }
  }
  return cudaSuccess;
}

cudaError_t max_active_clusters(int elem, const VerifyShape& shape, int* n) {
  void* fn = pick_rows_kernel(elem, shape.bulk, shape.threads);
  cudaError_t e = prepare(fn, shape.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = shape.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(shape.C, 1, 1);
  cfg.blockDim = dim3(shape.threads, 1, 1);
  cfg.dynamicSmemBytes = shape.smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, fn, &cfg);
}

cudaError_t launch_verify_rows(const VerifyParams& p, int elem, const VerifyShape& shape,
                               cudaStream_t s) {
  void* fn = pick_rows_kernel(elem, shape.bulk, shape.threads);
  cudaError_t e = prepare(fn, shape.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = shape.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(shape.clusters * shape.C, 1, 1);
  cfg.blockDim = dim3(shape.threads, 1, 1);
  cfg.dynamicSmemBytes = shape.smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<VerifyParams*>(&p)};
  e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_verify_finalize(const int* draft_ids, const int* cu, int bs, int k_max,
                                   int* accepted_len, int* out_tokens, int* err,
                                   const uint8_t* ws_accept, const int* ws_cand,
                                   const int* ws_status, cudaStream_t s) {
  const int threads = 128;
  const int blocks = (bs + threads - 1) / threads;
  finalize_kernel<<<blocks, threads, 0, s>>>(draft_ids, cu, bs, k_max, accepted_len, out_tokens,
                                             err, ws_accept, ws_cand, ws_status);
  return cudaGetLastError();
}

}  // namespace sdk
