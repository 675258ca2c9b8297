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

// Per-CTA values exchanged through distributed shared memory.
struct __align__(16) Slot {
  float a, b;  // pass A: max target / max draft; B: sum target / sum draft; C: residual sum
  float c, d;  // pass B: target / draft logit at the draft token (owner CTA only)
  unsigned long long key;  // pass A greedy: packed (value, -index) maximum
  int flag;    // greedy: row holds NaN; pass B: owns the draft token
  int pad;
};

__device__ __forceinline__ float from_ordered(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// Residual weight max(p - q, 0) of one element pair, with p = e_t / Z_t and
// q = e_d / Z_d; the same expression is used by the sum and by the search.
__device__ __forceinline__ float residual_w(float lt, float ld, float s2, float bt, float bd,
                                            float iZt, float iZd) {
  const float et = exp2_ftz(fmaf(lt, s2, -bt));
  const float ed = exp2_ftz(fmaf(ld, s2, -bd));
  return fmaxf(fmaf(et, iZt, -(ed * iZd)), 0.0f);
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
  __shared__ Slot slots[2][3];
  __shared__ float Wt[NW], Wd[NW], Wr[NW];
  __shared__ unsigned long long Wk[NW];
  __shared__ int Wn[NW];
  __shared__ int meta_x;
  __shared__ float meta_u, meta_ufin;

  cg::cluster_group cluster = cg::this_cluster();
  const int C = p.C;
  const int rank = static_cast<int>(cluster.block_rank());
  const int cid = blockIdx.x / C;
  const int G = gridDim.x / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V;
  const int SL = p.SL;

  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(p.S) * p.stage_bytes);
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
    for (int s = 0; s < p.S; ++s) mbar_init(&mbar[s], 1);
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
  // Producer (thread 0): stage item q's slices into stage s.
  auto issue = [&](int q, int s) {
    int i, j, n;
    locate(q, i, j, n);
    const bool hd = tau_s[i] > 0.0f && j < n;
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
    __syncthreads();
  };

  // Search for the element at which the running sum of weights first exceeds
  // theta, over this CTA's slice of the row.  `cta_inc` (per lane c < C) is
  // the inclusive scan of the CTA totals, `Wsm` the per-warp totals of this
  // CTA; `wfun(v, w)` fills the VE weights of vector v.  Only the CTA and the
  // warp holding the crossing continue to the element level; rounding
  // disagreements between levels fall back to the last positive weight.
  auto owner_search = [&](float theta, float cta_w, float cta_inc, const float* Wsm, int q,
                          auto wfun) {
    const unsigned cross = __ballot_sync(kFull, lane < C && cta_inc > theta);
    int cstar;
    if (cross) {
      cstar = __ffs(cross) - 1;
    } else {
      const unsigned pos = __ballot_sync(kFull, lane < C && cta_w > 0.0f);
      cstar = pos ? 31 - __clz(pos) : 0;
    }
    const float up_c = __shfl_up_sync(kFull, cta_inc, 1);
    const float excl_c = cstar == 0 ? 0.0f : __shfl_sync(kFull, up_c, cstar);
    if (rank != cstar) return;
    const float th_c = fmaxf(theta - excl_c, 0.0f);
    const float ww = lane < NW ? Wsm[lane] : 0.0f;
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
    float run = 0.0f;
    int last_pos = -1;
    for (int base = wb; base < we; base += 32) {
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
    if (lane == 0) p.ws_cand[q] = last_pos >= 0 ? last_pos : lo_e + wb * VE;
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
    const float* urow = p.uniforms + static_cast<size_t>(i) * (p.k_max + 1);

    int x_ld = -1;
    float u_ld = 0.0f, ufin_ld = 0.0f;
    if (tid == 0) {  // issued early, consumed after pass A
      ufin_ld = urow[p.k_max];
      if (!bonus) {
        u_ld = urow[j];
        x_ld = p.draft_ids[q - i];
      }
    }

    // ---------------- pass A: maxima (tau > 0) or argmax (tau = 0)
    if (greedy) {
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
    } else {
      float mt = -INFINITY, md = -INFINITY;
      for (int v = vb + lane; v < ve; v += 32) {
        float f[VE];
        Tr::unpack(vt[v], f);
#pragma unroll
        for (int e = 0; e < VE; ++e) mt = fmaxf(mt, f[e]);
        if (has_draft) {
          Tr::unpack(vd[v], f);
#pragma unroll
          for (int e = 0; e < VE; ++e) md = fmaxf(md, f[e]);
        }
      }
      mt = warp_max(mt);
      md = warp_max(md);
      if (lane == 0) { Wt[warp] = mt; Wd[warp] = md; }
    }
    if (tid == 0) { meta_x = x_ld; meta_u = u_ld; meta_ufin = ufin_ld; }
    __syncthreads();
    if (warp == 0) {
      Slot& sa = slots[par][0];
      if (greedy) {
        unsigned long long kk = warp_max_u64(lane < NW ? Wk[lane] : 0ull);
        const int nn = __any_sync(kFull, lane < NW ? Wn[lane] : 0);
        if (lane == 0) { sa.key = kk; sa.flag = nn; }
      } else {
        const float a = warp_max(lane < NW ? Wt[lane] : -INFINITY);
        const float b = warp_max(lane < NW ? Wd[lane] : -INFINITY);
        if (lane == 0) { sa.a = a; sa.b = b; }
      }
    }
    cluster.sync();
    const Slot* pa = cluster.map_shared_rank(&slots[par][0], lane < C ? lane : 0);
    const int x = meta_x;
    const bool x_ok = !bonus && x >= 0 && x < V;
    const bool lead = (rank == 0 && tid == 0);

    if (greedy) {
      const unsigned long long kk = warp_max_u64(lane < C ? pa->key : 0ull);
      const int nn = __any_sync(kFull, lane < C ? pa->flag : 0);
      const float best = from_ordered(static_cast<uint32_t>(kk >> 32));
      const bool rowbad = nn || kk == 0ull || !isfinite(best);
      const int amax = rowbad ? 0 : static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(kk));
      if (lead) {
        if (rowbad) raise_error(p.err, SD_DEV_ERR_LOGITS);
        if (!bonus && !x_ok) raise_error(p.err, SD_DEV_ERR_DRAFT_ID);
        p.ws_accept[q] = bonus ? 1 : static_cast<uint8_t>(x_ok && !rowbad && x == amax);
        p.ws_cand[q] = amax;
      }
    } else {
      const float Mt = warp_max(lane < C ? pa->a : -INFINITY);
      const float Md = warp_max(lane < C ? pa->b : -INFINITY);
      const float s2 = kLog2e / tau;
      const float bt = Mt * s2;
      const float bd = Md * s2;

      // ---------------- pass B: normalisers
      float zt = 0.0f, zd = 0.0f;
      for (int v = vb + lane; v < ve; v += 32) {
        float f[VE];
        Tr::unpack(vt[v], f);
#pragma unroll
        for (int e = 0; e < VE; ++e) zt += exp2_ftz(fmaf(f[e], s2, -bt));
        if (has_draft) {
          Tr::unpack(vd[v], f);
#pragma unroll
          for (int e = 0; e < VE; ++e) zd += exp2_ftz(fmaf(f[e], s2, -bd));
        }
      }
      zt = warp_sum(zt);
      zd = warp_sum(zd);
      if (lane == 0) { Wt[warp] = zt; Wd[warp] = zd; }
      __syncthreads();
      Slot& sb = slots[par][1];
      if (warp == 0) {
        const float it = warp_inclusive_scan(lane < NW ? Wt[lane] : 0.0f, lane);
        const float id = warp_inclusive_scan(lane < NW ? Wd[lane] : 0.0f, lane);
        if (lane == 31) { sb.a = it; sb.b = id; }
        if (lane == 0) {
          sb.flag = 0;
          if (x_ok && x >= lo_e && x < lo_e + len) {
            sb.c = Tr::at(stage_t(st), x - lo_e);
            sb.d = has_draft ? Tr::at(stage_d(st), x - lo_e) : 0.0f;
            sb.flag = 1;
          }
        }
      }
      cluster.sync();
      const Slot* pb = cluster.map_shared_rank(&slots[par][1], lane < C ? lane : 0);
      const float zt_c = lane < C ? pb->a : 0.0f;
      const float zd_c = lane < C ? pb->b : 0.0f;
      const float zt_inc = warp_inclusive_scan(zt_c, lane);
      const float Zt = __shfl_sync(kFull, zt_inc, 31);
      const float Zd = __shfl_sync(kFull, warp_inclusive_scan(zd_c, lane), 31);
      const int cx = x_ok ? min(x / SL, C - 1) : 0;
      const float ltx = __shfl_sync(kFull, lane < C ? pb->c : 0.0f, cx);
      const float ldx = __shfl_sync(kFull, lane < C ? pb->d : 0.0f, cx);
      const bool rowbad = !isfinite(Mt) || !(isfinite(Zt) && Zt > 0.0f) ||
                          (has_draft && (!isfinite(Md) || !(isfinite(Zd) && Zd > 0.0f)));
      const float ufin = meta_ufin;
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
          acc = (meta_u * qx) <= px;
        }
        need_residual = !acc && !rowbad;
        if (lead) {
          if (rowbad) raise_error(p.err, SD_DEV_ERR_LOGITS);
          if (!x_ok) raise_error(p.err, SD_DEV_ERR_DRAFT_ID);
          if (!(meta_u >= 0.0f && meta_u < 1.0f)) raise_error(p.err, SD_DEV_ERR_UNIFORM);
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
        // ---------------- pass C: residual mass max(p - q, 0)
        const float iZt = 1.0f / Zt, iZd = 1.0f / Zd;
        float sr = 0.0f;
        for (int v = vb + lane; v < ve; v += 32) {
          float f[VE], g[VE];
          Tr::unpack(vt[v], f);
          Tr::unpack(vd[v], g);
#pragma unroll
          for (int e = 0; e < VE; ++e) sr += residual_w(f[e], g[e], s2, bt, bd, iZt, iZd);
        }
        sr = warp_sum(sr);
        if (lane == 0) Wr[warp] = sr;
        __syncthreads();
        if (warp == 0) {
          const float ir = warp_inclusive_scan(lane < NW ? Wr[lane] : 0.0f, lane);
          if (lane == 31) slots[par][2].a = ir;
        }
        cluster.sync();
        const Slot* pc = cluster.map_shared_rank(&slots[par][2], lane < C ? lane : 0);
        const float sr_c = lane < C ? pc->a : 0.0f;
        const float sr_inc = warp_inclusive_scan(sr_c, lane);
        const float S = __shfl_sync(kFull, sr_inc, 31);
        if (S > 0.0f && isfinite(S)) {
          owner_search(ufin * S, sr_c, sr_inc, Wr, q, [&](int v, float (&w)[VE]) {
            float f[VE], g[VE];
            Tr::unpack(vt[v], f);
            Tr::unpack(vd[v], g);
#pragma unroll
            for (int e = 0; e < VE; ++e) w[e] = residual_w(f[e], g[e], s2, bt, bd, iZt, iZd);
          });
        } else {
          need_p = true;  // no residual mass in fp32: draw from p instead
        }
      }
      if (need_p) owner_search(ufin * Zt, zt_c, zt_inc, Wt, q, p_weight);
    }
    __syncthreads();  // stage st and the per-warp arrays are free again
    if (BULK && tid == 0 && k + p.S < nitems) issue(cid + (k + p.S) * G, st);
  }
  cluster.sync();  // peers may still read this CTA's slots
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

constexpr int kRowThreads = 512;

template <typename T, bool BULK>
void* rows_fn() {
  return reinterpret_cast<void*>(&rows_kernel<T, kRowThreads, BULK>);
}

void* const* kernel_table() {
  static void* const t[8] = {rows_fn<float, true>(), rows_fn<float, false>(),
                             rows_fn<uint16_t, true>(), rows_fn<uint16_t, false>(),
                             nullptr, nullptr, nullptr, nullptr};
  return t;
}

void* pick_rows_kernel(int elem, bool bulk) {
  if (elem == 4) return bulk ? rows_fn<float, true>() : rows_fn<float, false>();
  return bulk ? rows_fn<uint16_t, true>() : rows_fn<uint16_t, false>();
}

size_t meta_bytes(int bs) { return 4 * 8 + static_cast<size_t>(bs + 1) * 4 + static_cast<size_t>(bs) * 4; }

// Dynamic shared memory a kernel may use on the current device: the opt-in
// per-block maximum minus the kernel's static shared memory.
cudaError_t dyn_smem_limit(void* fn, int* limit) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  *limit = optin - static_cast<int>(fa.sharedSizeBytes);
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
      e = dyn_smem_limit(fn, &lim);
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

cudaError_t rows_smem_limit(int elem, bool bulk, int* limit) {
  void* fn = pick_rows_kernel(elem, bulk);
  cudaError_t e = prepare(fn, 0);
  if (e != cudaSuccess) return e;
  return dyn_smem_limit(fn, limit);
}

bool choose_verify_shape(int V, int elem, int bs, const sd_launch_cfg* req, bool bulk,
                         int dyn_limit, VerifyShape* out) {
  const size_t meta = meta_bytes(bs);
  if (dyn_limit <= 0 || meta >= static_cast<size_t>(dyn_limit)) return false;
  const size_t avail = static_cast<size_t>(dyn_limit) - meta;
  const int creq = req ? req->cluster : 0;
  const int sreq = req ? req->stages : 0;
  if (creq && creq != 1 && creq != 2 && creq != 4 && creq != 8 && creq != 16) return false;
  if (sreq < 0 || sreq > 4) return false;
  auto stage_of = [&](int C) {
    int SL = (V + C - 1) / C;
    SL = (SL + 63) / 64 * 64;
    return std::pair<int, size_t>(SL, 2 * static_cast<size_t>(SL) * elem);
  };
  int C = 0, S = 0, SL = 0;
  size_t stage = 0;
  const int want_s[3] = {3, 2, 1};
  for (int si = 0; si < 3 && !C; ++si) {
    const int s_try = sreq ? sreq : want_s[si];
    for (int c = 1; c <= 16; c <<= 1) {
      if (creq && c != creq) continue;
      auto st = stage_of(c);
      if (static_cast<size_t>(s_try) * st.second <= avail) {
        C = c; S = s_try; SL = st.first; stage = st.second;
        break;
      }
    }
    if (sreq) break;
  }
  if (!C) return false;
  out->C = C;
  out->S = bulk ? S : 1;
  out->SL = SL;
  out->threads = kRowThreads;
  out->smem = static_cast<size_t>(out->S) * stage + meta;
  out->bulk = bulk;
  out->clusters = req ? req->clusters : 0;
  return true;
}

cudaError_t max_active_clusters(int elem, const VerifyShape& shape, int* n) {
  void* fn = pick_rows_kernel(elem, shape.bulk);
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
  void* fn = pick_rows_kernel(elem, shape.bulk);
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
