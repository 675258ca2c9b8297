// sd_oracle.cpp -- TEST INFRASTRUCTURE, not product code.
//
// A plain, slow, sequential CPU restatement of one verification step of
// speculative decoding with adaptive verification, written from the pages'
// descriptions in fp64.  It is the yardstick the CUDA path is compared
// against.  Only the tests, the smoke check and the bench's CPU-baseline leg
// may load this library; the product path never does.
//
// It shares no code, header, table or helper with the CUDA library.  Every
// step follows the plain definition in the pages' order:
//
//   planning  (adaptive verification):
//     [fosworld blog "추측 디코딩과 vLLM 적응형 검증", section "동작", steps 1-3]
//     uniform-K mode: [discuss.pytorch.kr "DSD feat. Cohere", section
//      "동적 추측 디코딩(DSD)의 핵심 아이디어": one draft length K for the
//      whole batch, chosen to maximise goodput = AL / ITL]
//     [agentlenshq "vLLM DSpark을 활용한 적응형 검증", section
//      "DSpark 신뢰도 스케줄링 메커니즘": Global Top-B Selection,
//      Budget Calculation, Execution Pipeline]
//     [same page, section "기술적 구현 및 CUDA Graphs": Cost Modeling,
//      CUDA Graph Padding, Graph Capture]
//   sampling  (speculative rejection sampling, the rule of the original
//     papers the fosworld blog cites under "참고 링크 / 논문"; the blog's
//     "추측 디코딩이란" gives its greedy form and "속도, 메모리, 정확도에 주는
//     영향" (row 정확도) states that it preserves the target distribution).
//
// Readings adopted where the pages are silent (labelled O1..O24 below):
//   O1  acceptance estimate a = sigmoid(confidence logit)
//   O2  survival = running product in position order, fp64, rounded to fp32
//       to form the ranking key (the precision the kernel ranks in)
//   O3  ties in the global ranking broken by packed slot index (ascending)
//   O4  R = number of requests (one bonus/correction token each)
//   O6  B in [0, min(N, cost_len-1-T)], ties in the objective -> smallest B
//   O7  cost forced monotone: cost'[n] = max(cost[1..n]); cost[0] unused
//   O10 optional previous-step confidences size the budget, current ones
//       assign the slots (adaptive mode only)
//   O24 uniform K: AL(K) = R + sum_i sum_{j < min(K, K_i)} s_{i,j} (the same
//       survival estimates), ITL(K) = cost'[T + sum_i min(K, K_i)]; K ranges
//       over 0..max_i K_i with T + tokens <= cost_len-1; ties -> smallest K
//   O11 p = softmax(target/tau), q = softmax(draft/tau), same tau; tau = 0
//       is greedy
//   O12 uniforms[i][j] (j < k_max) test slot j, uniforms[i][k_max] is the
//       final draw
//   O13 accept iff u*q(x) <= p(x); taken in fp32 on correctly rounded p, q
//   O14 inverse CDF: smallest k (vocab order) with C_k > u*S
//   O15 residual mass S <= 0 or non-finite -> sample from p with the same u
//   O16 argmax ties -> lowest index
//   O17 draft rows of greedy requests are never read
//   O25 online calibration: per position j a logistic model
//       a = sigmoid(w_j * c + b_j) of the confidence logit c, moved by one
//       gradient step on the mean logistic loss of the step's observed slots
//       (those up to and including the first rejection)
//
// Near-boundary flags: decisions within 1e-5 relative of their boundary are
// reported so that a test can tell an fp32 rounding disagreement from a bug.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

constexpr double kNearRel = 1e-5;

enum { ORC_OK = 0, ORC_ERR_ARG = -1, ORC_ERR_DATA = -5 };
enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_MODE_ADAPTIVE = 0, ORC_MODE_ALL_SLOTS = 1, ORC_MODE_UNIFORM_K = 2 };

// Near flags of the plan.
enum { NEAR_TOPB = 1, NEAR_BUDGET = 2 };
// Near flags of one request's verification.
enum { NEAR_ACCEPT = 1, NEAR_CDF = 2, DEGENERATE_RESIDUAL = 4 };

// Decode one stored logit exactly.  bf16 is the upper half of an IEEE
// binary32, so widening is a 16-bit shift.
double load_logit(const void* base, int dtype, size_t idx) {
  if (dtype == ORC_F32) return static_cast<double>(static_cast<const float*>(base)[idx]);
  uint32_t bits = static_cast<uint32_t>(static_cast<const uint16_t*>(base)[idx]) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return static_cast<double>(f);
}

// Acceptance estimate from a confidence logit: the "small logistic model"
// of the fosworld blog's table under "동작" (reading O1).
double sigmoid(double c) { return 1.0 / (1.0 + std::exp(-c)); }

// Survival of every packed slot: s_{i,j} = prod_{m<=j} a_{i,m}, multiplied
// front to back ("동작" step 1).
void survival(const float* conf, const int* draft_lens, int bs, std::vector<double>& s) {
  size_t off = 0;
  for (int i = 0; i < bs; ++i) {
    double run = 1.0;
    for (int j = 0; j < draft_lens[i]; ++j) {
      run *= sigmoid(static_cast<double>(conf[off + j]));
      s.push_back(run);
    }
    off += static_cast<size_t>(draft_lens[i]);
  }
}

// Global ranking of all slots ("동작" step 2 / Global Top-B Selection):
// by survival key descending, ties by packed slot index ascending (O3).
std::vector<int> rank_order(const std::vector<float>& key) {
  std::vector<int> order(key.size());
  for (size_t q = 0; q < key.size(); ++q) order[q] = static_cast<int>(q);
  std::sort(order.begin(), order.end(), [&](int a, int b) {
    if (key[a] != key[b]) return key[a] > key[b];
    return a < b;
  });
  return order;
}

struct BudgetResult {
  int B = 0;
  int near = 0;
};

// Budget choice ("동작" step 3 / Budget Calculation): maximise expected
// tokens (R bonus tokens plus the survival of the B best slots) per unit of
// step cost cost'[T+B].  Ties go to the smallest B (O6).
BudgetResult budget_argmax(const std::vector<float>& key, const std::vector<int>& order, int R,
                           int T, const std::vector<double>& cost_mono, int cost_len,
                           double* obj_out) {
  const int N = static_cast<int>(key.size());
  const int L = cost_len - 1;
  const int Bmax = std::min(N, L - T);
  std::vector<double> obj(static_cast<size_t>(Bmax) + 1);
  double E = static_cast<double>(R);
  obj[0] = E / cost_mono[static_cast<size_t>(T)];
  for (int B = 1; B <= Bmax; ++B) {
    E += static_cast<double>(key[static_cast<size_t>(order[static_cast<size_t>(B - 1)])]);
    obj[static_cast<size_t>(B)] = E / cost_mono[static_cast<size_t>(T + B)];
  }
  BudgetResult r;
  double best = obj[0];
  for (int B = 1; B <= Bmax; ++B)
    if (obj[static_cast<size_t>(B)] > best) { best = obj[static_cast<size_t>(B)]; r.B = B; }
  double runner = -std::numeric_limits<double>::infinity();
  for (int B = 0; B <= Bmax; ++B)
    if (B != r.B) runner = std::max(runner, obj[static_cast<size_t>(B)]);
  if (Bmax >= 1 && best - runner <= kNearRel * std::fabs(best)) r.near |= NEAR_BUDGET;
  if (obj_out)
    for (int B = 0; B <= Bmax; ++B) obj_out[B] = obj[static_cast<size_t>(B)];
  return r;
}

// Uniform draft length (DSD, O24): every request verifies the first
// min(K, K_i) slots of its draft.  For each K, AL(K) is R plus the survival
// of those slots and ITL(K) the monotone cost of the step's T + (their
// number) tokens; the smallest K with the largest AL / ITL wins.  obj_out
// [max_i K_i + 1] receives the objective per K (NaN where the cost table is
// too short).
BudgetResult uniform_argmax(const std::vector<float>& key, const int* draft_lens, int bs, int T,
                            const std::vector<double>& cost_mono, int cost_len, double* obj_out) {
  const int L = cost_len - 1;
  int Kcap = 0;
  for (int i = 0; i < bs; ++i) Kcap = std::max(Kcap, draft_lens[i]);
  std::vector<double> obj(static_cast<size_t>(Kcap) + 1,
                          std::numeric_limits<double>::quiet_NaN());
  for (int K = 0; K <= Kcap; ++K) {
    double E = static_cast<double>(bs);
    int tokens = 0;
    size_t off = 0;
    for (int i = 0; i < bs; ++i) {
      const int n = std::min(K, draft_lens[i]);
      for (int j = 0; j < n; ++j) E += static_cast<double>(key[off + static_cast<size_t>(j)]);
      tokens += n;
      off += static_cast<size_t>(draft_lens[i]);
    }
    if (T + tokens > L) break;  // tokens grow with K: no larger K fits either
    obj[static_cast<size_t>(K)] = E / cost_mono[static_cast<size_t>(T + tokens)];
  }
  BudgetResult r;
  double best = obj[0];
  for (int K = 1; K <= Kcap; ++K)
    if (obj[static_cast<size_t>(K)] > best) { best = obj[static_cast<size_t>(K)]; r.B = K; }
  double runner = -std::numeric_limits<double>::infinity();
  for (int K = 0; K <= Kcap; ++K)
    if (K != r.B && !std::isnan(obj[static_cast<size_t>(K)]))
      runner = std::max(runner, obj[static_cast<size_t>(K)]);
  if (best - runner <= kNearRel * std::fabs(best)) r.near |= NEAR_BUDGET;
  if (obj_out)
    for (int K = 0; K <= Kcap; ++K) obj_out[K] = obj[static_cast<size_t>(K)];
  return r;
}

// Two-pass textbook softmax in fp64 at temperature tau (> 0).
void softmax_row(const void* base, int dtype, size_t row, int V, double tau, std::vector<double>& p) {
  p.resize(static_cast<size_t>(V));
  double m = -std::numeric_limits<double>::infinity();
  for (int k = 0; k < V; ++k) {
    p[k] = load_logit(base, dtype, row * V + k) / tau;
    m = std::max(m, p[k]);
  }
  double Z = 0.0;
  for (int k = 0; k < V; ++k) {
    p[k] = std::exp(p[k] - m);
    Z += p[k];
  }
  for (int k = 0; k < V; ++k) p[k] /= Z;
}

// Lowest index of the largest raw logit (greedy, O16).
int argmax_row(const void* base, int dtype, size_t row, int V) {
  int best = 0;
  double bv = load_logit(base, dtype, row * V);
  for (int k = 1; k < V; ++k) {
    double v = load_logit(base, dtype, row * V + k);
    if (v > bv) { bv = v; best = k; }
  }
  return best;
}

// A usable logit row holds finite values or -inf (a masked token, p = 0) and
// at least one finite value; NaN and +inf are errors.
bool row_finite(const void* base, int dtype, size_t row, int V) {
  bool any_finite = false;
  for (int k = 0; k < V; ++k) {
    const double v = load_logit(base, dtype, row * V + k);
    if (std::isnan(v) || v == std::numeric_limits<double>::infinity()) return false;
    any_finite = any_finite || std::isfinite(v);
  }
  return any_finite;
}

// Inverse-CDF draw over non-negative weights w (O14): smallest k whose
// running sum exceeds u*S.  Sets *near when some running sum lies within
// 1e-5*S of the threshold.
int inverse_cdf(const std::vector<double>& w, double u, bool* near) {
  double S = 0.0;
  for (double x : w) S += x;
  const double theta = u * S;
  double C = 0.0;
  int pick = -1;
  *near = false;
  for (size_t k = 0; k < w.size(); ++k) {
    C += w[k];
    if (std::fabs(C - theta) <= kNearRel * S) *near = true;
    if (pick < 0 && C > theta) pick = static_cast<int>(k);
  }
  if (pick < 0) {  // u*S == S can only arise from rounding; take the last positive weight
    for (size_t k = w.size(); k-- > 0;)
      if (w[k] > 0.0) { pick = static_cast<int>(k); break; }
    *near = true;
  }
  return pick;
}

}  // namespace

extern "C" {

int oracle_abi_version(void) { return 1; }

// Survival probabilities of the packed slots, in fp64.
int oracle_survival(const float* conf, const int* draft_lens, int bs, double* s_out) {
  if (!conf || !draft_lens || !s_out || bs < 0) return ORC_ERR_ARG;
  std::vector<double> s;
  survival(conf, draft_lens, bs, s);
  std::copy(s.begin(), s.end(), s_out);
  return ORC_OK;
}

// One planning stage.
//   conf          [N] packed confidence logits (offsets = exclusive scan of draft_lens)
//   budget_conf   [N'] previous-step confidence logits or NULL (O10)
//   cost          [cost_len] step cost by token count
//   outputs: *B_out, slot_mask [bs*k_max] (slot (i,j) at i*k_max+j),
//            num_verified [bs], cu_seqlens [bs+1] (n_i + 1 query rows each)
//   obj_out       [min(N, cost_len-1-T)+1] objective per B of the budget set, or NULL
//   near_out      NEAR_TOPB | NEAR_BUDGET
int oracle_plan(const float* conf, const int* draft_lens, int bs, int k_max,
                const float* budget_conf, const int* budget_draft_lens, int bs_budget,
                const float* cost, int cost_len, int T, int mode,
                int* B_out, uint8_t* slot_mask, int* num_verified, int* cu_seqlens,
                double* obj_out, int* near_out) {
  if (!draft_lens || !B_out || !slot_mask || !num_verified || !cu_seqlens) return ORC_ERR_ARG;
  if (bs < 1 || k_max < 0) return ORC_ERR_ARG;
  if (mode != ORC_MODE_ADAPTIVE && mode != ORC_MODE_ALL_SLOTS && mode != ORC_MODE_UNIFORM_K)
    return ORC_ERR_ARG;
  for (int i = 0; i < bs; ++i)
    if (draft_lens[i] < 0 || draft_lens[i] > k_max) return ORC_ERR_DATA;
  int N = 0;
  for (int i = 0; i < bs; ++i) N += draft_lens[i];
  std::vector<size_t> offset(static_cast<size_t>(bs) + 1, 0);
  for (int i = 0; i < bs; ++i) offset[i + 1] = offset[i] + static_cast<size_t>(draft_lens[i]);

  std::vector<uint8_t> selected(static_cast<size_t>(N), 0);
  int near = 0;
  int B = N;
  if (mode == ORC_MODE_UNIFORM_K) {
    if (!conf || !cost || T < 1 || cost_len < T + 1) return ORC_ERR_ARG;
    const int L = cost_len - 1;
    std::vector<double> cost_mono(static_cast<size_t>(cost_len), 0.0);
    double run = -std::numeric_limits<double>::infinity();
    for (int n = 1; n < cost_len; ++n) {
      run = std::max(run, static_cast<double>(cost[n]));
      cost_mono[static_cast<size_t>(n)] = run;
    }
    std::vector<double> s;
    survival(conf, draft_lens, bs, s);
    std::vector<float> key(s.size());
    for (size_t q = 0; q < s.size(); ++q) {
      if (!std::isfinite(s[q])) return ORC_ERR_DATA;
      key[q] = static_cast<float>(s[q]);
    }
    // the entries a budget of up to min(N, L-T) slots reads, as in adaptive mode
    for (int n = T; n <= T + std::min(N, L - T); ++n)
      if (!std::isfinite(cost[n]) || !(cost[n] > 0.0f)) return ORC_ERR_DATA;
    BudgetResult kr = uniform_argmax(key, draft_lens, bs, T, cost_mono, cost_len, obj_out);
    near |= kr.near;
    B = 0;
    size_t off = 0;
    for (int i = 0; i < bs; ++i) {
      const int n = std::min(kr.B, draft_lens[i]);
      for (int j = 0; j < n; ++j) selected[off + static_cast<size_t>(j)] = 1;
      B += n;
      off += static_cast<size_t>(draft_lens[i]);
    }
  } else if (mode == ORC_MODE_ADAPTIVE) {
    if (!conf || !cost || T < 1 || cost_len < T + 1) return ORC_ERR_ARG;
    if (budget_conf && (!budget_draft_lens || bs_budget < 1)) return ORC_ERR_ARG;
    const int L = cost_len - 1;
    // Monotone cost (O7).
    std::vector<double> cost_mono(static_cast<size_t>(cost_len), 0.0);
    double run = -std::numeric_limits<double>::infinity();
    for (int n = 1; n < cost_len; ++n) {
      run = std::max(run, static_cast<double>(cost[n]));
      cost_mono[static_cast<size_t>(n)] = run;
    }
    // Current slots: survival, fp32 ranking key, global order.
    std::vector<double> s;
    survival(conf, draft_lens, bs, s);
    std::vector<float> key(s.size());
    for (size_t q = 0; q < s.size(); ++q) {
      if (!std::isfinite(s[q])) return ORC_ERR_DATA;
      key[q] = static_cast<float>(s[q]);
    }
    std::vector<int> order = rank_order(key);

    const int Bmax_cur = std::min(N, L - T);
    for (int n = T; n <= T + Bmax_cur; ++n)
      if (!std::isfinite(cost[n]) || !(cost[n] > 0.0f)) return ORC_ERR_DATA;

    if (budget_conf) {
      for (int i = 0; i < bs_budget; ++i)
        if (budget_draft_lens[i] < 0) return ORC_ERR_DATA;
      std::vector<double> sb;
      survival(budget_conf, budget_draft_lens, bs_budget, sb);
      std::vector<float> keyb(sb.size());
      for (size_t q = 0; q < sb.size(); ++q) {
        if (!std::isfinite(sb[q])) return ORC_ERR_DATA;
        keyb[q] = static_cast<float>(sb[q]);
      }
      const int Bmax_b = std::min(static_cast<int>(keyb.size()), L - T);
      for (int n = T; n <= T + Bmax_b; ++n)
        if (!std::isfinite(cost[n]) || !(cost[n] > 0.0f)) return ORC_ERR_DATA;
      std::vector<int> orderb = rank_order(keyb);
      BudgetResult br = budget_argmax(keyb, orderb, bs, T, cost_mono, cost_len, obj_out);
      near |= br.near;
      B = std::min(br.B, Bmax_cur);
    } else {
      BudgetResult br = budget_argmax(key, order, bs, T, cost_mono, cost_len, obj_out);
      near |= br.near;
      B = br.B;
    }
    for (int r = 0; r < B; ++r) selected[static_cast<size_t>(order[static_cast<size_t>(r)])] = 1;
    if (B > 0 && B < N) {
      const double a = key[static_cast<size_t>(order[static_cast<size_t>(B - 1)])];
      const double b = key[static_cast<size_t>(order[static_cast<size_t>(B)])];
      if (std::fabs(a - b) <= kNearRel * std::max(std::fabs(a), std::fabs(b))) near |= NEAR_TOPB;
    }
  } else {
    std::fill(selected.begin(), selected.end(), 1);
  }

  // Compaction: n_i selected slots of request i form a prefix of its draft;
  // cu_seqlens counts n_i verified drafts plus one target/bonus row each.
  cu_seqlens[0] = 0;
  for (int i = 0; i < bs; ++i) {
    int n = 0;
    for (int j = 0; j < k_max; ++j) {
      uint8_t m = 0;
      if (j < draft_lens[i]) m = selected[offset[i] + static_cast<size_t>(j)];
      slot_mask[static_cast<size_t>(i) * k_max + j] = m;
      n += m;
    }
    num_verified[i] = n;
    cu_seqlens[i + 1] = cu_seqlens[i] + n + 1;
  }
  *B_out = B;
  if (near_out) *near_out = near;
  return ORC_OK;
}

// One sampling stage for the requests listed in req_list (all if NULL).
//   target        [cu_seqlens[bs], V] compacted target logits (row of (i,j): cu_seqlens[i]+j)
//   draft         [cu_seqlens[bs]-bs, V] compacted draft logits (row of (i,j): cu_seqlens[i]-i+j)
//   draft_ids     [cu_seqlens[bs]-bs] compacted like the draft rows
//   uniforms      [bs, k_max+1]
//   temps         [bs]  (0 = greedy)
//   outputs: accepted_len [bs], out_tokens [bs, k_max+1] (-1 padded)
//   px, qx        [cu_seqlens[bs]-bs] p(x_j), q(x_j) per verified slot up to the
//                 first rejection (NaN elsewhere and for greedy), or NULL
//   near_out      [bs] NEAR_ACCEPT | NEAR_CDF | DEGENERATE_RESIDUAL, or NULL
//   decisions_out number of accept tests plus final draws taken, or NULL
int oracle_verify(const void* target, const void* draft, int dtype, int V,
                  const int* draft_ids, const float* uniforms, const float* temps,
                  const int* cu_seqlens, int bs, int k_max,
                  const int* req_list, int n_req,
                  int* accepted_len, int* out_tokens,
                  double* px, double* qx, int* near_out, long long* decisions_out) {
  if (!target || !draft_ids || !uniforms || !temps || !cu_seqlens || !accepted_len || !out_tokens)
    return ORC_ERR_ARG;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_ERR_ARG;
  if (V < 1 || bs < 1 || k_max < 0) return ORC_ERR_ARG;
  if (cu_seqlens[0] != 0) return ORC_ERR_DATA;
  for (int i = 0; i < bs; ++i) {
    const int rows = cu_seqlens[i + 1] - cu_seqlens[i];
    if (rows < 1 || rows > k_max + 1) return ORC_ERR_DATA;
  }
  const int count = req_list ? n_req : bs;
  long long decisions = 0;
  std::vector<double> p, q, w;
  for (int t = 0; t < count; ++t) {
    const int i = req_list ? req_list[t] : t;
    if (i < 0 || i >= bs) return ORC_ERR_ARG;
    const int n = cu_seqlens[i + 1] - cu_seqlens[i] - 1;
    const size_t trow0 = static_cast<size_t>(cu_seqlens[i]);
    const size_t drow0 = static_cast<size_t>(cu_seqlens[i] - i);
    const double tau = static_cast<double>(temps[i]);
    const float* u = uniforms + static_cast<size_t>(i) * (k_max + 1);
    int* out = out_tokens + static_cast<size_t>(i) * (k_max + 1);
    int near = 0;
    if (!(tau >= 0.0) || !std::isfinite(tau)) return ORC_ERR_DATA;
    for (int j = 0; j <= k_max; ++j)
      if (!(u[j] >= 0.0f && u[j] < 1.0f)) return ORC_ERR_DATA;
    for (int j = 0; j < n; ++j)
      if (draft_ids[drow0 + j] < 0 || draft_ids[drow0 + j] >= V) return ORC_ERR_DATA;
    if (px) for (int j = 0; j < n; ++j) px[drow0 + j] = std::nan("");
    if (qx) for (int j = 0; j < n; ++j) qx[drow0 + j] = std::nan("");

    // Accept drafts front to back until the first rejection.
    int a = n;
    for (int j = 0; j < n; ++j) {
      const int x = draft_ids[drow0 + j];
      if (!row_finite(target, dtype, trow0 + j, V)) return ORC_ERR_DATA;
      ++decisions;
      bool accept;
      if (tau == 0.0) {
        accept = (x == argmax_row(target, dtype, trow0 + j, V));
      } else {
        if (!draft || !row_finite(draft, dtype, drow0 + j, V)) return ORC_ERR_DATA;
        softmax_row(target, dtype, trow0 + j, V, tau, p);
        softmax_row(draft, dtype, drow0 + j, V, tau, q);
        if (px) px[drow0 + j] = p[x];
        if (qx) qx[drow0 + j] = q[x];
        // O13: the comparison is taken in fp32 on correctly rounded operands.
        const float pf = static_cast<float>(p[x]);
        const float qf = static_cast<float>(q[x]);
        const float lhs = static_cast<float>(static_cast<double>(u[j]) * static_cast<double>(qf));
        accept = (lhs <= pf);
        const double exact_lhs = static_cast<double>(u[j]) * q[x];
        if (std::fabs(exact_lhs - p[x]) <= kNearRel * std::max(p[x], exact_lhs)) near |= NEAR_ACCEPT;
      }
      if (!accept) { a = j; break; }
    }

    // Final token from row a: residual at a rejection, bonus from p otherwise.
    if (!row_finite(target, dtype, trow0 + a, V)) return ORC_ERR_DATA;
    ++decisions;
    int y;
    if (tau == 0.0) {
      y = argmax_row(target, dtype, trow0 + a, V);
    } else {
      softmax_row(target, dtype, trow0 + a, V, tau, p);
      w.assign(p.begin(), p.end());
      if (a < n) {
        softmax_row(draft, dtype, drow0 + a, V, tau, q);
        double S = 0.0;
        for (int k = 0; k < V; ++k) {
          w[k] = std::max(p[k] - q[k], 0.0);
          S += w[k];
        }
        if (!(S > 0.0) || !std::isfinite(S)) {  // O15
          w.assign(p.begin(), p.end());
          near |= DEGENERATE_RESIDUAL;
        }
      }
      bool cdf_near = false;
      y = inverse_cdf(w, static_cast<double>(u[k_max]), &cdf_near);
      if (cdf_near) near |= NEAR_CDF;
    }

    accepted_len[i] = a;
    for (int j = 0; j <= k_max; ++j) out[j] = -1;
    for (int j = 0; j < a; ++j) out[j] = draft_ids[drow0 + j];
    out[a] = y;
    if (near_out) near_out[i] = near;
  }
  if (decisions_out) *decisions_out = decisions;
  return ORC_OK;
}

// Row statistics of one logit row, for pinning the softmax step on its own:
// returns p(k) for every k at temperature tau (> 0) into p_out [V].
int oracle_softmax(const void* row, int dtype, int V, double tau, double* p_out) {
  if (!row || !p_out || V < 1 || !(tau > 0.0)) return ORC_ERR_ARG;
  std::vector<double> p;
  softmax_row(row, dtype, 0, V, tau, p);
  std::copy(p.begin(), p.end(), p_out);
  return ORC_OK;
}

// Online calibration of the acceptance estimate (fosworld blog, the table
// under "동작": for model-based drafts a small logistic model predicts
// acceptance from the draft's logits and is corrected continuously with the
// verification outcomes; reading O25).  Slot (i, j) of the packed conf
// (offsets = exclusive scan of draft_lens) is observed when
// j < num_verified[i] and j <= accepted_len[i]: it was accepted (y = 1) when
// j < accepted_len[i], and it is the first rejection (y = 0) at
// j = accepted_len[i].  Later slots were never tested.  With m_j observed
// slots at position j, z = w_j * c + b_j and e = sigmoid(z) - y:
//   grad_w[j] = (1/m_j) sum e * c,  grad_b[j] = (1/m_j) sum e
// (the gradient of the mean of -[y log a + (1-y) log(1-a)]), and
//   w_j -= lr * grad_w[j],  b_j -= lr * grad_b[j]   (positions with m_j = 0
// keep their parameters; their gradient is reported as 0).
//   w, b      [k_max] in/out;  grad_w, grad_b [k_max] out (or NULL);
//   count     [k_max] out m_j (or NULL).
int oracle_calibrate(const float* conf, const int* draft_lens, const int* num_verified,
                     const int* accepted_len, int bs, int k_max, double lr, double* w,
                     double* b, double* grad_w, double* grad_b, int* count) {
  if (!draft_lens || !num_verified || !accepted_len || !w || !b) return ORC_ERR_ARG;
  if (bs < 1 || k_max < 0 || !std::isfinite(lr) || lr < 0.0) return ORC_ERR_ARG;
  size_t N = 0;
  for (int i = 0; i < bs; ++i) {
    if (draft_lens[i] < 0 || draft_lens[i] > k_max) return ORC_ERR_DATA;
    if (num_verified[i] < 0 || num_verified[i] > draft_lens[i]) return ORC_ERR_DATA;
    if (accepted_len[i] < 0 || accepted_len[i] > num_verified[i]) return ORC_ERR_DATA;
    N += static_cast<size_t>(draft_lens[i]);
  }
  if (N > 0 && !conf) return ORC_ERR_ARG;
  std::vector<double> ge(static_cast<size_t>(k_max), 0.0), gc(static_cast<size_t>(k_max), 0.0);
  std::vector<int> m(static_cast<size_t>(k_max), 0);
  size_t off = 0;
  for (int i = 0; i < bs; ++i) {
    const int observed = std::min(num_verified[i], accepted_len[i] + 1);
    for (int j = 0; j < observed; ++j) {
      const double c = static_cast<double>(conf[off + static_cast<size_t>(j)]);
      if (!std::isfinite(c)) return ORC_ERR_DATA;
      const double y = j < accepted_len[i] ? 1.0 : 0.0;
      const double e = sigmoid(w[j] * c + b[j]) - y;
      ge[static_cast<size_t>(j)] += e;
      gc[static_cast<size_t>(j)] += e * c;
      m[static_cast<size_t>(j)] += 1;
    }
    off += static_cast<size_t>(draft_lens[i]);
  }
  for (int j = 0; j < k_max; ++j) {
    const size_t q = static_cast<size_t>(j);
    const double gw = m[q] ? gc[q] / m[q] : 0.0;
    const double gb = m[q] ? ge[q] / m[q] : 0.0;
    w[j] -= lr * gw;
    b[j] -= lr * gb;
    if (grad_w) grad_w[j] = gw;
    if (grad_b) grad_b[j] = gb;
    if (count) count[j] = m[q];
  }
  return ORC_OK;
}

}  // extern "C"
