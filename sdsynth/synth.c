/* synth.c -- seeded synthetic inputs for the verification step.
 *
 * Shared by the tests, the bench and the smoke check.  It holds none of the
 * method's arithmetic (no softmax, no acceptance test, no sampling from a
 * residual): it only draws random numbers and writes them in the layouts the
 * step consumes.
 *
 * Every value is a pure function of (seed, stream, step, request i, position
 * j, element k), drawn from the SplitMix64 generator of Steele, Lea and
 * Flood ("Fast splittable pseudorandom number generators", OOPSLA 2014):
 * a 64-bit counter advanced by the golden-ratio increment and passed through
 * its published finaliser.  Values therefore do not depend on the thread
 * count or on which rows are generated together.
 *
 *   uniforms        u = (h >> 40) * 2^-24, in [0, 1) with 24 bits
 *   normals         Box-Muller on the two 32-bit halves of one draw
 *   draft ids       Gumbel-max: argmax_k (d_k / tau + G_k), G_k = -log(-log U_k),
 *                   which draws k with probability softmax(d / tau)_k
 *                   (Gumbel 1954; the "Gumbel-max trick"); tau = 0 takes argmax d
 *
 * Built with -ffp-contract=off so that x86 and Arm hosts produce the same bytes
 * wherever the C library's log/sin/cos agree.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYN_F32 0
#define SYN_BF16 1

static const uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Row key of (seed, stream, step, i, j). */
static inline uint64_t row_key(uint64_t seed, uint64_t stream, uint64_t step, uint64_t i,
                               uint64_t j) {
  uint64_t h = mix64(seed + kGamma);
  h = mix64(h ^ (stream * kGamma + 1));
  h = mix64(h ^ (step * kGamma + 2));
  h = mix64(h ^ (i * kGamma + 3));
  h = mix64(h ^ (j * kGamma + 4));
  return h;
}

static inline uint64_t draw(uint64_t key, uint64_t k) { return mix64(key + (k + 1) * kGamma); }

static inline float u24(uint64_t h) { return (float)(h >> 40) * (1.0f / 16777216.0f); }

/* Two standard normals from one 64-bit draw. */
static inline void normal_pair(uint64_t h, double* z0, double* z1) {
  const double u1 = ((double)(h >> 32) + 0.5) * (1.0 / 4294967296.0); /* (0,1) */
  const double u2 = (double)(h & 0xFFFFFFFFULL) * (1.0 / 4294967296.0);
  const double r = sqrt(-2.0 * log(u1));
  double s, c;
  sincos(6.283185307179586476925286766559 * u2, &s, &c);
  *z0 = r * c;
  *z1 = r * s;
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  b += 0x7FFFu + ((b >> 16) & 1u);
  return (uint16_t)(b >> 16);
}

static inline float bf16_to_f32(uint16_t v) {
  uint32_t b = (uint32_t)v << 16;
  float f;
  memcpy(&f, &b, 4);
  return f;
}

enum { ST_TARGET = 1, ST_DRAFT = 2, ST_GUMBEL = 3 };

typedef struct {
  uint64_t seed;
  uint64_t step;
  int64_t nrows;
  const int32_t* req;
  const int32_t* pos;
  int32_t V;
  int32_t dtype;
  double sigma_t;
  const double* sigma_d; /* per row, or NULL for target rows */
  void* out;
  /* draft-id job */
  const void* rows;
  const float* tau;
  int32_t* ids;
  int64_t r0, r1;
} job_t;

static void logit_rows_range(const job_t* jb) {
  const int V = jb->V;
  const int npair = (V + 1) / 2;
  for (int64_t r = jb->r0; r < jb->r1; ++r) {
    const uint64_t kt = row_key(jb->seed, ST_TARGET, jb->step, (uint64_t)jb->req[r], (uint64_t)jb->pos[r]);
    const uint64_t kd = row_key(jb->seed, ST_DRAFT, jb->step, (uint64_t)jb->req[r], (uint64_t)jb->pos[r]);
    const double sd = jb->sigma_d ? jb->sigma_d[r] : 0.0;
    for (int m = 0; m < npair; ++m) {
      double t0, t1, d0 = 0.0, d1 = 0.0;
      normal_pair(draw(kt, (uint64_t)m), &t0, &t1);
      if (jb->sigma_d) normal_pair(draw(kd, (uint64_t)m), &d0, &d1);
      const double v[2] = {jb->sigma_t * t0 + sd * d0, jb->sigma_t * t1 + sd * d1};
      for (int e = 0; e < 2; ++e) {
        const int k = 2 * m + e;
        if (k >= V) break;
        const size_t idx = (size_t)r * (size_t)V + (size_t)k;
        if (jb->dtype == SYN_F32)
          ((float*)jb->out)[idx] = (float)v[e];
        else
          ((uint16_t*)jb->out)[idx] = f32_to_bf16_rne((float)v[e]);
      }
    }
  }
}

static void draft_ids_range(const job_t* jb) {
  const int V = jb->V;
  for (int64_t r = jb->r0; r < jb->r1; ++r) {
    const float tau = jb->tau[r];
    const uint64_t kg = row_key(jb->seed, ST_GUMBEL, jb->step, (uint64_t)jb->req[r], (uint64_t)jb->pos[r]);
    int best = 0;
    double bv = -INFINITY;
    for (int k = 0; k < V; ++k) {
      const size_t idx = (size_t)r * (size_t)V + (size_t)k;
      double d = jb->dtype == SYN_F32 ? (double)((const float*)jb->rows)[idx]
                                      : (double)bf16_to_f32(((const uint16_t*)jb->rows)[idx]);
      double score = d;
      if (tau > 0.0f) {
        const double u = ((double)(draw(kg, (uint64_t)k) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
        score = d / (double)tau - log(-log(u));
      }
      if (score > bv) {
        bv = score;
        best = k;
      }
    }
    jb->ids[r] = best;
  }
}

static void* logit_thread(void* p) {
  logit_rows_range((const job_t*)p);
  return NULL;
}
static void* ids_thread(void* p) {
  draft_ids_range((const job_t*)p);
  return NULL;
}

static void run_parallel(job_t* base, int nthreads, void* (*fn)(void*)) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > base->nrows) nthreads = (int)(base->nrows > 0 ? base->nrows : 1);
  job_t jobs[256];
  pthread_t th[256];
  int started[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = *base;
    jobs[t].r0 = base->nrows * t / nthreads;
    jobs[t].r1 = base->nrows * (t + 1) / nthreads;
    started[t] = (t > 0) && pthread_create(&th[t], NULL, fn, &jobs[t]) == 0;
  }
  fn(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) {
    if (started[t])
      pthread_join(th[t], NULL);
    else
      fn(&jobs[t]);
  }
}

/* Logit rows: row r belongs to (req[r], pos[r]); element k of a target row is
 * sigma_t * N_target(k); of a draft row (sigma_d != NULL) it is
 * sigma_t * N_target(k) + sigma_d[r] * N_draft(k), i.e. the target row of the
 * same (i, j) plus independent noise.  out: [nrows, V] fp32 or bf16 bits. */
int synth_logit_rows(uint64_t seed, uint64_t step, int64_t nrows, const int32_t* req,
                     const int32_t* pos, int32_t V, int32_t dtype, double sigma_t,
                     const double* sigma_d, void* out, int nthreads) {
  if (nrows < 0 || V < 1 || (dtype != SYN_F32 && dtype != SYN_BF16) || (nrows > 0 && (!req || !pos || !out)))
    return -1;
  job_t jb;
  memset(&jb, 0, sizeof jb);
  jb.seed = seed;
  jb.step = step;
  jb.nrows = nrows;
  jb.req = req;
  jb.pos = pos;
  jb.V = V;
  jb.dtype = dtype;
  jb.sigma_t = sigma_t;
  jb.sigma_d = sigma_d;
  jb.out = out;
  if (nrows > 0) run_parallel(&jb, nthreads, logit_thread);
  return 0;
}

/* Draft token of each draft row, drawn from softmax(row / tau[r]) by the
 * Gumbel-max trick, or argmax(row) when tau[r] == 0 (lowest index on ties). */
int synth_draft_ids(uint64_t seed, uint64_t step, int64_t nrows, const int32_t* req,
                    const int32_t* pos, const void* rows, int32_t V, int32_t dtype,
                    const float* tau, int32_t* ids, int nthreads) {
  if (nrows < 0 || V < 1 || (dtype != SYN_F32 && dtype != SYN_BF16) ||
      (nrows > 0 && (!req || !pos || !rows || !tau || !ids)))
    return -1;
  job_t jb;
  memset(&jb, 0, sizeof jb);
  jb.seed = seed;
  jb.step = step;
  jb.nrows = nrows;
  jb.req = req;
  jb.pos = pos;
  jb.rows = rows;
  jb.V = V;
  jb.dtype = dtype;
  jb.tau = tau;
  jb.ids = ids;
  if (nrows > 0) run_parallel(&jb, nthreads, ids_thread);
  return 0;
}

/* One 24-bit uniform per (i[q], j[q]) of the given stream. */
int synth_uniforms(uint64_t seed, uint64_t stream, uint64_t step, int64_t n, const int32_t* i,
                   const int32_t* j, float* out) {
  if (n < 0 || (n > 0 && (!i || !j || !out))) return -1;
  for (int64_t q = 0; q < n; ++q)
    out[q] = u24(draw(row_key(seed, stream, step, (uint64_t)i[q], (uint64_t)j[q]), 0));
  return 0;
}

/* One standard normal per (i[q], j[q]) of the given stream. */
int synth_normals(uint64_t seed, uint64_t stream, uint64_t step, int64_t n, const int32_t* i,
                  const int32_t* j, double* out) {
  if (n < 0 || (n > 0 && (!i || !j || !out))) return -1;
  for (int64_t q = 0; q < n; ++q) {
    double z0, z1;
    normal_pair(draw(row_key(seed, stream, step, (uint64_t)i[q], (uint64_t)j[q]), 0), &z0, &z1);
    out[q] = z0;
  }
  return 0;
}
