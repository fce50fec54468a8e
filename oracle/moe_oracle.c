/*
 * moe_oracle.c -- plain fp64 CPU statement of the sparse-MoE block.
 *
 * TEST INFRASTRUCTURE (see moe_oracle.h): not part of the product path.
 * Written for a reader checking it against the pages by eye: one token at a
 * time, one dot product at a time, no blocking, fusion or reordering.
 */
#include "moe_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

int oracle_version(void) { return 1; }

/* ---------------------------------------------------------------- bf16 */

double oracle_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round |v| to a multiple of the bf16 quantum at its binade (2^(e-7) for a
 * normal value in [2^e, 2^(e+1)), 2^-133 below 2^-126), ties to even, then
 * read the bits of the (exactly representable) result. */
uint16_t oracle_f64_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int ex;
  (void)frexp(a, &ex);          /* a = m * 2^ex, m in [0.5, 1) */
  int e = ex - 1;               /* a in [2^e, 2^(e+1)) */
  if (e < -126) e = -126;       /* subnormal range shares the quantum 2^-133 */
  double quantum = ldexp(1.0, e - 7);
  double r = rint(a / quantum) * quantum; /* rint: nearest, ties to even */
  if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
  float f = (float)r;           /* exact: r has <= 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (u >> 16));
}

void oracle_bf16_to_f64_array(int64_t n, const uint16_t *in, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f64(in[i]);
}

void oracle_f64_to_bf16_array(int64_t n, const double *in, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16(in[i]);
}

static double bf(uint16_t b) { return oracle_bf16_to_f64(b); }

/* ------------------------------------------------------------ A1 router */

void oracle_router_logits(int T, int H, int E, const uint16_t *x,
                          const uint16_t *w_router, const uint16_t *w_gate,
                          float *logits, float *gate_logit) {
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int k = 0; k < H; ++k)
        acc += bf(x[(size_t)t * H + k]) * bf(w_router[(size_t)e * H + k]);
      logits[(size_t)t * E + e] = (float)acc;
    }
    if (w_gate && gate_logit) {
      double acc = 0.0;
      for (int k = 0; k < H; ++k)
        acc += bf(x[(size_t)t * H + k]) * bf(w_gate[k]);
      gate_logit[t] = (float)acc;
    }
  }
}

/* --------------------------------------------------------- A2 selection */

typedef struct {
  float v;
  int32_t id;
} ranked;

/* The total order of the selector: a ranks before b when its value is
 * greater, or the values compare equal and its expert id is lower. */
static int ranked_cmp(const void *pa, const void *pb) {
  const ranked *a = (const ranked *)pa, *b = (const ranked *)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->id > b->id) - (a->id < b->id);
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* One token: returns 1 if the row is non-finite (sentinel written). */
static int select_row(int E, int K, const float *row, int32_t *ids,
                      double *weights) {
  for (int e = 0; e < E; ++e) {
    if (!isfinite(row[e])) {
      for (int j = 0; j < K; ++j) {
        ids[j] = -1;
        weights[j] = 0.0;
      }
      return 1;
    }
  }
  ranked *all = (ranked *)malloc(sizeof(ranked) * (size_t)E);
  for (int e = 0; e < E; ++e) {
    all[e].v = row[e];
    all[e].id = e;
  }
  qsort(all, (size_t)E, sizeof(ranked), ranked_cmp);
  /* softmax over the K selected logits, max-subtracted (rank 0 is the max) */
  double zmax = (double)all[0].v, sum = 0.0;
  for (int j = 0; j < K; ++j) {
    ids[j] = all[j].id;
    weights[j] = exp((double)all[j].v - zmax);
    sum += weights[j];
  }
  for (int j = 0; j < K; ++j) weights[j] /= sum;
  free(all);
  return 0;
}

int oracle_select_topk(int T, int E, int K, int ld, const float *logits,
                       const float *gate_logit, int32_t *ids, double *weights,
                       double *sgate) {
  int bad = 0;
  for (int t = 0; t < T; ++t) {
    bad += select_row(E, K, logits + (size_t)t * ld, ids + (size_t)t * K,
                      weights + (size_t)t * K);
    if (sgate) sgate[t] = gate_logit ? sigmoid((double)gate_logit[t]) : 0.0;
  }
  return bad;
}

/* ------------------------------- residual add, RMS norm, weight multiply */

void oracle_add_rmsnorm(int T, int H, const uint16_t *resid_in, const double *block,
                        const uint16_t *gamma, double eps, uint16_t *resid_out,
                        uint16_t *x_next) {
  for (int t = 0; t < T; ++t) {
    const size_t o = (size_t)t * H;
    double ss = 0.0;
    for (int i = 0; i < H; ++i) {
      resid_out[o + i] = oracle_f64_to_bf16(bf(resid_in[o + i]) + block[o + i]);
      const double r = bf(resid_out[o + i]);
      ss += r * r;
    }
    const double inv = 1.0 / sqrt(ss / (double)H + eps);
    for (int i = 0; i < H; ++i)
      x_next[o + i] = oracle_f64_to_bf16(bf(resid_out[o + i]) * inv * bf(gamma[i]));
  }
}

/* ---------------------------------------- candidate lists: exact merge */

int oracle_merge_topk(int T, int n_lists, int K, const int32_t *ids,
                      const float *values, int32_t *ids_out, float *values_out) {
  const int n = n_lists * K;
  int bad = 0;
  ranked *all = (ranked *)malloc(sizeof(ranked) * (size_t)n);
  for (int t = 0; t < T; ++t) {
    const int32_t *ri = ids + (size_t)t * n;
    const float *rv = values + (size_t)t * n;
    int invalid = 0;
    for (int i = 0; i < n; ++i) {
      if (ri[i] < 0) invalid = 1;
      all[i].v = rv[i];
      all[i].id = ri[i];
    }
    if (invalid) {
      for (int j = 0; j < K; ++j) {
        ids_out[(size_t)t * K + j] = -1;
        values_out[(size_t)t * K + j] = 0.0f;
      }
      ++bad;
      continue;
    }
    /* the union sorted under the same total order as the selection */
    qsort(all, (size_t)n, sizeof(ranked), ranked_cmp);
    for (int j = 0; j < K; ++j) {
      ids_out[(size_t)t * K + j] = all[j].id;
      values_out[(size_t)t * K + j] = all[j].v;
    }
  }
  free(all);
  return bad;
}

/* ----------------------------------------------------- A3 expert lists */

void oracle_expert_lists(int T, int E, int K, const int32_t *ids,
                         int32_t *counts, int32_t *offsets, int32_t *perm) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int i = 0; i < T * K; ++i)
    if (ids[i] >= 0 && ids[i] < E) counts[ids[i]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  /* walk experts in order and, inside one expert, entries in (t, j) order */
  int p = 0;
  for (int e = 0; e < E; ++e)
    for (int i = 0; i < T * K; ++i)
      if (ids[i] == e) perm[p++] = i;
}

/* ------------------------------------------- groupwise int8 GEMV (A4/A5) */

void oracle_w8_gemv(int R, int C, int G, const int8_t *q, const uint16_t *s,
                    const uint16_t *v, double *out) {
  const int ng = C / G;
  for (int r = 0; r < R; ++r) {
    double acc = 0.0;
    for (int k = 0; k < C; ++k) {
      double w = (double)q[(size_t)r * C + k] * bf(s[(size_t)r * ng + k / G]);
      acc += w * bf(v[k]);
    }
    out[r] = acc;
  }
}

/* ------------------------------------------------------------ A4 SwiGLU */

void oracle_swiglu(int I, const double *a, double *h_exact, uint16_t *h_bf16) {
  for (int i = 0; i < I; ++i) {
    double g = a[i], u = a[I + i];
    double h = g * sigmoid(g) * u; /* silu(g) * up */
    if (h_exact) h_exact[i] = h;
    if (h_bf16) h_bf16[i] = oracle_f64_to_bf16(h);
  }
}

/* ----------------------------------------------------------- A7 combine */

void oracle_combine(int H, int K, const double *y, const double *w,
                    const double *ys, double sg, double *out,
                    uint16_t *out_bf16) {
  for (int n = 0; n < H; ++n) {
    double acc = 0.0;
    for (int j = 0; j < K; ++j) acc += w[j] * y[(size_t)j * H + n];
    if (ys) acc += sg * ys[n];
    out[n] = acc;
    if (out_bf16) out_bf16[n] = oracle_f64_to_bf16(acc);
  }
}

/* ---------------------------------------------------------- whole block */

typedef struct {
  const oracle_dims *d;
  const oracle_weights *w;
  const uint16_t *x;
  const int32_t *tokens;
  int n_tokens, first, step;
  const float *route_logits, *route_gate;
  uint16_t *out_bf16;
  double *out_f64;
  int32_t *ids;
  double *weights, *sgate;
  float *logits, *gate_logit;
  double *y;
  uint16_t *h;
  int bad;
} block_job;

/* One token through A1..A7. */
static int block_token(const block_job *jb, int t) {
  const oracle_dims *d = jb->d;
  const oracle_weights *w = jb->w;
  const int H = d->H, E = d->E, K = d->K, I = d->I, Is = d->Is, G = d->G;
  const int Imax = I > Is ? I : Is;
  const uint16_t *xt = jb->x + (size_t)t * H;

  /* A1: this token's own fp32 logits and gate logit */
  float *own = (float *)malloc(sizeof(float) * (size_t)E);
  float own_gate = 0.0f;
  oracle_router_logits(1, H, E, xt, w->w_router, Is > 0 ? w->w_gate : NULL,
                       own, &own_gate);
  if (jb->logits) memcpy(jb->logits + (size_t)t * E, own, sizeof(float) * E);
  if (jb->gate_logit) jb->gate_logit[t] = own_gate;

  /* A2: route on the supplied logits if any, else on our own */
  const float *route = jb->route_logits ? jb->route_logits + (size_t)t * E : own;
  float gl = jb->route_gate ? jb->route_gate[t] : own_gate;
  int32_t ids[64];
  double wts[64], sg = 0.0;
  int bad = select_row(E, K, route, ids, wts);
  if (Is > 0) sg = sigmoid((double)gl);
  if (jb->ids) memcpy(jb->ids + (size_t)t * K, ids, sizeof(int32_t) * K);
  if (jb->weights) memcpy(jb->weights + (size_t)t * K, wts, sizeof(double) * K);
  if (jb->sgate) jb->sgate[t] = sg;

  double *a = (double *)malloc(sizeof(double) * 2 * (size_t)Imax);
  uint16_t *hb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)Imax);
  double *y = (double *)calloc((size_t)(K + 1) * H, sizeof(double));
  double *out = (double *)malloc(sizeof(double) * (size_t)H);

  /* A4 + A5 for each routed slot (a non-finite row contributes nothing) */
  for (int j = 0; j < K; ++j) {
    if (ids[j] < 0) {
      if (jb->h) memset(jb->h + ((size_t)t * (K + 1) + j) * Imax, 0,
                        sizeof(uint16_t) * Imax);
      continue;
    }
    size_t e = (size_t)ids[j];
    oracle_w8_gemv(2 * I, H, G, w->w13_q + e * 2 * I * H,
                   w->w13_s + e * 2 * I * (H / G), xt, a);
    oracle_swiglu(I, a, NULL, hb);
    oracle_w8_gemv(H, I, G, w->w2_q + e * (size_t)H * I,
                   w->w2_s + e * (size_t)H * (I / G), hb, y + (size_t)j * H);
    if (jb->h) {
      uint16_t *dst = jb->h + ((size_t)t * (K + 1) + j) * Imax;
      memset(dst, 0, sizeof(uint16_t) * Imax);
      memcpy(dst, hb, sizeof(uint16_t) * I);
    }
  }
  /* A6: shared expert, every token */
  if (Is > 0) {
    oracle_w8_gemv(2 * Is, H, G, w->ws13_q, w->ws13_s, xt, a);
    oracle_swiglu(Is, a, NULL, hb);
    oracle_w8_gemv(H, Is, G, w->ws2_q, w->ws2_s, hb, y + (size_t)K * H);
    if (jb->h) {
      uint16_t *dst = jb->h + ((size_t)t * (K + 1) + K) * Imax;
      memset(dst, 0, sizeof(uint16_t) * Imax);
      memcpy(dst, hb, sizeof(uint16_t) * Is);
    }
  }
  /* A7 */
  for (int j = 0; j < K; ++j)
    if (ids[j] < 0) wts[j] = 0.0;
  oracle_combine(H, K, y, wts, Is > 0 ? y + (size_t)K * H : NULL, sg, out,
                 jb->out_bf16 ? jb->out_bf16 + (size_t)t * H : NULL);
  if (jb->out_f64) memcpy(jb->out_f64 + (size_t)t * H, out, sizeof(double) * H);
  if (jb->y) memcpy(jb->y + (size_t)t * (K + 1) * H, y,
                    sizeof(double) * (size_t)(K + 1) * H);
  free(own); free(a); free(hb); free(y); free(out);
  return bad;
}

static void *block_worker(void *arg) {
  block_job *jb = (block_job *)arg;
  jb->bad = 0;
  for (int i = jb->first; i < jb->n_tokens; i += jb->step) {
    int t = jb->tokens ? jb->tokens[i] : i;
    jb->bad += block_token(jb, t);
  }
  return NULL;
}

int oracle_block_forward(const oracle_dims *d, const oracle_weights *w,
                         const uint16_t *x, const int32_t *tokens,
                         int n_tokens, const float *route_logits,
                         const float *route_gate, uint16_t *out_bf16,
                         double *out_f64, int32_t *ids, double *weights,
                         double *sgate, float *logits, float *gate_logit,
                         double *y, uint16_t *h, int nthreads) {
  if (!d || !w || !x || d->T < 0 || d->H <= 0 || d->E <= 0 || d->K <= 0 ||
      d->K > 64 || d->K > d->E || d->I <= 0 || d->Is < 0 || d->G <= 0 ||
      d->H % d->G || d->I % d->G || (d->Is && d->Is % d->G))
    return -1;
  if (!tokens) n_tokens = d->T;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > n_tokens) nthreads = n_tokens > 0 ? n_tokens : 1;
  block_job *jobs = (block_job *)calloc((size_t)nthreads, sizeof(block_job));
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  for (int i = 0; i < nthreads; ++i) {
    block_job *jb = &jobs[i];
    jb->d = d; jb->w = w; jb->x = x; jb->tokens = tokens;
    jb->n_tokens = n_tokens; jb->first = i; jb->step = nthreads;
    jb->route_logits = route_logits; jb->route_gate = route_gate;
    jb->out_bf16 = out_bf16; jb->out_f64 = out_f64; jb->ids = ids;
    jb->weights = weights; jb->sgate = sgate; jb->logits = logits;
    jb->gate_logit = gate_logit; jb->y = y; jb->h = h;
  }
  for (int i = 1; i < nthreads; ++i)
    pthread_create(&th[i], NULL, block_worker, &jobs[i]);
  block_worker(&jobs[0]);
  int bad = jobs[0].bad;
  for (int i = 1; i < nthreads; ++i) {
    pthread_join(th[i], NULL);
    bad += jobs[i].bad;
  }
  free(jobs);
  free(th);
  return bad;
}
