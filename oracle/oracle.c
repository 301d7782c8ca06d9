/*
 * fp64 CPU oracle for long-context single-token decode attention in Embla 1.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg call this code.  It shares nothing with the CUDA library:
 * no headers, no helpers, no tables.  Inputs arrive as doubles (the bf16
 * values the GPU reads, widened exactly); every sum is a plain loop in fp64
 * in the order the definition states, with no blocking or reordering.
 *
 * Source: "The Architecture of Embla 1" (Sevren blog), sections
 *   "Three kinds of attention"                     (window, full, sparse layers)
 *   "Sevren Sparse Attention learns to be sparse"  (ReLU^2 weights over RMS-normalised q, k)
 *   "Skipping V"                                   (a value is needed when any head of the group weighs its key)
 *
 * Readings of points the page leaves open (its display equation was lost):
 *   - score  s_hj = alpha * (q_h / rms(q_h)) . (k_j / rms(k_j)),
 *            rms(x) = sqrt(mean(x^2) + eps); alpha and eps are arguments;
 *   - weight w_hj = max(s_hj, 0)^2;
 *   - output out_h = sum_j w_hj v_j / (c + sum_j w_hj), c an argument;
 *            0 when c + sum_j w_hj == 0;
 *   - selection score sigma_j = max over the group's heads of s_hj, rounded to
 *     fp32: survival (sigma_j > 0) and the top-k order are decided on that
 *     fp32 value, the precision the CUDA kernels decide in;
 *   - selection = the topk largest sigma_j among j < n - recent (ties to the
 *     smaller j) plus the `recent` newest keys; every key when n <= topk+recent;
 *   - sparse layer: softmax of tau * q'_h . k_j over the selected keys;
 *   - window layer: RoPE on q at position pos (pairs (2i, 2i+1) rotated by
 *     pos * base^(-2i/D)), keys stored already rotated, softmax of
 *     tau * q_rot . k over the valid ring slots.
 *
 * Build: gcc -O2 -fPIC -shared -fopenmp -ffp-contract=off oracle.c -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the batched functions below spread their units over (n >= 1); returns the
 * number they used before.  Only timing code changes it: results do not depend on it. */
int oracle_set_threads(int n) {
#ifdef _OPENMP
  int before = omp_get_max_threads();
  if (n >= 1) omp_set_num_threads(n);
  return before;
#else
  (void)n;
  return 1;
#endif
}

/* 1 / sqrt(mean(x^2) + eps) */
static double rms_inverse(const double *x, int D, double eps) {
  double ss = 0.0;
  for (int d = 0; d < D; ++d) ss += x[d] * x[d];
  return 1.0 / sqrt(ss / (double)D + eps);
}

static double dot(const double *a, const double *b, int D) {
  double s = 0.0;
  for (int d = 0; d < D; ++d) s += a[d] * b[d];
  return s;
}

/*
 * Full-layer scores of one (batch, KV-head) unit: s[h*n + j] = alpha * qhat_h . khat_j.
 * q: G x D; K: n rows with stride ldk.  Returns 0, or -1 on bad arguments.
 */
int oracle_full_scores(int G, int D, int64_t n, const double *q, const double *K, int64_t ldk,
                       double alpha, double eps, double *s) {
  if (G < 1 || D < 1 || n < 0 || ldk < D || !(eps >= 0.0)) return -1;
  double *qhat = (double *)malloc(sizeof(double) * (size_t)G * (size_t)D);
  double *khat = (double *)malloc(sizeof(double) * (size_t)D);
  if (!qhat || !khat) { free(qhat); free(khat); return -1; }
  for (int h = 0; h < G; ++h) {
    double r = rms_inverse(q + (size_t)h * D, D, eps);
    for (int d = 0; d < D; ++d) qhat[h * D + d] = q[(size_t)h * D + d] * r;
  }
  for (int64_t j = 0; j < n; ++j) {
    const double *k = K + j * ldk;
    double r = rms_inverse(k, D, eps);
    for (int d = 0; d < D; ++d) khat[d] = k[d] * r;
    for (int h = 0; h < G; ++h) s[(int64_t)h * n + j] = alpha * dot(qhat + h * D, khat, D);
  }
  free(qhat);
  free(khat);
  return 0;
}

/*
 * Full (ReLU^2) layer decode for one unit.
 *   out     : G x D
 *   sigma32 : n selection scores (fp32), may be NULL
 *   n_surv  : keys with sigma32 > 0 (their V rows are the only ones needed)
 *   n_zero  : per head, keys with exactly zero weight (s_hj <= 0), may be NULL
 */
int oracle_full_decode(int G, int D, int64_t n, const double *q, const double *K, int64_t ldk,
                       const double *V, int64_t ldv, double alpha, double c, double eps,
                       double *out, float *sigma32, int64_t *n_surv, int64_t *n_zero) {
  if (ldv < D) return -1;
  double *s = (double *)malloc(sizeof(double) * (size_t)G * (size_t)(n > 0 ? n : 1));
  double *num = (double *)calloc((size_t)G * (size_t)D, sizeof(double));
  double *den = (double *)calloc((size_t)G, sizeof(double));
  if (!s || !num || !den) { free(s); free(num); free(den); return -1; }
  if (oracle_full_scores(G, D, n, q, K, ldk, alpha, eps, s) != 0) {
    free(s); free(num); free(den);
    return -1;
  }
  int64_t surv = 0;
  if (n_zero) for (int h = 0; h < G; ++h) n_zero[h] = 0;
  for (int64_t j = 0; j < n; ++j) {
    double sigma = -INFINITY;
    for (int h = 0; h < G; ++h) {
      double shj = s[(int64_t)h * n + j];
      if (shj > sigma) sigma = shj;
      double w = shj > 0.0 ? shj * shj : 0.0;
      if (w == 0.0) {
        if (n_zero) n_zero[h] += 1;
        continue;
      }
      const double *v = V + j * ldv;
      for (int d = 0; d < D; ++d) num[h * D + d] += w * v[d];
      den[h] += w;
    }
    float sig32 = (float)sigma;
    if (sigma32) sigma32[j] = sig32;
    if (sig32 > 0.0f) ++surv;
  }
  for (int h = 0; h < G; ++h) {
    double z = c + den[h];
    for (int d = 0; d < D; ++d) out[h * D + d] = (z != 0.0) ? num[h * D + d] / z : 0.0;
  }
  *n_surv = surv;
  free(s); free(num); free(den);
  return 0;
}

typedef struct { float s; int32_t j; } cand;

/* higher score first; equal scores: smaller index first */
static int cand_order(const void *a, const void *b) {
  const cand *x = (const cand *)a, *y = (const cand *)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->j < y->j) ? -1 : (x->j > y->j);
}

/*
 * Sparse-layer selection for one unit: the topk highest sigma32 among the
 * candidates j < n - recent, plus the `recent` newest keys, ascending.
 * idx needs min(n, topk + recent) entries.
 */
int oracle_select_topk(int64_t n, const float *sigma32, int64_t topk, int64_t recent, int32_t *idx,
                       int64_t *count) {
  if (n < 0 || topk < 0 || recent < 0 || n > INT32_MAX) return -1;
  if (n <= topk + recent) {
    for (int64_t j = 0; j < n; ++j) idx[j] = (int32_t)j;
    *count = n;
    return 0;
  }
  int64_t n_cand = n - recent;
  cand *cs = (cand *)malloc(sizeof(cand) * (size_t)n_cand);
  unsigned char *mark = (unsigned char *)calloc((size_t)n, 1);
  if (!cs || !mark) { free(cs); free(mark); return -1; }
  for (int64_t j = 0; j < n_cand; ++j) { cs[j].s = sigma32[j]; cs[j].j = (int32_t)j; }
  qsort(cs, (size_t)n_cand, sizeof(cand), cand_order);
  for (int64_t i = 0; i < topk; ++i) mark[cs[i].j] = 1;
  for (int64_t j = n_cand; j < n; ++j) mark[j] = 1;
  int64_t m = 0;
  for (int64_t j = 0; j < n; ++j)
    if (mark[j]) idx[m++] = (int32_t)j;
  *count = m;
  free(cs);
  free(mark);
  return 0;
}

/*
 * Sparse-layer decode for one unit: softmax of tau * q'_h . k_j over the m
 * selected keys idx[0..m), output G x D.
 */
int oracle_sparse_decode(int G, int D, int64_t m, const double *q, const double *K, int64_t ldk,
                         const double *V, int64_t ldv, const int32_t *idx, double tau,
                         double *out) {
  if (G < 1 || D < 1 || m < 0 || ldk < D || ldv < D) return -1;
  double *z = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
  if (!z) return -1;
  for (int h = 0; h < G; ++h) {
    const double *qh = q + (size_t)h * D;
    double zmax = -INFINITY;
    for (int64_t i = 0; i < m; ++i) {
      z[i] = tau * dot(qh, K + (int64_t)idx[i] * ldk, D);
      if (z[i] > zmax) zmax = z[i];
    }
    double denom = 0.0;
    for (int64_t i = 0; i < m; ++i) { z[i] = exp(z[i] - zmax); denom += z[i]; }
    for (int d = 0; d < D; ++d) out[(size_t)h * D + d] = 0.0;
    for (int64_t i = 0; i < m; ++i) {
      double p = z[i] / denom;
      const double *v = V + (int64_t)idx[i] * ldv;
      for (int d = 0; d < D; ++d) out[(size_t)h * D + d] += p * v[d];
    }
  }
  free(z);
  return 0;
}

/*
 * Window-layer decode for one unit.  Kw, Vw: W ring slots (slot = position
 * mod W), keys already rotated at their own positions.  The valid positions
 * are max(0, pos-W+1) .. pos.  q is rotated at pos, then softmax attention.
 */
int oracle_window_decode(int G, int D, int64_t W, int64_t pos, const double *q, const double *Kw,
                         const double *Vw, double base, double tau, double *out) {
  if (G < 1 || D < 2 || (D & 1) || W < 1 || pos < 0) return -1;
  double *qr = (double *)malloc(sizeof(double) * (size_t)D);
  double *z = (double *)malloc(sizeof(double) * (size_t)W);
  int64_t *slot = (int64_t *)malloc(sizeof(int64_t) * (size_t)W);
  if (!qr || !z || !slot) { free(qr); free(z); free(slot); return -1; }
  int64_t first = pos - W + 1 > 0 ? pos - W + 1 : 0;
  int64_t nv = 0;
  for (int64_t p = first; p <= pos; ++p) slot[nv++] = p % W;
  for (int h = 0; h < G; ++h) {
    const double *qh = q + (size_t)h * D;
    for (int i = 0; i < D / 2; ++i) {
      double theta = (double)pos * pow(base, -2.0 * (double)i / (double)D);
      double cs = cos(theta), sn = sin(theta);
      qr[2 * i] = qh[2 * i] * cs - qh[2 * i + 1] * sn;
      qr[2 * i + 1] = qh[2 * i] * sn + qh[2 * i + 1] * cs;
    }
    double zmax = -INFINITY;
    for (int64_t i = 0; i < nv; ++i) {
      z[i] = tau * dot(qr, Kw + slot[i] * D, D);
      if (z[i] > zmax) zmax = z[i];
    }
    double denom = 0.0;
    for (int64_t i = 0; i < nv; ++i) { z[i] = exp(z[i] - zmax); denom += z[i]; }
    for (int d = 0; d < D; ++d) out[(size_t)h * D + d] = 0.0;
    for (int64_t i = 0; i < nv; ++i) {
      double p = z[i] / denom;
      const double *v = Vw + slot[i] * D;
      for (int d = 0; d < D; ++d) out[(size_t)h * D + d] += p * v[d];
    }
  }
  free(qr); free(z); free(slot);
  return 0;
}

/* ----------------------------------------------------------------------------
 * Batched forms: every (b, g) unit of a batch, units spread over OpenMP
 * threads.  Query head h belongs to KV head h / G with G = Hq / Hkv, so the
 * G query rows of unit (b, g) are rows g*G .. g*G+G-1 of q[b].
 * ------------------------------------------------------------------------- */

int oracle_full_decode_batch(int B, int Hq, int Hkv, int D, int64_t n, int64_t ncap,
                             const double *q, const double *K, const double *V, double alpha,
                             double c, double eps, double *out, float *sigma32, int64_t *n_surv) {
  if (B < 0 || Hkv < 1 || Hq % Hkv || ncap < n) return -1;
  int G = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int64_t u = 0; u < (int64_t)B * Hkv; ++u) {
    int64_t b = u / Hkv, g = u % Hkv;
    const double *qu = q + ((size_t)b * Hq + (size_t)g * G) * D;
    const double *Ku = K + (size_t)u * ncap * D;
    const double *Vu = V + (size_t)u * ncap * D;
    double *ou = out + ((size_t)b * Hq + (size_t)g * G) * D;
    float *su = sigma32 ? sigma32 + (size_t)u * ncap : NULL;
    err |= oracle_full_decode(G, D, n, qu, Ku, D, Vu, D, alpha, c, eps, ou, su, n_surv + u, NULL) != 0;
  }
  return err ? -1 : 0;
}

/*
 * Every query head's own full-layer scores, rounded to fp32: s32[b][h][j] = (float)
 * s_hj for j < n (rows j >= n of each head are not written).  These are the scores the
 * per-query-head reading of the selection ranks ("The Architecture of Embla 1", section
 * "Three kinds of attention", Sparse: the keys that layer scored highest, here each head's
 * own), rounded to the precision the CUDA kernels rank in.
 */
int oracle_head_scores_batch(int B, int Hq, int Hkv, int D, int64_t n, int64_t ncap,
                             const double *q, const double *K, double alpha, double eps,
                             float *s32) {
  if (B < 0 || Hkv < 1 || Hq % Hkv || ncap < n || n < 0) return -1;
  int G = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int64_t u = 0; u < (int64_t)B * Hkv; ++u) {
    int64_t b = u / Hkv, g = u % Hkv;
    double *s = (double *)malloc(sizeof(double) * (size_t)G * (size_t)(n > 0 ? n : 1));
    if (!s) { err |= 1; continue; }
    const double *qu = q + ((size_t)b * Hq + (size_t)g * G) * D;
    if (oracle_full_scores(G, D, n, qu, K + (size_t)u * ncap * D, D, alpha, eps, s) != 0) {
      err |= 1;
    } else {
      for (int h = 0; h < G; ++h) {
        float *o = s32 + ((size_t)b * Hq + (size_t)g * G + h) * ncap;
        for (int64_t j = 0; j < n; ++j) o[j] = (float)s[(int64_t)h * n + j];
      }
    }
    free(s);
  }
  return err ? -1 : 0;
}

/*
 * Causal full-layer (ReLU^2) attention over a prompt, for one (batch, KV-head) unit
 * ("The Architecture of Embla 1", section "KV bridge, KV reuse, and prefill": in prefill the
 * early layers run on every prompt token; their full layers apply the same ReLU^2 rule as
 * decode, and a token sees the keys up to and including its own, there being no position
 * encoding in a full layer).  The T prompt tokens are the last T of the n keys: query t of
 * head h sits at position p = n - T + t and attends to keys j = 0 .. p.
 *   q   : G x T x D (head-major)
 *   K, V: n rows with strides ldk, ldv
 *   out : G x T x D;  out = sum_{j<=p} w v_j / (c + sum_{j<=p} w), 0 when that is 0
 */
int oracle_prefill(int G, int D, int64_t n, int64_t T, const double *q, const double *K,
                   int64_t ldk, const double *V, int64_t ldv, double alpha, double c, double eps,
                   double *out) {
  if (G < 1 || D < 1 || T < 0 || n < T || ldk < D || ldv < D || !(eps >= 0.0)) return -1;
  double *khat = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)D);
  double *num = (double *)malloc(sizeof(double) * (size_t)D);
  if (!khat || !num) { free(khat); free(num); return -1; }
  for (int64_t j = 0; j < n; ++j) {
    double r = rms_inverse(K + j * ldk, D, eps);
    for (int d = 0; d < D; ++d) khat[j * D + d] = K[j * ldk + d] * r;
  }
  for (int h = 0; h < G; ++h) {
    for (int64_t t = 0; t < T; ++t) {
      const double *qt = q + ((size_t)h * T + t) * D;
      double r = rms_inverse(qt, D, eps);
      int64_t p = n - T + t;
      double den = 0.0;
      for (int d = 0; d < D; ++d) num[d] = 0.0;
      for (int64_t j = 0; j <= p; ++j) {
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += qt[d] * r * khat[j * D + d];
        s *= alpha;
        double w = s > 0.0 ? s * s : 0.0;
        if (w == 0.0) continue;
        for (int d = 0; d < D; ++d) num[d] += w * V[j * ldv + d];
        den += w;
      }
      double z = c + den;
      double *o = out + ((size_t)h * T + t) * D;
      for (int d = 0; d < D; ++d) o[d] = (z != 0.0) ? num[d] / z : 0.0;
    }
  }
  free(khat);
  free(num);
  return 0;
}

/* Every unit: q [B, Hq, T, D], K and V [B, Hkv, ncap, D], out [B, Hq, T, D]. */
int oracle_prefill_batch(int B, int Hq, int Hkv, int D, int64_t n, int64_t T, int64_t ncap,
                         const double *q, const double *K, const double *V, double alpha,
                         double c, double eps, double *out) {
  if (B < 0 || Hkv < 1 || Hq % Hkv || ncap < n) return -1;
  int G = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int64_t u = 0; u < (int64_t)B * Hkv; ++u) {
    int64_t b = u / Hkv, g = u % Hkv;
    const double *qu = q + ((size_t)b * Hq + (size_t)g * G) * T * D;
    double *ou = out + ((size_t)b * Hq + (size_t)g * G) * T * D;
    err |= oracle_prefill(G, D, n, T, qu, K + (size_t)u * ncap * D, D, V + (size_t)u * ncap * D,
                          D, alpha, c, eps, ou) != 0;
  }
  return err ? -1 : 0;
}

/*
 * ReLU^2 MLP of one token ("The Architecture of Embla 1", section "ReLU^2 activation":
 * negative pre-activations become zero and positive ones are squared; a zero neuron's row
 * of the down projection contributes nothing, so at batch size 1 only the rows of the
 * neurons that fired need reading).
 *   x      : d
 *   w_up   : f rows of d (row i = neuron i's input weights), stride d
 *   w_down : f rows of d (row i = neuron i's output weights), stride d
 *   h      : f (may be NULL): h_i = max(w_up_i . x, 0)^2
 *   y      : d, y = sum_i h_i w_down_i over the neurons with h_i > 0
 *   n_live : neurons with h_i > 0
 */
int oracle_relu2_mlp(int64_t d, int64_t f, const double *x, const double *w_up,
                     const double *w_down, double *h, double *y, int64_t *n_live) {
  if (d < 1 || f < 0 || !x || !w_up || !w_down || !y || !n_live) return -1;
  for (int64_t c = 0; c < d; ++c) y[c] = 0.0;
  int64_t live = 0;
  for (int64_t i = 0; i < f; ++i) {
    const double *wu = w_up + i * d;
    double a = 0.0;
    for (int64_t c = 0; c < d; ++c) a += wu[c] * x[c];
    double hi = a > 0.0 ? a * a : 0.0;
    if (h) h[i] = hi;
    if (hi == 0.0) continue;
    ++live;
    const double *wd = w_down + i * d;
    for (int64_t c = 0; c < d; ++c) y[c] += hi * wd[c];
  }
  *n_live = live;
  return 0;
}

/*
 * V-read accounting of one unit ("The Architecture of Embla 1", section "Skipping V": a
 * value row is needed only when some head of the group gives its key a weight above zero,
 * i.e. sigma_j > 0; the page's kernel checks keys in groups of 8).
 *   keys_needed   : keys j < n with sigma32[j] > 0
 *   chunks_needed : chunks [c*chunk, min(n, (c+1)*chunk)) holding at least one such key
 */
int oracle_skip_stats(int64_t n, const float *sigma32, int64_t chunk, int64_t *keys_needed,
                      int64_t *chunks_needed) {
  if (n < 0 || chunk < 1 || !keys_needed || !chunks_needed) return -1;
  int64_t keys = 0, chunks = 0;
  for (int64_t c0 = 0; c0 < n; c0 += chunk) {
    int any = 0;
    for (int64_t j = c0; j < n && j < c0 + chunk; ++j) {
      if (sigma32[j] > 0.0f) {
        ++keys;
        any = 1;
      }
    }
    chunks += any;
  }
  *keys_needed = keys;
  *chunks_needed = chunks;
  return 0;
}

int oracle_skip_stats_batch(int B, int Hkv, int64_t n, int64_t ncap, const float *sigma32,
                            int64_t chunk, int64_t *keys_needed, int64_t *chunks_needed) {
  int err = 0;
  for (int64_t u = 0; u < (int64_t)B * Hkv; ++u)
    err |= oracle_skip_stats(n, sigma32 + (size_t)u * ncap, chunk, keys_needed + u,
                             chunks_needed + u) != 0;
  return err ? -1 : 0;
}

int oracle_select_topk_batch(int B, int Hkv, int64_t n, int64_t ncap, const float *sigma32,
                             int64_t topk, int64_t recent, int32_t *idx, int64_t idx_stride,
                             int64_t *count) {
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int64_t u = 0; u < (int64_t)B * Hkv; ++u)
    err |= oracle_select_topk(n, sigma32 + (size_t)u * ncap, topk, recent, idx + u * idx_stride,
                              count + u) != 0;
  return err ? -1 : 0;
}

int oracle_sparse_decode_batch(int B, int Hq, int Hkv, int D, int64_t ncap, const double *q,
                               const double *K, const double *V, const int32_t *idx,
                               int64_t idx_stride, const int64_t *count, double tau, double *out) {
  if (B < 0 || Hkv < 1 || Hq % Hkv) return -1;
  int G = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int64_t u = 0; u < (int64_t)B * Hkv; ++u) {
    int64_t b = u / Hkv, g = u % Hkv;
    err |= oracle_sparse_decode(G, D, count[u], q + ((size_t)b * Hq + (size_t)g * G) * D,
                                K + (size_t)u * ncap * D, D, V + (size_t)u * ncap * D, D,
                                idx + u * idx_stride, tau,
                                out + ((size_t)b * Hq + (size_t)g * G) * D) != 0;
  }
  return err ? -1 : 0;
}

int oracle_window_decode_batch(int B, int Hq, int Hkv, int D, int64_t W, int64_t pos,
                               const double *q, const double *Kw, const double *Vw, double base,
                               double tau, double *out) {
  if (B < 0 || Hkv < 1 || Hq % Hkv) return -1;
  int G = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
  for (int64_t u = 0; u < (int64_t)B * Hkv; ++u) {
    int64_t b = u / Hkv, g = u % Hkv;
    err |= oracle_window_decode(G, D, W, pos, q + ((size_t)b * Hq + (size_t)g * G) * D,
                                Kw + (size_t)u * W * D, Vw + (size_t)u * W * D, base, tau,
                                out + ((size_t)b * Hq + (size_t)g * G) * D) != 0;
  }
  return err ? -1 : 0;
}
