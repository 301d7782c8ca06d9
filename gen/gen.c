/*
 * Seeded synthetic inputs for long-context decode attention.
 *
 * This module builds the query, key and value tensors that both the CUDA
 * path and the CPU oracle consume.  It holds none of the attention method's
 * arithmetic: no RMS normalisation, no ReLU^2 weight, no normaliser, no
 * selection and no softmax.  It only draws Gaussian numbers and steers the
 * sign of each key's raw dot product with the query heads of its group.
 *
 * Random numbers:
 *   - SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014) used as a counter-based generator: value i of
 *     a stream is the SplitMix64 output mix applied to stream + (i+1)*golden.
 *   - Box-Muller (Box and Muller, 1958) turns pairs of uniforms in (0,1] into
 *     pairs of standard normals.
 *   Every element is a pure function of (seed, stream, index), so any
 *   element can be regenerated alone and the loops run in parallel.
 *
 * Sign control (the construction used for "key signs set so a fraction f of
 * scores per head are > 0"): for a KV-head group with query rows Q (G x D),
 * a key z ~ N(0, I) with raw scores c = Q z and a target sign t in {+1,-1} is
 * moved inside span(Q) to k = z + Q^T (Q Q^T)^-1 (t|c| - c), so every head of
 * the group scores it with sign t and the natural Gaussian magnitude.  After
 * rounding to bf16 each key is checked against a margin on D*cos(q_h, k) and
 * redrawn if it misses; a candidate at a top-k boundary is redrawn until the
 * boundary gap is at least the requested gap both on max_h D*cos(q_h, k) (the
 * group's score) and on every head's own D*cos(q_h, k), so that a selection by
 * either score has a unique answer.
 *
 * Build: gcc -O2 -fPIC -shared -fopenmp -ffp-contract=off gen.c -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t x) {
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ULL;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBULL;
  return x ^ (x >> 31);
}

/* SplitMix64 value at counter i of a stream. */
static inline uint64_t sm_at(uint64_t stream, uint64_t i) {
  return mix64(stream + (i + 1) * GOLDEN);
}

/* Uniform double in (0, 1], 53 random bits. */
static inline double u01(uint64_t stream, uint64_t i) {
  return (double)((sm_at(stream, i) >> 11) + 1) * 0x1p-53;
}

/* Standard normal number `idx` of a stream (Box-Muller on counter pairs). */
static double normal_at(uint64_t stream, uint64_t idx) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t p = idx >> 1;
  double u1 = u01(stream, 2 * p);
  double u2 = u01(stream, 2 * p + 1);
  double r = sqrt(-2.0 * log(u1));
  return (idx & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

/* Derive a sub-stream key from a parent stream and two labels. */
uint64_t gen_substream(uint64_t parent, uint64_t a, uint64_t b) {
  return mix64(mix64(parent ^ mix64(a + GOLDEN)) ^ mix64(b + 2 * GOLDEN));
}

static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)0x7fc0u;
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

static double bf16_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* out[i] = bf16(N(0,1) number start+i of `stream`), i < count. */
void gen_normal_bf16(uint64_t stream, int64_t start, int64_t count, uint16_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i)
    out[i] = f32_to_bf16((float)normal_at(stream, (uint64_t)(start + i)));
}

/* 8-bit floats, E4M3 without infinities: sign, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN; the largest finite
 * magnitude is 448.  Rounding to nearest, ties to even; magnitudes past 448 saturate. */
static uint8_t f64_to_e4m3(double x) {
  const uint8_t sign = x < 0.0 ? 0x80 : 0x00;
  const double a = fabs(x);
  if (a != a) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    const double m = nearbyint(a * 512.0); /* units of 2^-9; 8 carries into the first normal */
    return sign | (uint8_t)m;
  }
  int e;
  frexp(a, &e); /* a in [2^(e-1), 2^e) */
  int E = e - 1 + 7;
  double r = nearbyint((a / ldexp(1.0, e - 1) - 1.0) * 8.0);
  if (r >= 8.0) { r = 0.0; E += 1; }
  if (E > 15 || (E == 15 && r > 6.0)) return sign | 0x7E;
  return sign | (uint8_t)(E << 3) | (uint8_t)r;
}

static double e4m3_to_f64(uint8_t b) {
  const int E = (b >> 3) & 15, m = b & 7;
  if (E == 15 && m == 7) return NAN;
  const double v = E == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, E - 7);
  return (b & 0x80) ? -v : v;
}

/* One row to 8 bits with its own scale (the largest magnitude maps to 448); deq, when
 * given, receives scale * value as the reader will see it. */
static void quantize_row_e4m3(const double *v, int D, uint8_t *out, float *scale, double *deq) {
  double amax = 0.0;
  for (int d = 0; d < D; ++d) if (fabs(v[d]) > amax) amax = fabs(v[d]);
  const float sc = amax > 0.0 ? (float)(amax / 448.0) : 1.0f;
  for (int d = 0; d < D; ++d) {
    out[d] = f64_to_e4m3(v[d] / (double)sc);
    if (deq) deq[d] = (double)sc * e4m3_to_f64(out[d]);
  }
  *scale = sc;
}

/* Rows of standard normals (row r uses draws r*D .. r*D+D-1 of the stream) in 8 bits. */
void gen_normal_e4m3(uint64_t stream, int64_t rows, int D, uint8_t *out, float *scale) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double v[1024];
    for (int d = 0; d < D && d < 1024; ++d) v[d] = normal_at(stream, (uint64_t)(r * D + d));
    quantize_row_e4m3(v, D, out + r * D, scale + r, NULL);
  }
}

/* Element codes to values (for tests of the encoder). */
void gen_e4m3_encode(const double *x, int64_t n, uint8_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f64_to_e4m3(x[i]);
}

/*
 * Target signs for n keys (t[j] = +1 means every head of the group scores
 * key j above zero).  kind 0: independent, P(+1) = frac.  kind 1: exactly
 * round(frac*n) keys chosen uniformly (selection sampling, Knuth's
 * Algorithm S).  kind 2: round(frac*n/run_len) non-overlapping runs of
 * run_len keys at uniformly random unaligned starts.  Returns the number of
 * +1 entries, or -1 on bad arguments.
 */
int64_t gen_targets(uint64_t stream, int64_t n, int kind, double frac, int64_t run_len,
                    int8_t *t) {
  if (n < 0 || frac < 0.0 || frac > 1.0) return -1;
  int64_t pos = 0;
  if (kind == 0) {
    for (int64_t j = 0; j < n; ++j) {
      t[j] = (u01(stream, (uint64_t)j) <= frac) ? 1 : -1;
      pos += t[j] > 0;
    }
    return pos;
  }
  for (int64_t j = 0; j < n; ++j) t[j] = -1;
  if (kind == 1) {
    int64_t m = (int64_t)llround(frac * (double)n);
    int64_t need = m;
    for (int64_t j = 0; j < n && need > 0; ++j) {
      /* select j with probability need / (n - j) */
      double u = (double)(sm_at(stream, (uint64_t)j) >> 11) * 0x1p-53;
      if (u * (double)(n - j) < (double)need) {
        t[j] = 1;
        --need;
      }
    }
    return m;
  }
  if (kind == 2) {
    if (run_len <= 0) return -1;
    int64_t runs = (int64_t)llround(frac * (double)n / (double)run_len);
    int64_t range = n - runs * run_len + runs; /* choose runs distinct x in [0, range) */
    if (runs < 0 || range < runs) return -1;
    int64_t need = runs, r = 0;
    for (int64_t x = 0; x < range && need > 0; ++x) {
      double u = (double)(sm_at(stream, (uint64_t)x) >> 11) * 0x1p-53;
      if (u * (double)(range - x) < (double)need) {
        int64_t start = x + r * (run_len - 1);
        for (int64_t j = start; j < start + run_len; ++j) t[j] = 1;
        ++r;
        --need;
      }
    }
    return runs * run_len;
  }
  return -1;
}

/* Solve the G x G system in place (Gauss-Jordan, partial pivoting). */
static int invert_small(int G, double *a, double *inv) {
  for (int i = 0; i < G; ++i)
    for (int j = 0; j < G; ++j) inv[i * G + j] = (i == j) ? 1.0 : 0.0;
  for (int col = 0; col < G; ++col) {
    int piv = col;
    for (int r = col + 1; r < G; ++r)
      if (fabs(a[r * G + col]) > fabs(a[piv * G + col])) piv = r;
    if (fabs(a[piv * G + col]) < 1e-12) return -1;
    if (piv != col)
      for (int j = 0; j < G; ++j) {
        double tmp = a[col * G + j]; a[col * G + j] = a[piv * G + j]; a[piv * G + j] = tmp;
        tmp = inv[col * G + j]; inv[col * G + j] = inv[piv * G + j]; inv[piv * G + j] = tmp;
      }
    double d = a[col * G + col];
    for (int j = 0; j < G; ++j) { a[col * G + j] /= d; inv[col * G + j] /= d; }
    for (int r = 0; r < G; ++r) {
      if (r == col) continue;
      double f = a[r * G + col];
      if (f == 0.0) continue;
      for (int j = 0; j < G; ++j) { a[r * G + j] -= f * a[col * G + j]; inv[r * G + j] -= f * inv[col * G + j]; }
    }
  }
  return 0;
}

#define MAXG 16
#define MAXD 512

typedef struct {
  int G, D;
  double q[MAXG * MAXD];
  double qnorm[MAXG];
  double minv[MAXG * MAXG];
  double margin;
  uint64_t stream;
  int e4m3;        /* keys stored in 8 bits with a scale per row, else bf16 */
  uint16_t *Kb;    /* bf16 keys (row stride D) */
  uint8_t *K8;     /* 8-bit keys (row stride D) */
  float *Ks;       /* their scales */
} signer;

/* Key j as the reader sees it (decoded), into kd. */
static void key_values(const signer *s, int64_t j, double *kd) {
  if (s->e4m3) {
    for (int d = 0; d < s->D; ++d) kd[d] = (double)s->Ks[j] * e4m3_to_f64(s->K8[j * s->D + d]);
  } else {
    for (int d = 0; d < s->D; ++d) kd[d] = bf16_to_f64(s->Kb[j * s->D + d]);
  }
}

/* Store key j from its exact values. */
static void store_key(const signer *s, int64_t j, const double *v) {
  if (s->e4m3) {
    quantize_row_e4m3(v, s->D, s->K8 + j * s->D, s->Ks + j, NULL);
  } else {
    for (int d = 0; d < s->D; ++d) s->Kb[j * s->D + d] = f32_to_bf16((float)v[d]);
  }
}

/* D*cos(q_h, k) of every head of the group (vals[0..G)) and their maximum (vals[G]),
 * in double, from key j as stored. */
static void proxy_values(const signer *s, int64_t j, double *vals) {
  double kk = 0.0;
  double kd[MAXD];
  key_values(s, j, kd);
  for (int d = 0; d < s->D; ++d) kk += kd[d] * kd[d];
  double kn = sqrt(kk), best = -INFINITY;
  for (int h = 0; h < s->G; ++h) {
    double dot = 0.0;
    for (int d = 0; d < s->D; ++d) dot += s->q[h * s->D + d] * kd[d];
    double v = (kn > 0.0 && s->qnorm[h] > 0.0) ? (double)s->D * dot / (s->qnorm[h] * kn) : 0.0;
    vals[h] = v;
    if (v > best) best = v;
  }
  vals[s->G] = best;
}

/* Draw key j (attempt a) with target sign t; returns 1 when it meets the margin. */
static int draw_key(const signer *s, int64_t j, int64_t a, int t) {
  const int G = s->G, D = s->D;
  uint64_t st = gen_substream(s->stream, (uint64_t)j, (uint64_t)a);
  double z[MAXD], c[MAXG], want[MAXG], delta[MAXG];
  double zz = 0.0;
  for (int d = 0; d < D; ++d) { z[d] = normal_at(st, (uint64_t)d); zz += z[d] * z[d]; }
  double zn = sqrt(zz);
  for (int h = 0; h < G; ++h) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += s->q[h * D + d] * z[d];
    c[h] = dot;
    double floor_raw = 2.0 * s->margin * s->qnorm[h] * zn / (double)D;
    double mag = fabs(dot) > floor_raw ? fabs(dot) : floor_raw;
    want[h] = (double)t * mag - dot;
  }
  for (int h = 0; h < G; ++h) {
    double acc = 0.0;
    for (int i = 0; i < G; ++i) acc += s->minv[h * G + i] * want[i];
    delta[h] = acc;
  }
  double v[MAXD];
  for (int d = 0; d < D; ++d) {
    v[d] = z[d];
    for (int h = 0; h < G; ++h) v[d] += delta[h] * s->q[h * D + d];
  }
  store_key(s, j, v);
  /* check every head's sign and margin on the stored (rounded) key */
  double kd[MAXD], kk = 0.0;
  key_values(s, j, kd);
  for (int d = 0; d < D; ++d) kk += kd[d] * kd[d];
  double kn = sqrt(kk);
  if (!(kn > 0.0)) return 0;
  for (int h = 0; h < G; ++h) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += s->q[h * D + d] * kd[d];
    double cs = (double)D * dot / (s->qnorm[h] * kn);
    if ((double)t * cs < s->margin) return 0;
  }
  return 1;
}

static void swap_d(double *a, double *b) { double t = *a; *a = *b; *b = t; }
static void swap_i(int64_t *a, int64_t *b) { int64_t t = *a; *a = *b; *b = t; }

/* Rearrange (v, id) so that positions [0, k) hold the k largest values and
 * position k holds the (k+1)-th largest (Hoare quickselect, descending). */
static void select_desc(double *v, int64_t *id, int64_t n, int64_t k) {
  int64_t lo = 0, hi = n - 1;
  while (lo < hi) {
    int64_t mid = lo + (hi - lo) / 2;
    double p = v[mid];
    int64_t i = lo, j = hi;
    while (i <= j) {
      while (v[i] > p) ++i;
      while (v[j] < p) --j;
      if (i <= j) { swap_d(&v[i], &v[j]); swap_i(&id[i], &id[j]); ++i; --j; }
    }
    if (k <= j) hi = j;
    else if (k >= i) lo = i;
    else return;
  }
}

/*
 * Sign-controlled keys for one (batch, KV-head) unit.
 *   q      : G x D bf16 bits, the query rows of the group (row-major)
 *   t      : n target signs
 *   n_cand : keys [0, n_cand) compete for the top-`topk` selection; when
 *            n_cand > topk the gap between the topk-th and (topk+1)-th
 *            largest max_h D*cos(q_h, k), and the same gap for every head's
 *            own D*cos(q_h, k), is made >= gap
 *   K      : n x D bf16 bits out (row stride D)
 * Returns the number of redraws (>= 0), or a negative error code:
 *   -1 bad arguments, -2 singular query group, -3 margin not met after
 *   max_attempts draws, -4 gap not met after max_gap_iters redraws.
 */
static int64_t signed_keys(uint64_t stream, int G, int D, int64_t n, const uint16_t *q,
                           const int8_t *t, int64_t n_cand, int64_t topk, double margin,
                           double gap, int max_attempts, int64_t max_gap_iters, uint16_t *Kb,
                           uint8_t *K8, float *Ks) {
  if (G < 1 || G > MAXG || D < 1 || D > MAXD || n < 0 || n_cand > n) return -1;
  signer *s = (signer *)malloc(sizeof(signer));
  if (!s) return -1;
  s->G = G; s->D = D; s->margin = margin; s->stream = stream;
  s->e4m3 = K8 != NULL; s->Kb = Kb; s->K8 = K8; s->Ks = Ks;
  for (int i = 0; i < G * D; ++i) s->q[i] = bf16_to_f64(q[i]);
  double m[MAXG * MAXG];
  for (int h = 0; h < G; ++h) {
    double nn = 0.0;
    for (int d = 0; d < D; ++d) nn += s->q[h * D + d] * s->q[h * D + d];
    s->qnorm[h] = sqrt(nn);
    for (int i = 0; i < G; ++i) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += s->q[h * D + d] * s->q[i * D + d];
      m[h * G + i] = dot;
    }
  }
  if (invert_small(G, m, s->minv) != 0) { free(s); return -2; }

  int64_t *attempt = (int64_t *)calloc((size_t)(n > 0 ? n : 1), sizeof(int64_t));
  int failed = 0;
  int64_t redraws = 0;
#pragma omp parallel for schedule(dynamic, 256) reduction(+ : redraws) reduction(| : failed)
  for (int64_t j = 0; j < n; ++j) {
    int64_t a = 0;
    while (!draw_key(s, j, a, t[j] > 0 ? 1 : -1)) {
      if (++a >= max_attempts) { failed = 1; break; }
    }
    attempt[j] = a;
    redraws += a;
  }
  if (failed) { free(attempt); free(s); return -3; }

  if (n_cand > topk && topk > 0) {
    /* The top-k boundary must be clear both for the group's score (the maximum over its
     * heads) and for every head's own score: column a of v holds, for a < G, head a's
     * D*cos and, for a = G, their maximum.  A pass checks every column; a key at a
     * boundary that is too narrow is redrawn and the pass starts again. */
    const int A = G + 1;
    double *v = (double *)malloc(sizeof(double) * (size_t)n_cand * (size_t)A);
    double *w = (double *)malloc(sizeof(double) * (size_t)n_cand);
    int64_t *id = (int64_t *)malloc(sizeof(int64_t) * (size_t)n_cand);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n_cand; ++j) {
      double vals[MAXG + 1];
      proxy_values(s, j, vals);
      for (int a = 0; a < A; ++a) v[(size_t)a * n_cand + j] = vals[a];
    }
    int64_t iters = 0;
    int a = 0, clean = 0;
    while (clean < A) {
      const double *va = v + (size_t)a * n_cand;
      for (int64_t j = 0; j < n_cand; ++j) { w[j] = va[j]; id[j] = j; }
      select_desc(w, id, n_cand, topk);
      /* w[topk] is the (topk+1)-th largest; the topk-th is the min of w[0..topk) */
      double lo_in = INFINITY;
      for (int64_t i = 0; i < topk; ++i) if (w[i] < lo_in) lo_in = w[i];
      if (lo_in - w[topk] >= gap) {
        ++clean;
        a = (a + 1) % A;
        continue;
      }
      if (++iters > max_gap_iters) { failed = 1; break; }
      int64_t j = id[topk];
      int64_t at = attempt[j];
      do {
        if (++at >= attempt[j] + max_attempts) { failed = 1; break; }
      } while (!draw_key(s, j, at, t[j] > 0 ? 1 : -1));
      if (failed) break;
      redraws += at - attempt[j];
      attempt[j] = at;
      double vals[MAXG + 1];
      proxy_values(s, j, vals);
      for (int b = 0; b < A; ++b) v[(size_t)b * n_cand + j] = vals[b];
      clean = 0;
    }
    free(v); free(w); free(id);
    if (failed) { free(attempt); free(s); return -4; }
  }
  free(attempt);
  free(s);
  return redraws;
}

int64_t gen_signed_keys(uint64_t stream, int G, int D, int64_t n, const uint16_t *q,
                        const int8_t *t, int64_t n_cand, int64_t topk, double margin,
                        double gap, int max_attempts, int64_t max_gap_iters, uint16_t *K) {
  return signed_keys(stream, G, D, n, q, t, n_cand, topk, margin, gap, max_attempts,
                     max_gap_iters, K, NULL, NULL);
}

/* The same keys stored in 8 bits (E4M3) with one scale per key; signs, margins and the
 * top-k gap hold for the decoded keys. */
int64_t gen_signed_keys_e4m3(uint64_t stream, int G, int D, int64_t n, const uint16_t *q,
                             const int8_t *t, int64_t n_cand, int64_t topk, double margin,
                             double gap, int max_attempts, int64_t max_gap_iters, uint8_t *K8,
                             float *Ks) {
  return signed_keys(stream, G, D, n, q, t, n_cand, topk, margin, gap, max_attempts,
                     max_gap_iters, NULL, K8, Ks);
}
