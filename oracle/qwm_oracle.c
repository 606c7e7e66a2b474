/*
 * qwm_oracle.c -- plain, slow CPU oracle of the QuantWM quantise-and-attend path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library and never calls it.
 *
 * Sources (cited by page and section):
 *   [QWM-zh]  QuantWM summary (Chinese), "前置知识" (affine quantiser, centroid-residual
 *             form, logits, second-order Query statistics), "核心方法" (QSAC score,
 *             INT2 error estimate, PSAC logit form), "方法步骤详情" steps 1-5.
 *   [QWM-ko]  QuantWM summary (Korean), "무엇과 다른가" (QSAC), "어떻게 쓰나" (PSAC).
 *   [QWM-en]  QuantWM v2 summary, §4.1, §4.2, §5.1, §C.3, §D.1.
 *   [QVG-ko]  Quant VideoGen summary, §2A (k-means smoothing), §2B (progressive residual
 *             quantisation), §2C (streaming centroid caching).
 *   KIVI-style baseline: the QuantWM summaries name KIVI as a baseline with finer groups and a
 *             bf16 recent window (Korean summary "전제와 한계"); its form here is the ablation
 *             workload's: per-channel Key and per-token Value INT2 in groups of 32.
 *
 * Floating point: accumulations in double (fp64).  The two places where the
 * pages' format fixes a 32-bit computation -- the residual r = k - mu and the
 * INT2 / INT8 encoders -- are written in float with explicit IEEE rounding
 * modes, so that integer codes can be compared bit for bit.
 * Build: gcc -std=c11 -O2 -fopenmp -frounding-math -ffp-contract=off -fno-fast-math.
 *
 * Readings of the pages (where they are silent or garbled):
 *   - Affine quantiser ([QWM-zh] 前置知识) prints X_q = clip(X/s + z) without a
 *     rounding step; round-half-even is used.  Per (token, group of 64 channels):
 *     m = round_down_fp16(min r), s = round_up_fp16(round_up_f32(round_up_f32(max r - m) / 3)),
 *     q = clamp(rint((r - m) * (1/s)), 0, 3), r_hat = m + s q.  This makes
 *     |r - r_hat| <= s/2 hold for every element.  When max r == m, s = 0 and q = 0.
 *   - INT8 of C: per token, symmetric, sC = round_up_fp16(round_up_f32(max|C| / 127)),
 *     c = clamp(rint(C * (1/sC)), -127, 127).
 *   - Eigenvector signs: the largest-magnitude component is made positive
 *     (lowest channel on ties); eigenvalues descend (lower index on ties).
 *   - k-means: Lloyd iterations, Euclidean, ties to the lower centroid,
 *     empty clusters keep their previous centroid, output rounded to bf16.
 */
#include <fenv.h>
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dynamic rounding modes are honoured because the file is built with -frounding-math */

/* ------------------------------------------------------------------ */
/* number formats                                                      */
/* ------------------------------------------------------------------ */

static double bf16_val(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static float bf16_valf(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round a double to a binary format with `p` significand bits, minimum normal
 * exponent `emin` (value 2^emin) -- i.e. quantum max(2^(e-p), 2^(emin-p+1)) --
 * in the given direction: 0 nearest-even, -1 down, +1 up.  Exact in double. */
static double round_to_format(double x, int p, int emin, int dir) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e;
  frexp(x, &e); /* |x| in [2^(e-1), 2^e) */
  int qexp = e - p;
  if (qexp < emin - p + 1) qexp = emin - p + 1;
  double scaled = ldexp(x, -qexp); /* exact */
  double r;
  if (dir < 0) r = floor(scaled);
  else if (dir > 0) r = ceil(scaled);
  else r = nearbyint(scaled); /* current mode is to-nearest-even */
  return ldexp(r, qexp);
}

static uint16_t bf16_bits_of(double x) { /* x must already be a bf16 value */
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

static uint16_t bf16_rne(double x) { return bf16_bits_of(round_to_format(x, 8, -126, 0)); }

#define FP16_MAX 65504.0
static double fp16_round(double x, int dir) { return round_to_format(x, 11, -14, dir); }

static uint16_t fp16_bits_of(double v) { /* v must be an fp16 value (or +-inf) */
  uint16_t sign = (v < 0 || (v == 0 && signbit(v))) ? 0x8000 : 0;
  double a = fabs(v);
  if (isinf(a) || a > FP16_MAX) return sign | 0x7C00;
  if (a == 0) return sign;
  if (a < ldexp(1.0, -14)) return sign | (uint16_t)(a / ldexp(1.0, -24));
  int e;
  double m = frexp(a, &e); /* a = m 2^e, m in [0.5, 1) */
  uint16_t ef = (uint16_t)(e - 1 + 15);
  uint16_t mant = (uint16_t)((m * 2.0 - 1.0) * 1024.0);
  return sign | (uint16_t)(ef << 10) | mant;
}

double oracle_fp16_val(uint16_t h) {
  int e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp(1.0 + m / 1024.0, e - 15);
  return (h & 0x8000) ? -v : v;
}

static float f32_sub_up(float a, float b) {
  int old = fegetround();
  fesetround(FE_UPWARD);
  volatile float va = a, vb = b;
  volatile float r = va - vb;
  fesetround(old);
  return r;
}

static float f32_div_up(float a, float b) {
  int old = fegetround();
  fesetround(FE_UPWARD);
  volatile float va = a, vb = b;
  volatile float r = va / vb;
  fesetround(old);
  return r;
}

/* round-to-nearest float ops (default mode); volatile keeps each one a single rounding */
static float f32_sub(float a, float b) { volatile float r = a - b; return r; }
static float f32_add(float a, float b) { volatile float r = a + b; return r; }
static float f32_mul(float a, float b) { volatile float r = a * b; return r; }
static float f32_rcp(float a) { volatile float one = 1.0f; volatile float r = one / a; return r; }

/* ------------------------------------------------------------------ */
/* step 1: Query statistics  ([QWM-zh] 二阶Query统计; steps (1),(4); [QWM-en] §D.1) */
/* ------------------------------------------------------------------ */

/* S[d][d] += sum over the nq Queries of q q^T (fp64).  Incremental: no Query is kept. */
void oracle_stats_accumulate(const uint16_t *q, int64_t nq, int d, double *S) {
  double *qd = (double *)malloc(sizeof(double) * d);
  for (int64_t i = 0; i < nq; i++) {
    for (int c = 0; c < d; c++) qd[c] = bf16_val(q[i * d + c]);
    for (int a = 0; a < d; a++)
      for (int b = 0; b < d; b++) S[a * d + b] += qd[a] * qd[b];
  }
  free(qd);
}

/* Channel sensitivity weights w_c = M_cc = S_cc / N (diagonal of the second moment).
 * Cold start (N == 0): uniform w = 1 ([QWM-zh] step (1), [QWM-en] §C.3). */
void oracle_weights(const double *S, int64_t n, int d, double *w) {
  for (int c = 0; c < d; c++) w[c] = (n == 0) ? 1.0 : S[c * d + c] / (double)n;
}

/* Symmetric eigendecomposition M = U diag(lambda) U^T by the cyclic Jacobi
 * method (Golub & Van Loan, "Matrix Computations", sec. 8.5 -- two-sided
 * rotations zeroing one off-diagonal pair at a time).
 * Output: lambda[d] descending; U[c*d + k] = component c of eigenvector k.
 * Returns the number of sweeps used, or -1 when max_sweeps was not enough. */
int oracle_eig_sym(const double *M, int d, double tol_rel, int max_sweeps, double *lambda, double *U) {
  double *A = (double *)malloc(sizeof(double) * d * d);
  double *V = (double *)malloc(sizeof(double) * d * d);
  memcpy(A, M, sizeof(double) * d * d);
  for (int i = 0; i < d * d; i++) V[i] = 0.0;
  for (int i = 0; i < d; i++) V[i * d + i] = 1.0;
  double fro = 0.0;
  for (int i = 0; i < d * d; i++) fro += M[i] * M[i];
  fro = sqrt(fro);
  int sweeps = 0, converged = 0;
  for (; sweeps <= max_sweeps; sweeps++) {
    double off = 0.0;
    for (int p = 0; p < d; p++)
      for (int q = 0; q < d; q++)
        if (p != q) off += A[p * d + q] * A[p * d + q];
    if (sqrt(off) <= tol_rel * fro || fro == 0.0) { converged = 1; break; }
    if (sweeps == max_sweeps) break;
    for (int p = 0; p < d - 1; p++) {
      for (int q = p + 1; q < d; q++) {
        double apq = A[p * d + q];
        if (apq == 0.0) continue;
        double app = A[p * d + p], aqq = A[q * d + q];
        double tau = (aqq - app) / (2.0 * apq);
        double t = (tau >= 0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
        double c = 1.0 / sqrt(1.0 + t * t), s = t * c;
        /* A <- J^T A J with J = rotation in the (p, q) plane */
        for (int k = 0; k < d; k++) { /* columns p and q */
          double akp = A[k * d + p], akq = A[k * d + q];
          A[k * d + p] = c * akp - s * akq;
          A[k * d + q] = s * akp + c * akq;
        }
        for (int k = 0; k < d; k++) { /* rows p and q */
          double apk = A[p * d + k], aqk = A[q * d + k];
          A[p * d + k] = c * apk - s * aqk;
          A[q * d + k] = s * apk + c * aqk;
        }
        A[p * d + q] = 0.0;
        A[q * d + p] = 0.0;
        for (int k = 0; k < d; k++) { /* V <- V J */
          double vkp = V[k * d + p], vkq = V[k * d + q];
          V[k * d + p] = c * vkp - s * vkq;
          V[k * d + q] = s * vkp + c * vkq;
        }
      }
    }
  }
  /* order by descending eigenvalue, ties to the lower original index (stable selection) */
  int *order = (int *)malloc(sizeof(int) * d);
  char *used = (char *)calloc(d, 1);
  for (int k = 0; k < d; k++) {
    int best = -1;
    for (int i = 0; i < d; i++)
      if (!used[i] && (best < 0 || A[i * d + i] > A[best * d + best])) best = i;
    used[best] = 1;
    order[k] = best;
  }
  for (int k = 0; k < d; k++) {
    int src = order[k];
    lambda[k] = A[src * d + src];
    /* sign: largest-magnitude component positive, lowest channel on ties */
    int arg = 0;
    for (int c = 1; c < d; c++)
      if (fabs(V[c * d + src]) > fabs(V[arg * d + src])) arg = c;
    double sg = V[arg * d + src] < 0 ? -1.0 : 1.0;
    for (int c = 0; c < d; c++) U[c * d + k] = sg * V[c * d + src];
  }
  free(order);
  free(used);
  free(A);
  free(V);
  return converged ? sweeps : -1;
}

/* U_r: the first r eigenvectors rounded to bf16 (PSAC stores U_r in BF16: [QWM-ko] 어떻게 쓰나,
 * [QWM-en] §5.1).  out[c*r + k] = bf16(U[c*d + k]). */
void oracle_basis_bf16(const double *U, int d, int r, uint16_t *out) {
  for (int c = 0; c < d; c++)
    for (int k = 0; k < r; k++) out[c * r + k] = bf16_rne(U[c * d + k]);
}

/* ------------------------------------------------------------------ */
/* step 2a: k-means codebook ([QVG-ko] §2A grouping along the sequence axis; §2C warm start) */
/* ------------------------------------------------------------------ */

static double sqdist_bf16_f64(const uint16_t *x, const double *mu, int d) {
  double s = 0.0;
  for (int c = 0; c < d; c++) {
    double t = bf16_val(x[c]) - mu[c];
    s += t * t;
  }
  return s;
}

/* Lloyd's algorithm on x[n][d] (bf16) with C centroids, `iters` iterations of
 * (assign to the nearest centroid; replace each centroid by the mean of its members).
 * init == NULL: centroid j starts at token floor(j n / C); else at init[j] (bf16).
 * cent_out[C][d] bf16; optional: assign_out[n] (assignment of the last iteration),
 * obj_out[iters] (sum of squared distances at each assignment step). */
void oracle_kmeans(const uint16_t *x, int64_t n, int d, int C, const uint16_t *init, int iters,
                   uint16_t *cent_out, double *cent_f64_out, int32_t *assign_out, double *obj_out) {
  double *mu = (double *)malloc(sizeof(double) * C * d);
  double *sum = (double *)malloc(sizeof(double) * C * d);
  int64_t *cnt = (int64_t *)malloc(sizeof(int64_t) * C);
  int32_t *asg = (int32_t *)malloc(sizeof(int32_t) * (n > 0 ? n : 1));
  for (int j = 0; j < C; j++) {
    const uint16_t *src = init ? init + (int64_t)j * d : x + ((int64_t)j * n / C) * d;
    for (int c = 0; c < d; c++) mu[j * d + c] = bf16_val(src[c]);
  }
  for (int it = 0; it < iters; it++) {
    double obj = 0.0;
#pragma omp parallel for reduction(+ : obj) schedule(static)
    for (int64_t i = 0; i < n; i++) {
      int best = 0;
      double bd = sqdist_bf16_f64(x + i * d, mu, d);
      for (int j = 1; j < C; j++) {
        double dj = sqdist_bf16_f64(x + i * d, mu + (int64_t)j * d, d);
        if (dj < bd) { bd = dj; best = j; }
      }
      asg[i] = best;
      obj += bd;
    }
    if (obj_out) obj_out[it] = obj;
    memset(sum, 0, sizeof(double) * C * d);
    memset(cnt, 0, sizeof(int64_t) * C);
    for (int64_t i = 0; i < n; i++) {
      int j = asg[i];
      cnt[j]++;
      for (int c = 0; c < d; c++) sum[j * d + c] += bf16_val(x[i * d + c]);
    }
    for (int j = 0; j < C; j++)
      if (cnt[j] > 0)
        for (int c = 0; c < d; c++) mu[j * d + c] = sum[j * d + c] / (double)cnt[j];
  }
  for (int j = 0; j < C * d; j++) cent_out[j] = bf16_rne(mu[j]);
  if (cent_f64_out) memcpy(cent_f64_out, mu, sizeof(double) * C * d);
  if (assign_out) memcpy(assign_out, asg, sizeof(int32_t) * n);
  free(mu);
  free(sum);
  free(cnt);
  free(asg);
}

/* Sum over tokens of the squared distance to the nearest centroid (bf16 centroids). */
double oracle_kmeans_objective(const uint16_t *x, int64_t n, int d, const uint16_t *cent, int C) {
  double *mu = (double *)malloc(sizeof(double) * C * d);
  for (int j = 0; j < C * d; j++) mu[j] = bf16_val(cent[j]);
  double obj = 0.0;
#pragma omp parallel for reduction(+ : obj) schedule(static)
  for (int64_t i = 0; i < n; i++) {
    double bd = INFINITY;
    for (int j = 0; j < C; j++) {
      double dj = sqdist_bf16_f64(x + i * d, mu + (int64_t)j * d, d);
      if (dj < bd) bd = dj;
    }
    obj += bd;
  }
  free(mu);
  return obj;
}

/* ------------------------------------------------------------------ */
/* step 3: INT2 affine quantiser ([QWM-zh] 前置知识 "低比特KV缓存量化", step (3); [QWM-en] §D.1) */
/* ------------------------------------------------------------------ */

/* Encode one group of g float residuals.  Writes codes[g] in 0..3 and the fp16
 * bit patterns of the scale s and the offset m. */
void oracle_int2_encode_group(const float *r, int g, uint8_t *codes, uint16_t *s_bits, uint16_t *m_bits) {
  float mn = r[0], mx = r[0];
  for (int c = 1; c < g; c++) {
    if (r[c] < mn) mn = r[c];
    if (r[c] > mx) mx = r[c];
  }
  double m = fp16_round((double)mn, -1);            /* m <= min r */
  float range = f32_sub_up(mx, (float)m);             /* >= max r - m */
  double s = (range == 0.0f) ? 0.0 : fp16_round((double)f32_div_up(range, 3.0f), +1); /* >= range / 3 */
  *s_bits = fp16_bits_of(s);
  *m_bits = fp16_bits_of(m);
  if (s == 0.0) {
    for (int c = 0; c < g; c++) codes[c] = 0;
    return;
  }
  float inv = f32_rcp((float)s);
  for (int c = 0; c < g; c++) {
    float y = f32_mul(f32_sub(r[c], (float)m), inv);
    float q = nearbyintf(y); /* ties to even */
    if (q < 0.0f) q = 0.0f;
    if (q > 3.0f) q = 3.0f;
    codes[c] = (uint8_t)q;
  }
}

/* r_hat = m + s q, computed in float (s q is exact; one rounding for the sum). */
static float int2_decode(uint16_t s_bits, uint16_t m_bits, int q) {
  float s = (float)oracle_fp16_val(s_bits), m = (float)oracle_fp16_val(m_bits);
  return f32_add(m, f32_mul(s, (float)q));
}

/* Pack codes[d] (0..3) four per byte: channel 4j+t goes to bits 2t..2t+1 of byte j
 * ([QWM-zh] step (3): "INT2残差4码并1字节"). */
void oracle_pack2(const uint8_t *codes, int d, uint8_t *packed) {
  for (int j = 0; j < d / 4; j++) {
    uint8_t b = 0;
    for (int t = 0; t < 4; t++) b |= (uint8_t)((codes[4 * j + t] & 3) << (2 * t));
    packed[j] = b;
  }
}

static int unpack2(const uint8_t *packed, int c) { return (packed[c >> 2] >> (2 * (c & 3))) & 3; }

/* INT8 of one token's PSAC coefficients C[r] (fp32 in): per-token symmetric scale. */
void oracle_int8_encode_token(const float *C, int r, int8_t *c_out, uint16_t *sc_bits) {
  float a = 0.0f;
  for (int k = 0; k < r; k++)
    if (fabsf(C[k]) > a) a = fabsf(C[k]);
  double sc = (a == 0.0f) ? 0.0 : fp16_round((double)f32_div_up(a, 127.0f), +1);
  *sc_bits = fp16_bits_of(sc);
  if (sc == 0.0) {
    for (int k = 0; k < r; k++) c_out[k] = 0;
    return;
  }
  float inv = f32_rcp((float)sc);
  for (int k = 0; k < r; k++) {
    float q = nearbyintf(f32_mul(C[k], inv));
    if (q < -127.0f) q = -127.0f;
    if (q > 127.0f) q = 127.0f;
    c_out[k] = (int8_t)q;
  }
}

/* ------------------------------------------------------------------ */
/* steps 2-4 for one head of one chunk                                 */
/* ------------------------------------------------------------------ */

/* Query-aware distance d_Q(k, mu) = sum_c w_c (k_c - mu_c)^2  ([QWM-zh] 核心方法; [QWM-ko] 무엇과 다른가) */
static double dq_dist(const uint16_t *k, const uint16_t *mu, const double *w, int d) {
  double s = 0.0;
  for (int c = 0; c < d; c++) {
    double t = bf16_val(k[c]) - bf16_val(mu[c]);
    s += w[c] * t * t;
  }
  return s;
}

/* The full quadratic form of the Query-aware distance ([QWM-en] §C.4 ablation): (k - mu)^T M (k - mu). */
static double dq_dist_full(const uint16_t *k, const uint16_t *mu, const double *M, int d, double *e) {
  for (int c = 0; c < d; c++) e[c] = bf16_val(k[c]) - bf16_val(mu[c]);
  double s = 0.0;
  for (int c = 0; c < d; c++) {
    double t = 0.0;
    for (int c2 = 0; c2 < d; c2++) t += M[c * d + c2] * e[c2];
    s += e[c] * t;
  }
  return s;
}

/* QSAC score S(k, mu) = sum_g (sum_{c in G_g} w_c) R_g(k - mu)^2 with R_g = max - min of the
 * residual over the group (INT2 error estimate R_g^2 / [12 (2^b - 1)^2] with the constant dropped). */
static double qsac_score(const uint16_t *k, const uint16_t *mu, const double *w, int d, int group) {
  double S = 0.0;
  for (int g0 = 0; g0 < d; g0 += group) {
    float mn = INFINITY, mx = -INFINITY;
    double W = 0.0;
    for (int c = g0; c < g0 + group; c++) {
      float r = f32_sub(bf16_valf(k[c]), bf16_valf(mu[c]));
      if (r < mn) mn = r;
      if (r > mx) mx = r;
      W += w[c];
    }
    double R = (double)mx - (double)mn;
    S += W * R * R;
  }
  return S;
}

/* The paper's compact metadata ([QWM-zh] step (3) "组缩放INT8+FP16二级缩放"; [QWM-en] §D.1
 * "bit-packed INT2 zero-points"): r_hat = s (q - z) with an integer zero-point z in {0..3} and a step
 * s = sigma * s8, s8 an unsigned 8-bit integer and sigma a second-level scale shared, per group of
 * channels, by a tile of 128 tokens.  Readings (the pages give neither granularity nor rounding):
 * sigma is a power of two (an fp16 value), so s and every s (q - z) are exact in fp16 and fp32; each
 * (token, group) takes the zero-point whose grid [-z s, (3 - z) s] covers its residual range with the
 * smallest s (lower z on ties); sigma is the smallest power of two with 255 sigma >= the tile's
 * largest such s; s8 = ceil(s / sigma); q = clamp(rint(r (1/s) + z), 0, 3).  So |r - r_hat| <= s/2. */
#define ZP_TILE 128
static void zp_range(float a, float b, float *s_need, int *z_out) {
  *s_need = 0.0f;
  *z_out = 0;
  if (a == 0.0f && b == 0.0f) return;
  float best = INFINITY;
  for (int z = 0; z < 4; z++) {
    const float lo = (a >= 0.0f) ? 0.0f : (z > 0 ? f32_div_up(-a, (float)z) : INFINITY);
    const float hi = (b <= 0.0f) ? 0.0f : (z < 3 ? f32_div_up(b, (float)(3 - z)) : INFINITY);
    const float sz = lo > hi ? lo : hi;
    if (sz < best) { best = sz; *z_out = z; }
  }
  *s_need = best;
}
static float pow2_sigma(float smax) {
  if (smax == 0.0f) return 0.0f;
  const float t = f32_div_up(smax, 255.0f);
  int e;
  const double m = frexp((double)t, &e); /* t = m 2^e, m in [1/2, 1) */
  float sg = (m == 0.5) ? (float)ldexp(1.0, e - 1) : (float)ldexp(1.0, e);
  if (sg < 5.9604644775390625e-08f) sg = 5.9604644775390625e-08f; /* 2^-24, the smallest fp16 */
  return sg;
}
static void zp_encode_group(const float *r, int g, float s, int z, uint8_t *codes) {
  if (s == 0.0f) {
    for (int c = 0; c < g; c++) codes[c] = 0;
    return;
  }
  const float inv = f32_rcp(s);
  for (int c = 0; c < g; c++) {
    float q = nearbyintf(f32_add(f32_mul(r[c], inv), (float)z));
    if (q < 0.0f) q = 0.0f;
    if (q > 3.0f) q = 3.0f;
    codes[c] = (uint8_t)q;
  }
}

typedef struct {
  /* inputs */
  const uint16_t *k, *v;          /* [n][d] bf16 */
  const uint16_t *cent_k, *cent_v;/* [C][d] bf16 */
  const double *w;                /* [d] or NULL (uniform) */
  const double *M_full;           /* [d][d] or NULL: rank the top-M candidates by (k - mu)^T M (k - mu)
                                     ([QWM-en] §C.4); w must then be diag(M) (the range score keeps w) */
  const uint16_t *u_r;            /* [d][rank] bf16 or NULL (PSAC off) */
  const double *u_r_f64;          /* optional [d][rank] double basis used instead of u_r (exactness checks) */
  const int32_t *force_idx_k;     /* [n] or NULL: use these Key centroids instead of QSAC */
  const int32_t *force_idx_v;     /* [n] or NULL */
  int64_t n;
  int32_t d, C, group, top_m, rank;
  int32_t storage;                /* 0: fp16 step and offset per group; 1: the compact metadata */
  int32_t psac_gate;              /* 1: keep C only where it lowers sum_c w_c e_c^2 ([QWM-zh] step (4)) */
  /* outputs */
  int32_t *idx_k, *idx_v;         /* [n] */
  uint8_t *k_codes, *v_codes;     /* [n][d/4] */
  uint16_t *k_scale, *k_min, *v_scale, *v_min; /* fp16 [n][d/group] */
  int8_t *c;                      /* [n][rank] (when u_r) */
  uint16_t *c_scale;              /* fp16 [n] (when u_r) */
  double *c_real;                 /* optional [n][rank]: C before INT8 */
  int32_t *cand;                  /* optional [n][top_m]: candidates, ascending d_Q */
  double *score2;                 /* optional [n][2]: best and second-best S over the candidates */
  double *dq_edge;                /* optional [n][2]: the M-th and (M+1)-th smallest d_Q */
  double *vdist2;                 /* optional [n][2]: best and second-best Value distance */
  uint8_t *k_s8, *v_s8;           /* storage 1: [n][d/group] steps */
  uint8_t *k_zp, *v_zp;           /* storage 1: [n] zero-points, group g in bits 2g..2g+1 */
  uint16_t *k_sigma, *v_sigma;    /* storage 1: fp16 [ceil(n/128)][d/group] second-level scales */
  double *gate_err;               /* optional [n][2]: w-weighted error without and with C */
} oracle_quant_args;

/* Step 4 for one token: C = E U_r with E = K - K_hat_0 (double accumulation), INT8 per token; with
 * the gate, C is kept only when sum_c w_c (E_c - (C_hat U_r^T)_c)^2 < sum_c w_c E_c^2 (C_hat the
 * decoded INT8 coefficients), else stored as zeros with a zero scale. */
static void psac_token(const oracle_quant_args *a, int64_t i, const uint16_t *k, const float *khat0,
                       const double *w, float *Cf) {
  const int d = a->d, r = a->rank;
  for (int kk = 0; kk < r; kk++) {
    double acc = 0.0;
    for (int c = 0; c < d; c++) {
      double e = (double)bf16_valf(k[c]) - (double)khat0[c];
      acc += e * (a->u_r_f64 ? a->u_r_f64[c * r + kk] : bf16_val(a->u_r[c * r + kk]));
    }
    if (a->c_real) a->c_real[i * r + kk] = acc;
    Cf[kk] = (float)acc;
  }
  oracle_int8_encode_token(Cf, r, a->c + i * r, a->c_scale + i);
  if (a->psac_gate || a->gate_err) {
    const double sc = oracle_fp16_val(a->c_scale[i]);
    double e0 = 0.0, e1 = 0.0;
    for (int c = 0; c < d; c++) {
      const double e = (double)bf16_valf(k[c]) - (double)khat0[c];
      double corr = 0.0;
      for (int kk = 0; kk < r; kk++)
        corr += sc * (double)a->c[i * r + kk] * (a->u_r_f64 ? a->u_r_f64[c * r + kk] : bf16_val(a->u_r[c * r + kk]));
      e0 += w[c] * e * e;
      e1 += w[c] * (e - corr) * (e - corr);
    }
    if (a->gate_err) { a->gate_err[2 * i] = e0; a->gate_err[2 * i + 1] = e1; }
    if (a->psac_gate && !(e1 < e0)) {
      for (int kk = 0; kk < r; kk++) a->c[i * r + kk] = 0;
      a->c_scale[i] = 0;
    }
  }
}

void oracle_quantize_head(const oracle_quant_args *a) {
  const int d = a->d, C = a->C, G = d / a->group, M = a->top_m, r = a->rank;
  const int compact = a->storage == 1;
  double *w = (double *)malloc(sizeof(double) * d);
  for (int c = 0; c < d; c++) w[c] = a->w ? a->w[c] : 1.0;
  /* compact metadata: per (token, K/V, group) the needed step and zero-point, then sigma per tile */
  float *s_need = compact ? (float *)malloc(sizeof(float) * (size_t)(a->n > 0 ? a->n : 1) * 2 * G) : NULL;
  int *zp = compact ? (int *)malloc(sizeof(int) * (size_t)(a->n > 0 ? a->n : 1) * 2 * G) : NULL;
#pragma omp parallel
  {
    double *dq = (double *)malloc(sizeof(double) * C);
    int *sel = (int *)malloc(sizeof(int) * (M + 1));
    float *res = (float *)malloc(sizeof(float) * d);
    uint8_t *codes = (uint8_t *)malloc(d);
    float *khat0 = (float *)malloc(sizeof(float) * d);
    float *Cf = (float *)malloc(sizeof(float) * (r > 0 ? r : 1));
    double *khat0_e = (double *)malloc(sizeof(double) * d); /* scratch of the full-form distance */
#pragma omp for schedule(static)
    for (int64_t i = 0; i < a->n; i++) {
      const uint16_t *k = a->k + i * d, *v = a->v + i * d;
      int jk;
      /* ---- step 2: QSAC Key centroid ---- */
      for (int j = 0; j < C; j++)
        dq[j] = a->M_full ? dq_dist_full(k, a->cent_k + (int64_t)j * d, a->M_full, d, (double *)khat0_e)
                          : dq_dist(k, a->cent_k + (int64_t)j * d, w, d);
      int nsel = (M + 1 <= C) ? M + 1 : C;
      for (int t = 0; t < nsel; t++) { /* t-th smallest d_Q, ties to the lower index */
        int best = -1;
        for (int j = 0; j < C; j++) {
          int taken = 0;
          for (int u = 0; u < t; u++) taken |= (sel[u] == j);
          if (!taken && (best < 0 || dq[j] < dq[best])) best = j;
        }
        sel[t] = best;
      }
      int ncand = (M <= C) ? M : C;
      int bj = -1;
      double bs = INFINITY, s2 = INFINITY;
      for (int t = 0; t < ncand; t++) {
        int j = sel[t];
        double S = qsac_score(k, a->cent_k + (int64_t)j * d, w, d, a->group);
        if (S < bs || (S == bs && j < bj)) { s2 = bs; bs = S; bj = j; }
        else if (S < s2) s2 = S;
      }
      if (a->cand) for (int t = 0; t < M; t++) a->cand[i * M + t] = (t < ncand) ? sel[t] : -1;
      if (a->score2) { a->score2[2 * i] = bs; a->score2[2 * i + 1] = s2; }
      if (a->dq_edge) {
        a->dq_edge[2 * i] = dq[sel[ncand - 1]];
        a->dq_edge[2 * i + 1] = (nsel > ncand) ? dq[sel[ncand]] : INFINITY;
      }
      jk = a->force_idx_k ? a->force_idx_k[i] : bj;
      a->idx_k[i] = jk;
      /* ---- Values: nearest centroid, as in QVG ---- */
      int jv = 0;
      double bv = INFINITY, bv2 = INFINITY;
      for (int j = 0; j < C; j++) {
        double s = 0.0;
        const uint16_t *mu = a->cent_v + (int64_t)j * d;
        for (int c = 0; c < d; c++) {
          double t = bf16_val(v[c]) - bf16_val(mu[c]);
          s += t * t;
        }
        if (s < bv) { bv2 = bv; bv = s; jv = j; }
        else if (s < bv2) bv2 = s;
      }
      if (a->vdist2) { a->vdist2[2 * i] = bv; a->vdist2[2 * i + 1] = bv2; }
      if (a->force_idx_v) jv = a->force_idx_v[i];
      a->idx_v[i] = jv;
      /* ---- step 3: INT2 residuals, Keys then Values ---- */
      for (int pass = 0; pass < 2; pass++) {
        const uint16_t *x = pass ? v : k;
        const uint16_t *mu = pass ? a->cent_v + (int64_t)jv * d : a->cent_k + (int64_t)jk * d;
        for (int c = 0; c < d; c++) res[c] = f32_sub(bf16_valf(x[c]), bf16_valf(mu[c]));
        if (compact) { /* the residual ranges only; the codes follow once sigma is known */
          for (int g = 0; g < G; g++) {
            float mn = res[g * a->group], mx = mn;
            for (int c = 1; c < a->group; c++) {
              const float t = res[g * a->group + c];
              if (t < mn) mn = t;
              if (t > mx) mx = t;
            }
            zp_range(mn, mx, &s_need[(i * 2 + pass) * G + g], &zp[(i * 2 + pass) * G + g]);
          }
          continue;
        }
        uint8_t *packed = (pass ? a->v_codes : a->k_codes) + i * (d / 4);
        uint16_t *sc = (pass ? a->v_scale : a->k_scale) + i * G;
        uint16_t *mn = (pass ? a->v_min : a->k_min) + i * G;
        for (int g = 0; g < G; g++)
          oracle_int2_encode_group(res + g * a->group, a->group, codes + g * a->group, sc + g, mn + g);
        oracle_pack2(codes, d, packed);
        if (pass == 0) /* K_hat_0 = mu + r_hat, float */
          for (int c = 0; c < d; c++) {
            int g = c / a->group;
            khat0[c] = f32_add(bf16_valf(mu[c]), int2_decode(sc[g], mn[g], codes[c]));
          }
      }
      /* ---- step 4: PSAC ---- */
      if (!compact && (a->u_r || a->u_r_f64) && r > 0) psac_token(a, i, k, khat0, w, Cf);
    }
#pragma omp barrier
    if (compact) {
      /* second-level scales: per tile of 128 tokens and group, the power of two for the largest step */
#pragma omp for schedule(static)
      for (int64_t tg = 0; tg < (a->n + ZP_TILE - 1) / ZP_TILE; tg++)
        for (int pass = 0; pass < 2; pass++)
          for (int g = 0; g < G; g++) {
            float smax = 0.0f;
            for (int64_t i = tg * ZP_TILE; i < a->n && i < (tg + 1) * ZP_TILE; i++)
              if (s_need[(i * 2 + pass) * G + g] > smax) smax = s_need[(i * 2 + pass) * G + g];
            (pass ? a->v_sigma : a->k_sigma)[tg * G + g] = fp16_bits_of((double)pow2_sigma(smax));
          }
#pragma omp for schedule(static)
      for (int64_t i = 0; i < a->n; i++) {
        const uint16_t *k = a->k + i * d, *v = a->v + i * d;
        for (int pass = 0; pass < 2; pass++) {
          const uint16_t *x = pass ? v : k;
          const int j = pass ? a->idx_v[i] : a->idx_k[i];
          const uint16_t *mu = (pass ? a->cent_v : a->cent_k) + (int64_t)j * d;
          uint8_t zbits = 0;
          for (int c = 0; c < d; c++) res[c] = f32_sub(bf16_valf(x[c]), bf16_valf(mu[c]));
          for (int g = 0; g < G; g++) {
            const float sg = (float)oracle_fp16_val((pass ? a->v_sigma : a->k_sigma)[(i / ZP_TILE) * G + g]);
            const float need = s_need[(i * 2 + pass) * G + g];
            const int z = zp[(i * 2 + pass) * G + g];
            const int s8 = (need == 0.0f) ? 0 : (int)ceilf(need / sg); /* exact: sigma is a power of two */
            const float s = sg * (float)s8;                             /* exact */
            (pass ? a->v_s8 : a->k_s8)[i * G + g] = (uint8_t)s8;
            zbits |= (uint8_t)(z << (2 * g));
            zp_encode_group(res + g * a->group, a->group, s, z, codes + g * a->group);
            if (pass == 0)
              for (int c = g * a->group; c < (g + 1) * a->group; c++)
                khat0[c] = f32_add(bf16_valf(mu[c]), s * (float)((int)codes[c] - z)); /* s (q - z) exact */
          }
          (pass ? a->v_zp : a->k_zp)[i] = zbits;
          oracle_pack2(codes, d, (pass ? a->v_codes : a->k_codes) + i * (d / 4));
        }
        if ((a->u_r || a->u_r_f64) && r > 0) psac_token(a, i, k, khat0, w, Cf);
      }
    }
    free(dq);
    free(sel);
    free(res);
    free(codes);
    free(khat0);
    free(Cf);
    free(khat0_e);
  }
  free(w);
  free(s_need);
  free(zp);
}

/* ------------------------------------------------------------------ */
/* step 5: attention over the compressed cache, and the BF16 decoder     */
/* ([QWM-zh] logits L = Q K^T / sqrt(d); PSAC form Q K_hat_0^T + (Q U_r) C^T; step (5)) */
/* ------------------------------------------------------------------ */

typedef struct {
  int64_t n;
  int32_t rank; /* 0: no PSAC term */
  const int32_t *idx_k, *idx_v;
  const uint8_t *k_codes, *v_codes;
  const uint16_t *k_scale, *k_min, *v_scale, *v_min;
  const uint16_t *cent_k, *cent_v;
  const int8_t *c;
  const uint16_t *c_scale;
  const uint16_t *u_r; /* [d][rank] */
  /* The chunk still being generated, kept in bf16 ([QWM-en] §5.1, §D.1: a chunk is quantised once
   * it is complete): k_raw != NULL makes every field above except n unused; keys are k_raw[j],
   * values v_raw[j].  causal_tpf > 0 adds the block-causal mask of frames of causal_tpf tokens:
   * the Query in row q (token q of this chunk) sees key j only when j / tpf <= q / tpf. */
  const uint16_t *k_raw, *v_raw; /* [n][d] bf16 */
  int64_t causal_tpf;
  /* 1: cent_k / cent_v hold the chunk's stored codebooks as fp16 bit patterns (the fp16 value of
   * each bf16 centroid element) instead of the bf16 codebooks; decoding uses the values given. */
  int32_t cent_fp16;
} oracle_chunk_head;

static double centroid_val(const oracle_chunk_head *ch, uint16_t b) {
  return ch->cent_fp16 ? oracle_fp16_val(b) : bf16_val(b);
}

/* dequantised Key base k_hat_0 = mu_idx + r_hat and Value v_hat, as doubles */
static void decode_token(const oracle_chunk_head *ch, int d, int group, int64_t j, double *kh0, double *vh) {
  if (ch->k_raw) {
    for (int c = 0; c < d; c++) {
      kh0[c] = bf16_val(ch->k_raw[j * d + c]);
      vh[c] = bf16_val(ch->v_raw[j * d + c]);
    }
    return;
  }
  const int G = d / group;
  const uint16_t *muk = ch->cent_k + (int64_t)ch->idx_k[j] * d;
  const uint16_t *muv = ch->cent_v + (int64_t)ch->idx_v[j] * d;
  for (int c = 0; c < d; c++) {
    int g = c / group;
    kh0[c] = centroid_val(ch, muk[c]) + (double)int2_decode(ch->k_scale[j * G + g], ch->k_min[j * G + g],
                                                            unpack2(ch->k_codes + j * (d / 4), c));
    vh[c] = centroid_val(ch, muv[c]) + (double)int2_decode(ch->v_scale[j * G + g], ch->v_min[j * G + g],
                                                           unpack2(ch->v_codes + j * (d / 4), c));
  }
}

/* For each listed query row, o = softmax(l) V_hat over every token of every chunk, with
 * l_j = scale * (q . k_hat_0_j + (q U_r^(chunk)) . c_hat_j),  c_hat = sC * c.
 * Softmax in double with the running maximum subtracted.  out[rows][d] double.  lse (may be NULL):
 * [rows] double, the base-2 log of sum_j exp(l_j) = (lmax + ln(sum_j exp(l_j - lmax))) / ln 2. */
void oracle_attend_rows(const uint16_t *q, int d, int group, const int64_t *rows, int64_t n_rows,
                        const oracle_chunk_head *chunks, int n_chunks, double scale, double *out, double *lse) {
  int64_t total = 0;
  for (int t = 0; t < n_chunks; t++) total += chunks[t].n;
#pragma omp parallel
  {
    double *l = (double *)malloc(sizeof(double) * (total > 0 ? total : 1));
    double *kh0 = (double *)malloc(sizeof(double) * d);
    double *vh = (double *)malloc(sizeof(double) * d);
    double *qd = (double *)malloc(sizeof(double) * d);
    double *qu = (double *)malloc(sizeof(double) * 64);
#pragma omp for schedule(dynamic, 1)
    for (int64_t ri = 0; ri < n_rows; ri++) {
      const uint16_t *qq = q + rows[ri] * d;
      for (int c = 0; c < d; c++) qd[c] = bf16_val(qq[c]);
      double lmax = -INFINITY;
      int64_t off = 0;
      for (int t = 0; t < n_chunks; t++) {
        const oracle_chunk_head *ch = &chunks[t];
        for (int kk = 0; kk < ch->rank; kk++) {
          double s = 0.0;
          for (int c = 0; c < d; c++) s += qd[c] * bf16_val(ch->u_r[c * ch->rank + kk]);
          qu[kk] = s;
        }
        for (int64_t j = 0; j < ch->n; j++) {
          if (ch->k_raw && ch->causal_tpf > 0 && j / ch->causal_tpf > rows[ri] / ch->causal_tpf) {
            l[off + j] = -INFINITY; /* a later frame of the chunk being generated */
            continue;
          }
          decode_token(ch, d, group, j, kh0, vh);
          double s = 0.0;
          for (int c = 0; c < d; c++) s += qd[c] * kh0[c];
          if (ch->rank > 0) {
            double sc = oracle_fp16_val(ch->c_scale[j]);
            for (int kk = 0; kk < ch->rank; kk++) s += qu[kk] * (sc * (double)ch->c[j * ch->rank + kk]);
          }
          l[off + j] = scale * s;
          if (l[off + j] > lmax) lmax = l[off + j];
        }
        off += ch->n;
      }
      double *o = out + ri * d;
      for (int c = 0; c < d; c++) o[c] = 0.0;
      double denom = 0.0;
      off = 0;
      for (int t = 0; t < n_chunks; t++) {
        const oracle_chunk_head *ch = &chunks[t];
        for (int64_t j = 0; j < ch->n; j++) {
          if (l[off + j] == -INFINITY) continue;
          double p = exp(l[off + j] - lmax);
          denom += p;
          decode_token(ch, d, group, j, kh0, vh);
          for (int c = 0; c < d; c++) o[c] += p * vh[c];
        }
        off += ch->n;
      }
      for (int c = 0; c < d; c++) o[c] /= denom;
      if (lse) lse[ri] = (lmax + log(denom)) / log(2.0);
    }
    free(l);
    free(kh0);
    free(vh);
    free(qd);
    free(qu);
  }
}

/* BF16 reconstruction of one head of one chunk ([QWM-zh] step (5) fused decoder semantics):
 * K_hat = K_hat_0 + c_hat U_r^T, V_hat = mu^V_idx + r_hat; optional double outputs. */
void oracle_dequantize_head(const oracle_chunk_head *ch, int d, int group, uint16_t *k_hat, uint16_t *v_hat,
                            double *k_hat_f64, double *v_hat_f64) {
#pragma omp parallel
  {
    double *kh0 = (double *)malloc(sizeof(double) * d);
    double *vh = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(static)
    for (int64_t j = 0; j < ch->n; j++) {
      decode_token(ch, d, group, j, kh0, vh);
      for (int c = 0; c < d; c++) {
        double kv = kh0[c];
        if (ch->rank > 0) {
          double sc = oracle_fp16_val(ch->c_scale[j]);
          for (int kk = 0; kk < ch->rank; kk++)
            kv += sc * (double)ch->c[j * ch->rank + kk] * bf16_val(ch->u_r[c * ch->rank + kk]);
        }
        if (k_hat) k_hat[j * d + c] = bf16_rne(kv);
        if (v_hat) v_hat[j * d + c] = bf16_rne(vh[c]);
        if (k_hat_f64) k_hat_f64[j * d + c] = kv;
        if (v_hat_f64) v_hat_f64[j * d + c] = vh[c];
      }
    }
    free(kh0);
    free(vh);
  }
}

/* ------------------------------------------------------------------ */
/* comparison baselines of the ablation workload                        */
/* ------------------------------------------------------------------ */

/* QVG progressive residual quantisation ([QVG-ko] §2B), stage residual: the next stage quantises
 * r = x - mu_idx, computed in float and rounded to bf16 (nearest-even) so that it can be fed to
 * the next stage's k-means and quantiser like the tokens themselves.  x, cent: bf16 bits. */
void oracle_prq_residual(const uint16_t *x, int64_t n, int d, const uint16_t *cent, const int32_t *idx,
                         uint16_t *out) {
  for (int64_t t = 0; t < n; t++)
    for (int c = 0; c < d; c++) {
      volatile float a = (float)bf16_val(x[t * d + c]), b = (float)bf16_val(cent[(int64_t)idx[t] * d + c]);
      volatile float r = a - b;
      out[t * d + c] = bf16_rne((double)r);
    }
}

/* KIVI-style INT2 ([QWM-ko] "전제와 한계": finer groups; the ablation workload's reading):
 * Keys per channel over groups of g consecutive tokens (the last group may be shorter), Values
 * per token over groups of g consecutive channels; the same affine INT2 encoder as the QuantWM
 * residuals, applied to the raw values.  Codes are packed per token like the QuantWM codes.
 *   k_scale, k_min: fp16 [ceil(n/g)][d];  v_scale, v_min: fp16 [n][d/g]. */
void oracle_kivi_quantize_head(const uint16_t *k, const uint16_t *v, int64_t n, int d, int g, uint8_t *k_codes,
                               uint16_t *k_scale, uint16_t *k_min, uint8_t *v_codes, uint16_t *v_scale,
                               uint16_t *v_min) {
  float *r = (float *)malloc(sizeof(float) * (size_t)(g > d ? g : d));
  uint8_t *q = (uint8_t *)malloc((size_t)(g > d ? g : d));
  uint8_t *codes = (uint8_t *)calloc((size_t)(n > 0 ? n : 1) * d, 1);
  const int64_t ng = (n + g - 1) / g;
  for (int64_t tg = 0; tg < ng; tg++) {
    const int len = (int)((n - tg * g) < g ? (n - tg * g) : g);
    for (int c = 0; c < d; c++) {
      for (int t = 0; t < len; t++) r[t] = (float)bf16_val(k[(tg * g + t) * d + c]);
      oracle_int2_encode_group(r, len, q, &k_scale[tg * d + c], &k_min[tg * d + c]);
      for (int t = 0; t < len; t++) codes[(tg * g + t) * d + c] = q[t];
    }
  }
  for (int64_t t = 0; t < n; t++) oracle_pack2(codes + t * d, d, k_codes + t * (d / 4));
  for (int64_t t = 0; t < n; t++) {
    for (int cg = 0; cg < d / g; cg++) {
      for (int c = 0; c < g; c++) r[c] = (float)bf16_val(v[t * d + cg * g + c]);
      oracle_int2_encode_group(r, g, q, &v_scale[t * (d / g) + cg], &v_min[t * (d / g) + cg]);
      for (int c = 0; c < g; c++) codes[t * d + cg * g + c] = q[c];
    }
    oracle_pack2(codes + t * d, d, v_codes + t * (d / 4));
  }
  free(r);
  free(q);
  free(codes);
}

/* KIVI-style decode: x_hat = m + s q per element (float, as for the residuals), as doubles. */
void oracle_kivi_dequantize_head(const uint8_t *k_codes, const uint16_t *k_scale, const uint16_t *k_min,
                                 const uint8_t *v_codes, const uint16_t *v_scale, const uint16_t *v_min, int64_t n,
                                 int d, int g, double *k_hat, double *v_hat) {
  for (int64_t t = 0; t < n; t++)
    for (int c = 0; c < d; c++) {
      const int64_t kg = (t / g) * d + c, vg = t * (d / g) + c / g;
      k_hat[t * d + c] = (double)int2_decode(k_scale[kg], k_min[kg], unpack2(k_codes + t * (d / 4), c));
      v_hat[t * d + c] = (double)int2_decode(v_scale[vg], v_min[vg], unpack2(v_codes + t * (d / 4), c));
    }
}

/* Small helpers exported for the oracle's own tests. */
double oracle_round_fp16(double x, int dir) { return fp16_round(x, dir); }
uint16_t oracle_fp16_bits(double v) { return fp16_bits_of(v); }
uint16_t oracle_bf16_rne(double x) { return bf16_rne(x); }
