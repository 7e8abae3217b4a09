/* CPU oracle of one int4 routed-expert MoE layer.  TEST INFRASTRUCTURE ONLY (see oracle.h
 * for the page citations, the canonical fp32 arithmetic and the pins).
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp (no -ffast-math): every fp32 expression below
 * rounds exactly as written, and fmaf() is used wherever the canonical arithmetic says fma.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QB 32 /* activation block length (Q8_0-style blocks of 32) */


int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* threads the parallel loops use from now on (n >= 1); the results do not depend on it */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------------------------------
 * Formats.  P1 §3.1 "int4 packed": two 4-bit values per byte, one f32 scale per row.
 * Readings (the pages are silent): symmetric scale s = max|w| / 7, codes round(w/s) clamped to
 * [-7, 7] (half away from zero), two's-complement nibbles, element 2i in the low nibble and
 * element 2i+1 in the high nibble, rows stored one after another.
 * ---------------------------------------------------------------------------------------- */
int orc_i4_get(const uint8_t* row, int j) {
  int byte = row[j >> 1];
  int nib = (j & 1) ? (byte >> 4) : (byte & 15);
  return nib >= 8 ? nib - 16 : nib;
}

void orc_pack_i4_row(const int8_t* q, int cols, uint8_t* packed_row) {
  for (int i = 0; i < cols / 2; ++i)
    packed_row[i] = (uint8_t)((q[2 * i] & 15) | ((q[2 * i + 1] & 15) << 4));
}

void orc_quantize_i4_rows(const float* w, int64_t rows, int cols, uint8_t* packed, float* scales) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const float* wr = w + r * cols;
    float amax = 0.0f;
    for (int j = 0; j < cols; ++j) {
      float a = fabsf(wr[j]);
      if (a > amax) amax = a;
    }
    float s = amax / 7.0f;
    int8_t* q = (int8_t*)malloc((size_t)cols);
    for (int j = 0; j < cols; ++j) {
      int v = 0;
      if (s != 0.0f) {
        float t = roundf(wr[j] / s);
        v = (int)t;
        if (v > 7) v = 7;
        if (v < -7) v = -7;
      }
      q[j] = (int8_t)v;
    }
    orc_pack_i4_row(q, cols, packed + r * (cols / 2));
    free(q);
    scales[r] = s;
  }
}

/* ------------------------------------------------------------------------------------------
 * Activation quantisation.  P1 §3.1 IDOT path: decode activations are quantised to int8;
 * P3 "Что реализовано": Q8_0-style int8 activations.  Per block of 32: d = max|x| / 127,
 * q = round(x / d) clamped to [-127, 127]; an all-zero block gets d = 0 and q = 0.
 * ---------------------------------------------------------------------------------------- */
void orc_quantize_q8(const float* x, int64_t n, int8_t* q, float* d) {
  for (int64_t b = 0; b < n / QB; ++b) {
    const float* xb = x + b * QB;
    float amax = 0.0f;
    for (int j = 0; j < QB; ++j) {
      float a = fabsf(xb[j]);
      if (a > amax) amax = a;
    }
    float db = amax / 127.0f;
    for (int j = 0; j < QB; ++j) {
      int v = 0;
      if (db != 0.0f) {
        v = (int)roundf(xb[j] / db);
        if (v > 127) v = 127;
        if (v < -127) v = -127;
      }
      q[b * QB + j] = (int8_t)v;
    }
    d[b] = db;
  }
}

/* ------------------------------------------------------------------------------------------
 * Own fp32 exp, written from the mathematics: exp(x) = 2^k * exp(r), k = nearest integer to
 * x / ln2, r = x - k*ln2 by Cody-Waite reduction with ln2 split in two floats (the high part
 * has 12 fractional bits so k*hi is exact), exp(r) by its degree-7 Taylor polynomial in
 * Horner form (|r| <= ln2/2, truncation below 0.05 ulp), and an exact scaling by 2^k done in
 * two halves so that only a subnormal result rounds.
 * ---------------------------------------------------------------------------------------- */
static float pow2i(int k) { /* 2^k for -126 <= k <= 127 */
  union { uint32_t u; float f; } v;
  v.u = (uint32_t)(k + 127) << 23;
  return v.f;
}

float orc_exp(float x) {
  if (x != x) return x + x;
  if (x > 89.0f) return INFINITY;
  if (x < -104.0f) return 0.0f;
  const float log2e = 0x1.715476p+0f;   /* 1/ln2 rounded to fp32 */
  const float ln2_hi = 0x1.62ep-1f;     /* ln2 truncated to 12 fractional bits */
  const float ln2_lo = 0x1.0bfbe8p-15f; /* fp32(ln2 - ln2_hi) */
  const float shifter = 12582912.0f;    /* 1.5 * 2^23: (t + c) - c rounds t to an integer */
  float t = x * log2e;
  float kf = (t + shifter) - shifter;
  float r = fmaf(-kf, ln2_hi, x);
  r = fmaf(-kf, ln2_lo, r);
  float p = 0x1.a01a02p-13f;     /* 1/7! */
  p = fmaf(p, r, 0x1.6c16c2p-10f); /* 1/6! */
  p = fmaf(p, r, 0x1.111112p-7f);  /* 1/5! */
  p = fmaf(p, r, 0x1.555556p-5f); /* 1/4! */
  p = fmaf(p, r, 0x1.555556p-3f);  /* 1/3! */
  p = fmaf(p, r, 0.5f);            /* 1/2! */
  p = fmaf(p, r, 1.0f);            /* 1/1! */
  p = fmaf(p, r, 1.0f);            /* 1/0! */
  int k = (int)kf;
  int k1 = k / 2, k2 = k - k1;
  return (p * pow2i(k1)) * pow2i(k2);
}

void orc_exp_n(const float* x, float* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_exp(x[i]);
}

float orc_sigmoid(float x) { return 1.0f / (1.0f + orc_exp(-x)); }

/* SwiGLU element: SiLU(g) * u with SiLU(g) = g / (1 + exp(-g)) */
float orc_silu_mul(float g, float u) {
  float s = g / (1.0f + orc_exp(-g));
  return s * u;
}

float orc_pairwise32(const float* p) {
  float v[32];
  for (int i = 0; i < 32; ++i) v[i] = p[i];
  for (int n = 16; n >= 1; n /= 2)
    for (int i = 0; i < n; ++i) v[i] = v[2 * i] + v[2 * i + 1];
  return v[0];
}

float orc_canon_dot(const float* a, const float* b, int n) {
  int G = (n + 31) / 32;
  float p[32];
  for (int g = 0; g < 32; ++g) {
    p[g] = 0.0f;
    for (int j = g * G; j < (g + 1) * G && j < n; ++j) {
      p[g] = fmaf(a[j], b[j], p[g]);
    }
  }
  return orc_pairwise32(p);
}

float orc_canon_blocksum(const float* d, const int32_t* A, int nb) {
  int G = (nb + 31) / 32;
  float p[32];
  for (int g = 0; g < 32; ++g) {
    p[g] = 0.0f;
    for (int b = g * G; b < (g + 1) * G && b < nb; ++b) p[g] = fmaf(d[b], (float)A[b], p[g]);
  }
  return orc_pairwise32(p);
}

/* ------------------------------------------------------------------------------------------
 * Integer dot of block b (32 elements) of an int4 row with int8 activation codes:
 * P1 §4 kernel layer, dot_i4i8.  Exact in int32: |sum| <= 32*8*127.
 * ---------------------------------------------------------------------------------------- */
int32_t orc_block_dot(const uint8_t* wrow, const int8_t* qx, int b) {
  int32_t acc = 0;
  for (int j = b * QB; j < (b + 1) * QB; ++j) acc += orc_i4_get(wrow, j) * (int32_t)qx[j];
  return acc;
}

/* out[r] = s[r] * canon_blocksum(dx, A[r, :]),  A[r,b] = block_dot(row r, b).
 * Dequant-on-use: the int4 matrix is never expanded (P1 §3.1). */
void orc_i4_matvec(const uint8_t* W, const float* s, int rows, int cols, const int8_t* qx,
                   const float* dx, float* out, int32_t* A) {
  const int nb = cols / QB;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    int32_t* Ar = (int32_t*)malloc(sizeof(int32_t) * (size_t)nb);
    const uint8_t* wrow = W + (int64_t)r * (cols / 2);
    for (int b = 0; b < nb; ++b) Ar[b] = orc_block_dot(wrow, qx, b);
    out[r] = s[r] * orc_canon_blocksum(dx, Ar, nb);
    if (A) memcpy(A + (int64_t)r * nb, Ar, sizeof(int32_t) * (size_t)nb);
    free(Ar);
  }
}

/* ------------------------------------------------------------------------------------------
 * int8 rows.  P1 §3.1: "int8 (dense and MTP-head precision)", one value per byte
 * (quantize_rows), and the IDOT fast path's integer dot of int8 weights with int8 activation
 * codes (dot_i8i8).  Reading (the pages say no more): one f32 scale per row, symmetric
 * s = max|w| / 127, code = round(w / s) half away from zero clamped to [-127, 127], as for the
 * int4 rows and the activation blocks; an all-zero row has s = 0 and codes 0.
 * ---------------------------------------------------------------------------------------- */
void orc_quantize_i8_rows(const float* w, int64_t rows, int cols, int8_t* q, float* scales) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const float* wr = w + r * cols;
    float amax = 0.0f;
    for (int j = 0; j < cols; ++j) {
      float a = fabsf(wr[j]);
      if (a > amax) amax = a;
    }
    const float s = amax / 127.0f;
    const int lim = 127;
    for (int j = 0; j < cols; ++j) {
      int v = 0;
      if (s != 0.0f) {
        v = (int)roundf(wr[j] / s);
        if (v > lim) v = lim;
        if (v < -lim) v = -lim;
      }
      q[r * cols + j] = (int8_t)v;
    }
    scales[r] = s;
  }
}

/* Integer dot of block b (32 elements) of an int8 row with int8 activation codes; exact in
 * int32: |sum| <= 32 * 127 * 127. */
int32_t orc_i8_block_dot(const int8_t* wrow, const int8_t* qx, int b) {
  int32_t acc = 0;
  const int end = (b + 1) * QB;
  for (int j = b * QB; j < end; ++j) acc += (int32_t)wrow[j] * (int32_t)qx[j];
  return acc;
}

/* out[r] = s[r] * canon_blocksum(dx, A[r, :]) with A[r,b] = i8_block_dot(row r, b): the int8
 * counterpart of orc_i4_matvec (same canonical fp32 epilogue). */
void orc_i8_matvec(const int8_t* W, const float* s, int rows, int cols, const int8_t* qx,
                   const float* dx, float* out, int32_t* A) {
  const int nb = cols / QB;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    int32_t* Ar = (int32_t*)malloc(sizeof(int32_t) * (size_t)nb);
    const int8_t* wrow = W + (int64_t)r * cols;
    for (int b = 0; b < nb; ++b) Ar[b] = orc_i8_block_dot(wrow, qx, b);
    out[r] = s[r] * orc_canon_blocksum(dx, Ar, nb);
    if (A) memcpy(A + (int64_t)r * nb, Ar, sizeof(int32_t) * (size_t)nb);
    free(Ar);
  }
}

/* ------------------------------------------------------------------------------------------
 * int2 rows.  P1 §3.1 "int2 packed (experimental)": four 2-bit values per byte (pack_int2),
 * used by matmul_i2 with dequant-on-use.  Readings (the pages say no more):
 *   - one f32 scale per row and symmetric codes, as for int4: s = max|w| / 1 (the largest
 *     symmetric 2-bit code is 1, as 7 is for 4 bits), code = round(w / s) half away from zero
 *     clamped to [-1, 1]; an all-zero row has s = 0 and codes 0;
 *   - two's-complement 2-bit fields; the pattern 10 (-2) is never written but decodes;
 *   - element 4i+k in bits 2k..2k+1 of byte i (lowest bits first, as the int4 low nibble);
 *   - the matvec takes the int4 rows' IDOT route: int8 activation codes in blocks of 32,
 *     exact int32 block dots, the same canonical fp32 epilogue.
 * ---------------------------------------------------------------------------------------- */
int orc_i2_get(const uint8_t* row, int j) {
  const int k = j & 3;
  const int code = (row[j >> 2] >> (2 * k)) & 3;
  return code >= 2 ? code - 4 : code;
}

void orc_pack_i2_row(const int8_t* q, int cols, uint8_t* packed_row) {
  for (int i = 0; i < cols / 4; ++i) {
    int byte = 0;
    for (int k = 0; k < 4; ++k) byte |= (q[4 * i + k] & 3) << (2 * k);
    packed_row[i] = (uint8_t)byte;
  }
}

void orc_quantize_i2_rows(const float* w, int64_t rows, int cols, uint8_t* packed, float* scales) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const float* wr = w + r * cols;
    float amax = 0.0f;
    for (int j = 0; j < cols; ++j) {
      float a = fabsf(wr[j]);
      if (a > amax) amax = a;
    }
    const float s = amax / 1.0f;
    int8_t* q = (int8_t*)malloc((size_t)cols);
    for (int j = 0; j < cols; ++j) {
      int v = 0;
      if (s != 0.0f) {
        v = (int)roundf(wr[j] / s);
        if (v > 1) v = 1;
        if (v < -1) v = -1;
      }
      q[j] = (int8_t)v;
    }
    orc_pack_i2_row(q, cols, packed + r * (cols / 4));
    free(q);
    scales[r] = s;
  }
}

/* Integer dot of block b (32 elements) of an int2 row with int8 activation codes; exact in
 * int32: |sum| <= 32 * 2 * 127. */
int32_t orc_i2_block_dot(const uint8_t* wrow, const int8_t* qx, int b) {
  int32_t acc = 0;
  for (int j = b * QB; j < (b + 1) * QB; ++j) acc += orc_i2_get(wrow, j) * (int32_t)qx[j];
  return acc;
}

/* out[r] = s[r] * canon_blocksum(dx, A[r, :]) with A[r,b] = i2_block_dot(row r, b): the int2
 * counterpart of orc_i4_matvec; the rows stay packed (dequant-on-use). */
void orc_i2_matvec(const uint8_t* W, const float* s, int rows, int cols, const int8_t* qx,
                   const float* dx, float* out, int32_t* A) {
  const int nb = cols / QB;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    int32_t* Ar = (int32_t*)malloc(sizeof(int32_t) * (size_t)nb);
    const uint8_t* wrow = W + (int64_t)r * (cols / 4);
    for (int b = 0; b < nb; ++b) Ar[b] = orc_i2_block_dot(wrow, qx, b);
    out[r] = s[r] * orc_canon_blocksum(dx, Ar, nb);
    if (A) memcpy(A + (int64_t)r * nb, Ar, sizeof(int32_t) * (size_t)nb);
    free(Ar);
  }
}

/* ------------------------------------------------------------------------------------------
 * Router.  P1 §5 (moe step: sigmoid routing, pick the top-8 experts) and P3 (DeepSeek-V3-style
 * sigmoid router).  Readings: the optional per-expert bias changes only which experts are
 * selected (DeepSeek-V3 semantics); weights come from the unbiased scores, renormalised over
 * the selected experts by their sum taken in rank order; ties go to the lower expert index.
 * ---------------------------------------------------------------------------------------- */
void orc_topk(const float* sel, int E, int K, int32_t* ids) {
  char* taken = (char*)calloc((size_t)E, 1);
  for (int k = 0; k < K; ++k) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || sel[e] > sel[best])
        best = e; /* strict: the lower index keeps a tie */
    }
    taken[best] = 1;
    ids[k] = best;
  }
  free(taken);
}

void orc_route_token(const float* Wr, const float* bias, const float* x, int E, int d, int K,
                     float routed_scale, float* logits, float* scores, int32_t* ids, float* w) {
  float* sel = (float*)malloc(sizeof(float) * (size_t)E);
  for (int e = 0; e < E; ++e) {
    logits[e] = orc_canon_dot(Wr + (int64_t)e * d, x, d);
    scores[e] = orc_sigmoid(logits[e]);
    sel[e] = bias ? scores[e] + bias[e] : scores[e];
  }
  orc_topk(sel, E, K, ids);
  float S = scores[ids[0]];
  for (int k = 1; k < K; ++k) S = S + scores[ids[k]];
  for (int k = 0; k < K; ++k)
    w[k] = (scores[ids[k]] / S) * routed_scale;
  free(sel);
}

/* RMSNorm: x * (1 / sqrt(mean(x^2) + eps)) * gamma */
void orc_rmsnorm(const float* x, const float* gamma, int d, float eps, float* out) {
  float ms = orc_canon_dot(x, x, d) / (float)d;
  float r = 1.0f / sqrtf(ms + eps);
  for (int j = 0; j < d; ++j) out[j] = (x[j] * r) * gamma[j];
}

/* ------------------------------------------------------------------------------------------
 * Batch union (P2 "絕不為同一次硬碟讀取等待兩遍"): the T*K (token, expert) pairs are grouped
 * by expert so each distinct expert is visited once.  Stable counting sort by expert id, then token; union
 * slots in ascending expert id; the shared expert (id E) is appended as the last slot with
 * every token.  Returns the number of union slots.
 * ---------------------------------------------------------------------------------------- */
int orc_union_bucket(const int32_t* ids, int T, int K, int E, int n_shared, int32_t* union_ids,
                     int32_t* offsets, int32_t* pair_token, int32_t* pair_rank, int32_t* inv) {
  int32_t* count = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (int i = 0; i < T * K; ++i) count[ids[i]]++;
  int nu = 0, p = 0;
  for (int e = 0; e < E; ++e) {
    if (!count[e]) continue;
    union_ids[nu] = e;
    offsets[nu] = p;
    for (int t = 0; t < T; ++t)
      for (int k = 0; k < K; ++k)
        if (ids[t * K + k] == e) {
          pair_token[p] = t;
          pair_rank[p] = k;
          inv[t * K + k] = p;
          ++p;
        }
    ++nu;
  }
  if (n_shared) {
    union_ids[nu] = E;
    offsets[nu] = p;
    for (int t = 0; t < T; ++t) {
      pair_token[p] = t;
      pair_rank[p] = -1;
      ++p;
    }
    ++nu;
  }
  offsets[nu] = p;
  free(count);
  return nu;
}

/* ------------------------------------------------------------------------------------------
 * One expert on one token (P1 §5: gate/up/SiLU/down on the IDOT fast path).
 *   g = W_g x, u = W_u x (int4 x int8 with per-row and per-block scales), h = SiLU(g) * u,
 *   h re-quantised to int8 blocks of 32 (every IDOT activation is int8, P1 §3.1), e = W_d h.
 * ---------------------------------------------------------------------------------------- */
void orc_expert_ffn(const uint8_t* rec, const float* sc, int d, int f, const int8_t* qx,
                    const float* dx, int8_t* qh, float* dh, float* e, float* g_out,
                    float* u_out, float* h_out, int32_t* Ag, int32_t* Au, int32_t* Ad) {
  const uint8_t* Wg = rec;
  const uint8_t* Wu = rec + (int64_t)f * d / 2;
  const uint8_t* Wd = rec + (int64_t)f * d;
  const float* sg = sc;
  const float* su = sc + f;
  const float* sd = sc + 2 * f;
  float* g = (float*)malloc(sizeof(float) * (size_t)f);
  float* u = (float*)malloc(sizeof(float) * (size_t)f);
  float* h = (float*)malloc(sizeof(float) * (size_t)f);
  orc_i4_matvec(Wg, sg, f, d, qx, dx, g, Ag);
  orc_i4_matvec(Wu, su, f, d, qx, dx, u, Au);
  for (int r = 0; r < f; ++r) h[r] = orc_silu_mul(g[r], u[r]);
  orc_quantize_q8(h, f, qh, dh);
  orc_i4_matvec(Wd, sd, d, f, qh, dh, e, Ad);
  if (g_out) memcpy(g_out, g, sizeof(float) * (size_t)f);
  if (u_out) memcpy(u_out, u, sizeof(float) * (size_t)f);
  if (h_out) memcpy(h_out, h, sizeof(float) * (size_t)f);
  free(g);
  free(u);
  free(h);
}

/* ------------------------------------------------------------------------------------------
 * One expert whose rows are int8, int4 or int2 (P1 §3.1 "int8", "int4 packed", "int2 packed";
 * P1 §5 gate/up/SiLU/down).  Reading: the record keeps the int4 layout [gate f x d | up f x d |
 * down d x f] at bits/8 bytes per weight (int8: one code per byte; int2: four per byte), with
 * the same f32 row scales [s_g | s_u | s_d]; the steps are those of orc_expert_ffn, each
 * matvec taking the rows' own format.  bits = 4 gives orc_expert_ffn's result.
 * ---------------------------------------------------------------------------------------- */
static void matvec_bits(int bits, const uint8_t* W, const float* s, int rows, int cols,
                        const int8_t* q, const float* dq, float* out) {
  if (bits == 8) orc_i8_matvec((const int8_t*)W, s, rows, cols, q, dq, out, NULL);
  else if (bits == 2) orc_i2_matvec(W, s, rows, cols, q, dq, out, NULL);
  else orc_i4_matvec(W, s, rows, cols, q, dq, out, NULL);
}

int orc_expert_ffn_bits(int bits, const uint8_t* rec, const float* sc, int d, int f,
                        const int8_t* qx, const float* dx, int8_t* qh, float* dh, float* e,
                        float* g_out, float* u_out, float* h_out) {
  if (bits != 8 && bits != 4 && bits != 2) return -1;
  const int64_t mat = (int64_t)f * d * bits / 8;
  const uint8_t* Wg = rec;
  const uint8_t* Wu = rec + mat;
  const uint8_t* Wd = rec + 2 * mat;
  float* g = (float*)malloc(sizeof(float) * (size_t)f);
  float* u = (float*)malloc(sizeof(float) * (size_t)f);
  float* h = (float*)malloc(sizeof(float) * (size_t)f);
  matvec_bits(bits, Wg, sc, f, d, qx, dx, g);
  matvec_bits(bits, Wu, sc + f, f, d, qx, dx, u);
  for (int r = 0; r < f; ++r) h[r] = orc_silu_mul(g[r], u[r]);
  orc_quantize_q8(h, f, qh, dh);
  matvec_bits(bits, Wd, sc + 2 * f, d, f, qh, dh, e);
  if (g_out) memcpy(g_out, g, sizeof(float) * (size_t)f);
  if (u_out) memcpy(u_out, u, sizeof(float) * (size_t)f);
  if (h_out) memcpy(h_out, h, sizeof(float) * (size_t)f);
  free(g);
  free(u);
  free(h);
  return 0;
}

/* fp64 value of one output row of int8, int4 or int2 rows x int8 codes, from the same
 * integer codes */
static double matvec_row64(int bits, const uint8_t* W, const float* s, int r, int cols,
                           const int8_t* q, const float* dq) {
  const uint8_t* wrow = W + (int64_t)r * cols * bits / 8;
  double acc = 0.0;
  for (int b = 0; b < cols / QB; ++b) {
    const int32_t A = bits == 8   ? orc_i8_block_dot((const int8_t*)wrow, q, b)
                      : bits == 2 ? orc_i2_block_dot(wrow, q, b)
                                  : orc_block_dot(wrow, q, b);
    acc += (double)dq[b] * (double)A;
  }
  return (double)s[r] * acc;
}

/* ------------------------------------------------------------------------------------------
 * Full layer (P1 §5 moe step; P2 batch union; combine order fixed).
 *   x_n = RMSNorm(x) if has_norm else x; q8(x_n); route each token; union/bucket; each pair
 *   runs its expert; y_t = e(shared, t), then y_t = fma(w_{t,k}, e(t,k), y_t) for k = 0..K-1;
 *   with has_norm the residual is added last: y_t = x_t + y_t.
 * ---------------------------------------------------------------------------------------- */
int orc_moe_forward(const orc_cfg* c, const float* x, int T, const float* Wr, const float* bias,
                    const float* gamma, const uint8_t* const* rec, const float* const* sc, float* y,
                    double* y64, const orc_dump* dump) {
  const int d = c->d, f = c->f, E = c->n_experts, K = c->top_k, bits = c->wbits;
  if (T <= 0) return 0;
  if (d % 64 || f % 64 || K < 1 || K > E || c->qblock != QB) return -1;
  if (bits != 4 && bits != 8 && bits != 2) return -1;
  /* the down rows of a record */
  const int64_t down_at = 2 * ((int64_t)f * d * bits / 8);
  const int P = T * K + (c->n_shared ? T : 0);
  float* xn = (float*)malloc(sizeof(float) * (size_t)T * d);
  int8_t* qx = (int8_t*)malloc((size_t)T * d);
  float* dx = (float*)malloc(sizeof(float) * (size_t)T * (d / QB));
  float* logits = (float*)malloc(sizeof(float) * (size_t)T * E);
  float* scores = (float*)malloc(sizeof(float) * (size_t)T * E);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * K);
  float* w = (float*)malloc(sizeof(float) * (size_t)T * K);
  int32_t* union_ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
  int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 2));
  int32_t* pair_token = (int32_t*)malloc(sizeof(int32_t) * (size_t)P);
  int32_t* pair_rank = (int32_t*)malloc(sizeof(int32_t) * (size_t)P);
  int32_t* inv = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * K);
  int8_t* qh = (int8_t*)malloc((size_t)P * f);
  float* dh = (float*)malloc(sizeof(float) * (size_t)P * (f / QB));
  float* e = (float*)malloc(sizeof(float) * (size_t)P * d);
  int rc = 0;

  for (int t = 0; t < T; ++t) {
    if (c->has_norm)
      orc_rmsnorm(x + (int64_t)t * d, gamma, d, c->rms_eps, xn + (int64_t)t * d);
    else
      memcpy(xn + (int64_t)t * d, x + (int64_t)t * d, sizeof(float) * (size_t)d);
    orc_quantize_q8(xn + (int64_t)t * d, d, qx + (int64_t)t * d, dx + (int64_t)t * (d / QB));
    orc_route_token(Wr, bias, xn + (int64_t)t * d, E, d, K, c->routed_scale,
                    logits + (int64_t)t * E, scores + (int64_t)t * E, ids + t * K, w + t * K);
  }
  int nu = orc_union_bucket(ids, T, K, E, c->n_shared, union_ids, offsets, pair_token, pair_rank,
                            inv);
  for (int s = 0; s < nu; ++s) {
    int ex = union_ids[s];
    if (!rec[ex] || !sc[ex]) { rc = -1; goto done; }
    for (int p = offsets[s]; p < offsets[s + 1]; ++p) {
      int t = pair_token[p];
      if (bits != 4) { /* int8 / int2 experts (no per-block accumulator dump) */
        orc_expert_ffn_bits(bits, rec[ex], sc[ex], d, f, qx + (int64_t)t * d,
                            dx + (int64_t)t * (d / QB), qh + (int64_t)p * f,
                            dh + (int64_t)p * (f / QB), e + (int64_t)p * d,
                            dump && dump->g ? dump->g + (int64_t)p * f : NULL,
                            dump && dump->u ? dump->u + (int64_t)p * f : NULL,
                            dump && dump->h ? dump->h + (int64_t)p * f : NULL);
        continue;
      }
      orc_expert_ffn(rec[ex], sc[ex], d, f, qx + (int64_t)t * d, dx + (int64_t)t * (d / QB),
                     qh + (int64_t)p * f, dh + (int64_t)p * (f / QB), e + (int64_t)p * d,
                     dump && dump->g ? dump->g + (int64_t)p * f : NULL,
                     dump && dump->u ? dump->u + (int64_t)p * f : NULL,
                     dump && dump->h ? dump->h + (int64_t)p * f : NULL,
                     dump && dump->Ag ? dump->Ag + (int64_t)p * f * (d / QB) : NULL,
                     dump && dump->Au ? dump->Au + (int64_t)p * f * (d / QB) : NULL,
                     dump && dump->Ad ? dump->Ad + (int64_t)p * d * (f / QB) : NULL);
    }
  }
  for (int t = 0; t < T; ++t) {
    const int ps = c->n_shared ? T * K + t : -1;
    for (int r = 0; r < d; ++r) {
      float acc = ps >= 0 ? e[(int64_t)ps * d + r] : 0.0f;
      for (int k = 0; k < K; ++k) acc = fmaf(w[t * K + k], e[(int64_t)inv[t * K + k] * d + r], acc);
      if (c->has_norm) acc = x[(int64_t)t * d + r] + acc;
      y[(int64_t)t * d + r] = acc;
    }
    if (y64) {
      for (int r = 0; r < d; ++r) {
        double acc = 0.0;
        if (ps >= 0) {
          const uint8_t* Wd = rec[E] + down_at;
          acc = matvec_row64(bits, Wd, sc[E] + 2 * f, r, f, qh + (int64_t)ps * f,
                             dh + (int64_t)ps * (f / QB));
        }
        for (int k = 0; k < K; ++k) {
          int p = inv[t * K + k], ex = ids[t * K + k];
          const uint8_t* Wd = rec[ex] + down_at;
          acc += (double)w[t * K + k] * matvec_row64(bits, Wd, sc[ex] + 2 * f, r, f,
                                                     qh + (int64_t)p * f, dh + (int64_t)p * (f / QB));
        }
        if (c->has_norm) acc += (double)x[(int64_t)t * d + r];
        y64[(int64_t)t * d + r] = acc;
      }
    }
  }
  if (dump) {
    if (dump->xn) memcpy(dump->xn, xn, sizeof(float) * (size_t)T * d);
    if (dump->qx) memcpy(dump->qx, qx, (size_t)T * d);
    if (dump->dx) memcpy(dump->dx, dx, sizeof(float) * (size_t)T * (d / QB));
    if (dump->logits) memcpy(dump->logits, logits, sizeof(float) * (size_t)T * E);
    if (dump->scores) memcpy(dump->scores, scores, sizeof(float) * (size_t)T * E);
    if (dump->ids) memcpy(dump->ids, ids, sizeof(int32_t) * (size_t)T * K);
    if (dump->w) memcpy(dump->w, w, sizeof(float) * (size_t)T * K);
    if (dump->n_union) *dump->n_union = nu;
    if (dump->union_ids) memcpy(dump->union_ids, union_ids, sizeof(int32_t) * (size_t)nu);
    if (dump->offsets) memcpy(dump->offsets, offsets, sizeof(int32_t) * (size_t)(nu + 1));
    if (dump->pair_token) memcpy(dump->pair_token, pair_token, sizeof(int32_t) * (size_t)P);
    if (dump->pair_rank) memcpy(dump->pair_rank, pair_rank, sizeof(int32_t) * (size_t)P);
    if (dump->inv) memcpy(dump->inv, inv, sizeof(int32_t) * (size_t)T * K);
    if (dump->qh) memcpy(dump->qh, qh, (size_t)P * f);
    if (dump->dh) memcpy(dump->dh, dh, sizeof(float) * (size_t)P * (f / QB));
    if (dump->e) memcpy(dump->e, e, sizeof(float) * (size_t)P * d);
  }
done:
  free(xn); free(qx); free(dx); free(logits); free(scores); free(ids); free(w);
  free(union_ids); free(offsets); free(pair_token); free(pair_rank); free(inv);
  free(qh); free(dh); free(e);
  return rc;
}

/* fp64 dequant-on-use layer with fp64 activations: W = s*q (int4 codes), no activation or h
 * quantisation.  The comparator of the integer-dot path's accuracy (P1 §3.1, §6). */
int orc_moe_dequant64(const orc_cfg* c, const float* xn, int T, const int32_t* ids,
                      const float* w, const uint8_t* const* rec, const float* const* sc,
                      const float* x_resid, double* y) {
  const int d = c->d, f = c->f, E = c->n_experts, K = c->top_k;
  if (c->wbits != 4) return -1; /* the dequantised reference is written for int4 records */
  double* g = (double*)malloc(sizeof(double) * (size_t)f);
  double* u = (double*)malloc(sizeof(double) * (size_t)f);
  double* e = (double*)malloc(sizeof(double) * (size_t)d);
  for (int t = 0; t < T; ++t) {
    const float* xt = xn + (int64_t)t * d;
    double* yt = y + (int64_t)t * d;
    for (int r = 0; r < d; ++r) yt[r] = x_resid ? (double)x_resid[(int64_t)t * d + r] : 0.0;
    for (int k = -1; k < K; ++k) {
      int ex;
      double wk;
      if (k < 0) {
        if (!c->n_shared) continue;
        ex = E;
        wk = 1.0;
      } else {
        ex = ids[t * K + k];
        wk = (double)w[t * K + k];
      }
      if (!rec[ex] || !sc[ex]) { free(g); free(u); free(e); return -1; }
      const uint8_t* Wg = rec[ex];
      const uint8_t* Wu = rec[ex] + (int64_t)f * d / 2;
      const uint8_t* Wd = rec[ex] + (int64_t)f * d;
      const float* s = sc[ex];
#pragma omp parallel for schedule(static)
      for (int r = 0; r < f; ++r) {
        double ag = 0.0, au = 0.0;
        for (int j = 0; j < d; ++j) {
          ag += (double)orc_i4_get(Wg + (int64_t)r * (d / 2), j) * (double)xt[j];
          au += (double)orc_i4_get(Wu + (int64_t)r * (d / 2), j) * (double)xt[j];
        }
        g[r] = (double)s[r] * ag;
        u[r] = (double)s[f + r] * au;
      }
      for (int r = 0; r < f; ++r) g[r] = g[r] / (1.0 + exp(-g[r])) * u[r];
#pragma omp parallel for schedule(static)
      for (int r = 0; r < d; ++r) {
        double a = 0.0;
        for (int j = 0; j < f; ++j) a += (double)orc_i4_get(Wd + (int64_t)r * (f / 2), j) * g[j];
        e[r] = (double)s[2 * f + r] * a;
      }
      for (int r = 0; r < d; ++r) yt[r] += wk * e[r];
    }
  }
  free(g); free(u); free(e);
  return 0;
}
