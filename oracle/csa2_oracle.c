/*
 * CPU oracle for the CSA2 FP4 compressed global KV cache.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  It shares no code with
 * the CUDA library.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math (see oracle/build.py).
 * No fused multiply-add contraction, so every float32 operation written here is
 * one correctly rounded IEEE operation.
 */
#include "csa2_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static float u32_as_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static double bf16_value(uint16_t b) { return (double)u32_as_f32((uint32_t)b << 16); }

/* ---------------------------------------------------------------- E2M1 ---------
 * OCP E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit.  Exponent field 0 encodes
 * the subnormal 0.m * 2^0 = {0, 0.5}; fields 1..3 encode 1.m * 2^(e-1).  The
 * representable magnitudes are therefore 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7).
 *
 * Encoding reading (ezic blog gives the format, not the rounding): round to nearest,
 * ties to the even code (mantissa bit 0), saturate to 6, keep the sign bit even
 * when the magnitude rounds to zero.  Written as the decision table that this rule
 * produces between consecutive magnitudes:
 *   |y| <= 0.25 -> 0     (0.25 is halfway between 0 and 0.5: even code 0)
 *   |y| <  0.75 -> 0.5   (0.75 halfway between 0.5 and 1: even code 2 = 1.0)
 *   |y| <= 1.25 -> 1     (1.25 halfway between 1 and 1.5: even code 2)
 *   |y| <  1.75 -> 1.5
 *   |y| <= 2.5  -> 2
 *   |y| <  3.5  -> 3
 *   |y| <= 5    -> 4
 *   otherwise   -> 6
 */
uint8_t orc_e2m1_encode(float y) {
  uint8_t sign = signbit(y) ? 0x8 : 0x0;
  double a = fabs((double)y);
  uint8_t mag;
  if (a <= 0.25) mag = 0;
  else if (a < 0.75) mag = 1;
  else if (a <= 1.25) mag = 2;
  else if (a < 1.75) mag = 3;
  else if (a <= 2.5) mag = 4;
  else if (a < 3.5) mag = 5;
  else if (a <= 5.0) mag = 6;
  else mag = 7;
  return (uint8_t)(sign | mag);
}

double orc_e2m1_decode(uint8_t code) {
  int e = (code >> 1) & 3, m = code & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return (code & 8) ? -v : v;
}

/* ---------------------------------------------------------------- E4M3 ---------
 * OCP E4M3FN: 1 sign, 4 exponent (bias 7), 3 mantissa bits, no infinities, only
 * S.1111.111 is NaN.  Largest finite 448 = 1.75 * 2^8, smallest normal 2^-6,
 * smallest subnormal 2^-9.  Encoding: round to nearest, ties to even mantissa,
 * saturate finite values above 448 to 448 ("satfinite").
 */
static double round_half_even(double q) { /* q >= 0, exact input */
  double r = floor(q), f = q - r;
  if (f > 0.5 || (f == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  return r;
}

uint8_t orc_e4m3_encode(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: multiples of 2^-9; 8 * 2^-9 is the smallest normal (code 0x08) */
    double r = round_half_even(a * 512.0);
    return (uint8_t)(sign | (uint8_t)r);
  }
  int E;
  double f = frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) */
  int e = E - 1;           /* a = (2f) * 2^e, 2f in [1, 2) */
  double r = round_half_even((2.0 * f - 1.0) * 8.0);
  if (r == 8.0) { r = 0.0; e += 1; }
  int field = e + 7; /* 1..15; a < 448 keeps (field, r) below (15, 7) */
  return (uint8_t)(sign | (field << 3) | (int)r);
}

double orc_e4m3_decode(uint8_t b) {
  int e = (b >> 3) & 0xF, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return (b & 0x80) ? -v : v;
}

/* ---------------------------------------------------------------- blocks -------
 * Page 1 ("FP4主KVキャッシュ"): 4-bit E2M1 values with one E4M3 scale per 16
 * channels.  Reading of the open steps:
 *   amax = max |x_i| over the 16 channels (float32),
 *   s    = E4M3(fl32(amax / 6))  (6 = largest E2M1 magnitude; IEEE division),
 *   y_i  = fl32(x_i / decode(s)) (IEEE division by the decoded scale),
 *   code_i = E2M1(y_i); if decode(s) == 0 every code is 0.
 * No second-level (per-tensor) scale: the pages mention none.
 */
static void quantize_block16(const float* x, uint8_t* codes8, uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float t = amax / 6.0f;
  uint8_t sb = orc_e4m3_encode(t);
  float s = (float)orc_e4m3_decode(sb);
  *scale = sb;
  for (int j = 0; j < 8; ++j) {
    uint8_t lo = 0, hi = 0;
    if (s > 0.0f) {
      float y0 = x[2 * j] / s;
      float y1 = x[2 * j + 1] / s;
      lo = orc_e2m1_encode(y0);
      hi = orc_e2m1_encode(y1);
    }
    codes8[j] = (uint8_t)(lo | (hi << 4));
  }
}

void orc_quantize_rows(const float* x, int64_t T, int32_t D, uint8_t* codes, uint8_t* scales) {
  int32_t nb = D / 16;
  for (int64_t t = 0; t < T; ++t)
    for (int32_t b = 0; b < nb; ++b)
      quantize_block16(x + t * D + b * 16, codes + t * (D / 2) + b * 8, scales + t * nb + b);
}

void orc_dequantize_rows(const uint8_t* codes, const uint8_t* scales, int64_t T, int32_t D,
                         double* out) {
  int32_t nb = D / 16;
  for (int64_t t = 0; t < T; ++t)
    for (int32_t c = 0; c < D; ++c) {
      uint8_t byte = codes[t * (D / 2) + c / 2];
      uint8_t code = (c & 1) ? (byte >> 4) : (byte & 0xF);
      out[t * D + c] = orc_e2m1_decode(code) * orc_e4m3_decode(scales[t * nb + c / 16]);
    }
}

/* ---------------------------------------------------------------- MXFP4 --------
 * Tech-report digest, "FP4 メイン KV Cache と SWA Bounded Replay": the main KV cache is
 * quantised to FP4 in the OCP-standard MXFP4 format (E2M1 elements).  The pages give
 * nothing more; the format is read as the OCP Microscaling (MX) definition:
 *   blocks of 32 elements share one E8M0 scale X = 2^(floor(log2 amax) - 2), where 2 is
 *   the exponent of E2M1's largest power of two (4; the largest magnitude is 6 = 1.5 * 4),
 *   clamped to E8M0's finite range 2^-127 .. 2^127 (byte = exponent + 127, 255 = NaN is
 *   never produced);
 *   each element is E2M1(x_i / X): round to nearest, ties to the even code, saturating at
 *   6, sign kept;
 *   a block whose amax is 0 gets scale byte 0 and zero codes.
 * Values x_i / X lie in [0, 8), so the top E2M1 step [6, 8) saturates.  Footprint: 256 B
 * of codes + 16 B of scales per 512 channels (272 B, against 288 B for E4M3 / 16).
 */
uint8_t orc_e8m0_scale_for(float amax) {
  if (!(amax > 0.0f)) return 0;
  int e;
  (void)frexp((double)amax, &e); /* amax = f * 2^e, f in [0.5, 1): floor(log2 amax) = e - 1 */
  int se = (e - 1) - 2;
  if (se < -127) se = -127;
  if (se > 127) se = 127;
  return (uint8_t)(se + 127);
}

double orc_e8m0_decode(uint8_t b) { return ldexp(1.0, (int)b - 127); }

static void quantize_block32_mx(const float* x, uint8_t* codes16, uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  uint8_t sb = orc_e8m0_scale_for(amax);
  double X = orc_e8m0_decode(sb);
  *scale = sb;
  for (int j = 0; j < 16; ++j) {
    uint8_t lo = 0, hi = 0;
    if (amax > 0.0f) {
      lo = orc_e2m1_encode((float)((double)x[2 * j] / X));
      hi = orc_e2m1_encode((float)((double)x[2 * j + 1] / X));
    }
    codes16[j] = (uint8_t)(lo | (hi << 4));
  }
}

void orc_mx_quantize_rows(const float* x, int64_t T, int32_t D, uint8_t* codes, uint8_t* scales) {
  int32_t nb = D / 32;
  for (int64_t t = 0; t < T; ++t)
    for (int32_t b = 0; b < nb; ++b)
      quantize_block32_mx(x + t * D + b * 32, codes + t * (D / 2) + b * 16, scales + t * nb + b);
}

void orc_mx_dequantize_rows(const uint8_t* codes, const uint8_t* scales, int64_t T, int32_t D,
                            double* out) {
  int32_t nb = D / 32;
  for (int64_t t = 0; t < T; ++t)
    for (int32_t c = 0; c < D; ++c) {
      uint8_t byte = codes[t * (D / 2) + c / 2];
      uint8_t code = (c & 1) ? (byte >> 4) : (byte & 0xF);
      out[t * D + c] = orc_e2m1_decode(code) * orc_e8m0_decode(scales[t * nb + c / 32]);
    }
}

/* ---------------------------------------------------------------- projection ---*/
void orc_project_rows(const uint16_t* H, const uint16_t* Wt, int64_t nrows, int32_t d_model,
                      int32_t n_out, float* C) {
  for (int64_t r = 0; r < nrows; ++r)
    for (int32_t n = 0; n < n_out; ++n) {
      double acc = 0.0;
      for (int32_t k = 0; k < d_model; ++k)
        acc += bf16_value(H[r * d_model + k]) * bf16_value(Wt[(int64_t)n * d_model + k]);
      C[r * n_out + n] = (float)acc;
    }
}

/* ---------------------------------------------------------------- indexer ------*/
void orc_index_scores(const uint16_t* q, const uint16_t* keys, int64_t n, double* score) {
  for (int64_t s = 0; s < n; ++s) {
    double total = 0.0;
    for (int h = 0; h < 4; ++h) {
      double dot = 0.0;
      for (int d = 0; d < 128; ++d) dot += bf16_value(q[h * 128 + d]) * bf16_value(keys[s * 128 + d]);
      if (dot > 0.0) total += dot;
    }
    score[s] = total;
  }
}

typedef struct {
  double score;
  int32_t token;
} cand_t;

static int by_rank(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->token > y->token) - (x->token < y->token);
}

static int by_token(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

void orc_select_topk(const double* score, const int32_t* token, int64_t n, int32_t k,
                     int32_t* out) {
  cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)(n > 0 ? n : 1));
  for (int64_t i = 0; i < n; ++i) {
    c[i].score = score[i];
    c[i].token = token[i];
  }
  qsort(c, (size_t)n, sizeof(cand_t), by_rank);
  int64_t m = n < k ? n : k;
  for (int64_t i = 0; i < m; ++i) out[i] = c[i].token;
  qsort(out, (size_t)m, sizeof(int32_t), by_token);
  for (int64_t i = m; i < k; ++i) out[i] = -1;
  free(c);
}

/* ---------------------------------------------------------------- attention ----*/
void orc_sparse_attention(const uint16_t* q, const double* chat, int64_t n, float softmax_scale,
                          float* out, float* lse) {
  double* z = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int h = 0; h < 16; ++h) {
    if (n == 0) {
      for (int c = 0; c < 512; ++c) out[h * 512 + c] = 0.0f;
      lse[h] = -INFINITY;
      continue;
    }
    double m = -INFINITY;
    for (int64_t s = 0; s < n; ++s) {
      double dot = 0.0;
      for (int c = 0; c < 512; ++c) dot += bf16_value(q[h * 512 + c]) * chat[s * 512 + c];
      z[s] = dot * (double)softmax_scale;
      if (z[s] > m) m = z[s];
    }
    double l = 0.0;
    for (int64_t s = 0; s < n; ++s) {
      z[s] = exp(z[s] - m);
      l += z[s];
    }
    for (int c = 0; c < 512; ++c) {
      double acc = 0.0;
      for (int64_t s = 0; s < n; ++s) acc += z[s] * chat[s * 512 + c];
      out[h * 512 + c] = (float)(acc / l);
    }
    lse[h] = (float)(m + log(l));
  }
  free(z);
}

void orc_e2m1_encode_array(const float* y, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_encode(y[i]);
}

void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}
