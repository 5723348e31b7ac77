/*
 * CPU oracle for the CSA2 FP4 compressed global KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load or call this code.  The product path (libcsa2) shares
 * no code, header, table or helper with it.
 *
 * Plain, slow, single-threaded C.  Floating-point sums are carried in double.
 * Each function cites the passage of the pages of the "DeepSeek-V4.1-Flash" web pages it
 * follows: the ai2.x.ezic.info blog ("ezic blog"), the zaikei.co.jp article ("zaikei
 * article") and the jiwasawa.github.io tech-report digest ("tech-report digest").
 */
#ifndef CSA2_ORACLE_H
#define CSA2_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* FP4 E2M1 element codec (ezic blog "KVを捨てる、共有する、作り直す": main KV held as
 * 4-bit E2M1 floats; tech-report digest "FP4 メイン KV Cache": OCP E2M1).  code = s<<3|e<<1|m. */
uint8_t orc_e2m1_encode(float y);
double orc_e2m1_decode(uint8_t code);

/* FP8 E4M3 (OCP E4M3FN) scale codec (ezic blog: one E4M3 scale per 16 channels). */
uint8_t orc_e4m3_encode(float v);
double orc_e4m3_decode(uint8_t b);

/* Block quantiser: rows of D fp32 values (D a multiple of 16) -> packed codes
 * [T][D/2] (element 2j in the low nibble of byte j) and scales [T][D/16]. */
void orc_quantize_rows(const float* x, int64_t T, int32_t D, uint8_t* codes, uint8_t* scales);
/* Dequantiser: c = e2m1(code) * e4m3(scale), exact, as double [T][D]. */
void orc_dequantize_rows(const uint8_t* codes, const uint8_t* scales, int64_t T, int32_t D,
                         double* out);

/* MXFP4 variant (tech-report digest "FP4 メイン KV Cache": OCP-standard MXFP4, E2M1),
 * read as OCP MX: one E8M0 scale per 32 channels, X = 2^(floor(log2 amax) - 2) clamped to
 * 2^-127..2^127; codes = E2M1_RNE_sat(x / X); zero block -> scale byte 0, zero codes.
 * Codes [T][D/2] as above, scales [T][D/32]; D a multiple of 32. */
uint8_t orc_e8m0_scale_for(float amax);
double orc_e8m0_decode(uint8_t b);
void orc_mx_quantize_rows(const float* x, int64_t T, int32_t D, uint8_t* codes, uint8_t* scales);
void orc_mx_dequantize_rows(const uint8_t* codes, const uint8_t* scales, int64_t T, int32_t D,
                            double* out);

/* CED projection (tech-report digest "Causal Encoder-Decoder (CED)" equation C_l = H_{L/2} W_l^KV):
 * C[r][n] = fl32(sum_k H[r][k] * Wt[n][k]) with the sum in double.  H is bf16
 * [nrows][d_model]; the projection is stored output-major, Wt[n][k] = W[k][n]. */
void orc_project_rows(const uint16_t* H, const uint16_t* Wt, int64_t nrows, int32_t d_model,
                      int32_t n_out, float* C);

/* Indexer score (tech-report digest "CSA2" Full/Reindex modes; scoring formula is a reading):
 * score[s] = sum_{h<4} max(0, sum_{d<128} q[h][d] * key[s][d]) in double. */
void orc_index_scores(const uint16_t* q, const uint16_t* keys, int64_t n, double* score);

/* Top-k selection: rank candidates by (score descending, token ascending), keep the
 * first min(k, n), emit their tokens in ascending order, pad with -1 up to k. */
void orc_select_topk(const double* score, const int32_t* token, int64_t n, int32_t k,
                     int32_t* out);

/* Sparse attention over selected latent rows (tech-report digest "Reuse Mode": sparse attention
 * over the top-K entries; zaikei article: the FP4 cache is dequantised before attention).
 * q bf16 [16][512]; chat double [n][512] (dequantised rows); K = V = latent.
 * out[h] = softmax_s(scale * q_h.chat_s) . chat, lse[h] = natural-log sum-exp.
 * n == 0 gives out = 0 and lse = -inf. */
void orc_sparse_attention(const uint16_t* q, const double* chat, int64_t n, float softmax_scale,
                          float* out, float* lse);

/* Array helpers used by exhaustive checks. */
void orc_e2m1_encode_array(const float* y, int64_t n, uint8_t* out);
void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out);

#ifdef __cplusplus
}
#endif
#endif
