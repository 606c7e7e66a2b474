/*
 * qwm_baselines.h -- comparison baselines of the ablation workload, in libqwm.so.
 *
 * These are not part of the QuantWM path; they let the ablation compare it with the two methods
 * the QuantWM pages measure against, on the same device and the same synthetic cache.
 *  - QVG (Quant VideoGen summary §2A k-means smoothing, §2B progressive residual quantisation):
 *    a chunk is quantised in stages; each stage takes the nearest centroid of the previous stage's
 *    residual (qwm_quantize_kv with a 1-candidate, rank-0 context and no weights is exactly
 *    that), qwm_prq_residual forms the next stage's input, and the last stage's residual is INT2.
 *    qwm_prq_dequantize is the fused decoder of a two-stage chunk (all centroids + the INT2 residual
 *    in one pass).
 *  - KIVI-style INT2 (named by the QuantWM summaries as the baseline with finer groups and a bf16
 *    recent window, Korean summary "전제와 한계"; the form used is the ablation workload's):
 *    Keys per channel over groups of 32 consecutive tokens, Values per token over groups of 32
 *    consecutive channels, the QuantWM INT2 encoder applied to the raw values.  The bf16 recent
 *    window is the caller's: it simply does not quantise the last tokens.
 * Conventions as in qwm.h: device pointers, caller-owned, 16-byte aligned; asynchronous on the
 * stream; a qwm_status return; H = config.heads, d = 128.
 */
#ifndef QWM_BASELINES_H_
#define QWM_BASELINES_H_

#include "qwm.h"

#ifdef __cplusplus
extern "C" {
#endif

#define QWM_KIVI_GROUP 32

typedef struct {
  int64_t n_tokens;  /* N >= 0 */
  uint8_t *k_codes;  /* [H][N][d/4], channel 4j+t -> bits 2t..2t+1 of byte j */
  uint8_t *v_codes;  /* [H][N][d/4] */
  uint16_t *k_scale; /* fp16 [H][ceil(N/32)][d]: per (token group, channel) step */
  uint16_t *k_min;   /* fp16 [H][ceil(N/32)][d]: offset */
  uint16_t *v_scale; /* fp16 [H][N][d/32]: per (token, channel group) step */
  uint16_t *v_min;   /* fp16 [H][N][d/32] */
} qwm_kivi_chunk;

/* KIVI-style INT2 of one chunk: k, v bf16 [H][n][d]; out->n_tokens must equal n.  Per group:
 * m = fp16 round-down of the minimum, s = fp16 round-up of (max - m)/3, q = clamp(rint((x-m)/s), 0, 3). */
QWM_API qwm_status qwm_kivi_quantize(qwm_ctx *ctx, const uint16_t *k, const uint16_t *v, int64_t n,
                                     qwm_kivi_chunk *out, qwm_stream stream);

/* bf16 [H][N][d] reconstruction m + s q (either output may be NULL). */
QWM_API qwm_status qwm_kivi_dequantize(qwm_ctx *ctx, const qwm_kivi_chunk *chunk, uint16_t *k_hat, uint16_t *v_hat,
                                       qwm_stream stream);

/* QVG stage residual: out = bf16(x - mu_idx) (fp32 difference, nearest-even), all heads.
 *   x bf16 [H][n][d]; cent bf16 [H][C][d]; idx [H][n] (uint8, or uint16 when C = 1024); out bf16 [H][n][d]. */
QWM_API qwm_status qwm_prq_residual(qwm_ctx *ctx, const uint16_t *x, int64_t n, const uint16_t *cent,
                                    const void *idx, uint16_t *out, qwm_stream stream);

/* Fused decoder of a two-stage QVG chunk: x_hat = bf16(mu1_idx1 + (mu2_idx2 + (m + s q))), where
 * `last` is the second stage's chunk (qwm_quantize_kv output; rank_eff must be 0) and cent1_* /
 * idx1_* the first stage's codebooks and indices (layouts as in qwm_chunk).  Either output may be NULL. */
QWM_API qwm_status qwm_prq_dequantize(qwm_ctx *ctx, const qwm_chunk *last, const uint16_t *cent1_k,
                                      const void *idx1_k, const uint16_t *cent1_v, const void *idx1_v,
                                      uint16_t *k_hat, uint16_t *v_hat, qwm_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* QWM_BASELINES_H_ */
