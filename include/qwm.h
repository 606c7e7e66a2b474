/*
 * qwm.h -- C ABI of libqwm.so, the GB300 (sm_103a) QuantWM quantise-and-attend path.
 *
 * QuantWM ("QuantWM: Temporally Consistent 2-Bit KV Cache Quantization for
 * Video World Models"; summaries in Chinese, Korean and English) compresses
 * each completed chunk of a video model's KV cache to 2 bits:
 *   1. per-head Query second moment M_h = (1/N) sum q q^T, its diagonal
 *      channel weights w_{h,c} and its top-r eigenvectors U_r;
 *   2. QSAC: the top-M centroids by the weighted distance
 *      d_Q = sum_c w_c (k_c - mu_c)^2, then the one minimising
 *      S = sum_g (sum_{c in G_g} w_c) R_g(k - mu)^2 (R_g = range of the residual
 *      over a group of 64 channels); Values take their nearest centroid (QVG);
 *   3. INT2 affine codes of the residual per group of 64, four codes per byte;
 *   4. PSAC: E = K - K_hat_0, C = E U_r stored as INT8, U_r as BF16;
 *   5. attention with logits Q K_hat_0^T + (Q U_r) C^T over the packed cache.
 * Cited passages: Chinese summary, "前置知识" (affine quantiser, centroid-residual
 * form, logits, Query second moment), "核心方法" (QSAC, PSAC), "方法步骤详情"
 * steps (1)-(5); English v2 summary §4.1, §4.2, §5.1, §C.3, §D.1; QVG summary
 * §2A (k-means along the sequence axis) and §2C (warm-started centroids).
 *
 * Conventions (every entry point):
 *  - Returns a qwm_status; no exception or abort crosses the ABI.
 *  - Asynchronous on the caller's stream.  Errors that only the device can see
 *    (an eigenvector that inverse iteration could not form, a residual out of fp16 range) are
 *    recorded in a status word inside the context; qwm_sync_status() waits on
 *    the stream, returns the first recorded error and clears it.
 *  - Every device buffer is owned by the caller.  The library allocates device
 *    memory only in qwm_create (its workspace, qwm_workspace_bytes() bytes)
 *    and frees it in qwm_destroy.
 *  - Every pointer must be 16-byte aligned and the tensor dense, in the layout
 *    given; bf16 and fp16 values travel as uint16_t bit patterns.  Pointers to empty arrays
 *    (a chunk with n_tokens == 0, Keys of a 0-token call, q and out of a 0-Query attention) may
 *    be NULL: such calls and chunks do nothing.
 *  - Head-major layouts: [H][tokens][channels] with H = config.heads.
 *  - A context is not thread-safe: its calls are made from one host thread at a time.  Calls that
 *    share part of its workspace must be ordered on one stream (the workspace is reused between
 *    calls): qwm_fit_centroids, qwm_fit_centroids_kv and qwm_quantize_kv (the k-means and packing
 *    workspaces, the context's second stream and its events) with one another, and
 *    qwm_update_query_stats with itself (its partial sums).  Those two groups use disjoint
 *    workspace, and qwm_attend, qwm_attend_merge, qwm_dequantize, qwm_dequantize_chunks,
 *    qwm_select_rank and the coefficient-layout calls use none (only the status word, which any
 *    number of kernels may write), so these may run on other streams beside the rest, ordered
 *    only by their own data.
 */
#ifndef QWM_H_
#define QWM_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QWM_API __attribute__((visibility("default")))
#else
#define QWM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qwm_stream; /* a cudaStream_t; NULL = the legacy default stream */

typedef enum {
  QWM_OK = 0,
  QWM_ERR_ARG = 1,           /* NULL pointer, negative size, bad enum value */
  QWM_ERR_SHAPE = 2,         /* a size the kernels do not support (see qwm_config) */
  QWM_ERR_ALIGN = 3,         /* a pointer that is not 16-byte aligned */
  QWM_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
  QWM_ERR_NOT_CONVERGED = 5, /* the eigensolver could not form an eigenvector (results still written) */
  QWM_ERR_UNSUPPORTED = 6,   /* a configuration the library does not implement */
  QWM_ERR_RANGE = 7,         /* a residual, scale or coefficient outside the fp16 range */
  QWM_ERR_DEVICE_TIMEOUT = 8 /* a kernel's internal wait ran past its time limit and the kernel gave up */
} qwm_status;

/* Hyper-parameters (Chinese summary "复现评估": 256 centroids, group size 64, BF16
 * centroids + INT2 residuals, r = 8, INT8 C, BF16 U_r, M = 4). */
typedef struct {
  int32_t heads;        /* H >= 1 */
  int32_t head_dim;     /* d; must be 128 */
  int32_t n_centroids;  /* C in {64, 128, 256} (uint8 indices) or 1024 (uint16 indices) */
  int32_t group;        /* channels per INT2 group; must be 64 */
  int32_t top_m;        /* QSAC candidates M, 1..16 and <= n_centroids */
  int32_t rank;         /* PSAC rank r, 0..16 */
  int32_t bits;         /* residual bits; must be 2 */
  int32_t kmeans_iters; /* Lloyd iterations per qwm_fit_centroids call, 1..100 */
  uint64_t seed;        /* reserved (no randomness on the path); pass 0 */
  int32_t storage;      /* qwm_storage: how a chunk's INT2 metadata is stored */
  int32_t psac_gate;    /* 1: keep a token's C only where it lowers sum_c w_c e_c^2 (Chinese summary
                           step (4): "仅当降低Query加权误差时保留"); 0: always keep */
  int32_t test_flags;   /* 0 in production; QWM_TEST_EXPIRE_WAIT for tests of the error path */
} qwm_config;

/* Test hooks (qwm_config.test_flags).
 *  QWM_TEST_EXPIRE_WAIT: in qwm_attend, the thread that issues the tensor-core work waits, before
 *    its first key tile, on a barrier that nothing completes, with a 1 ms limit.  The wait runs
 *    out, the kernel takes the path every expired wait takes (it records QWM_ERR_DEVICE_TIMEOUT,
 *    every role stops within its own bounded waits, issued tensor-core work is drained and tensor
 *    memory freed) and the call's output is undefined; the context stays usable.  This exercises
 *    the recovery path without a GPU fault. */
enum { QWM_TEST_EXPIRE_WAIT = 1 };

/* INT2 metadata layouts.
 *  QWM_STORAGE_FP16: per (token, group of 64) an fp16 offset m (round-down of the minimum) and an
 *    fp16 step s (round-up of the range / 3): r_hat = m + s q.
 *  QWM_STORAGE_COMPACT: the paper's packed form (Chinese summary step (3) "组缩放INT8+FP16二级缩放";
 *    English v2 §D.1 "bit-packed INT2 zero-points"): per (token, group) an 8-bit step s8 and a 2-bit
 *    zero-point z, per (128-token tile, group) an fp16 second-level scale sigma, a power of two:
 *    s = sigma s8, r_hat = s (q - z) (exact in fp16).  Each (token, group) takes the zero-point whose
 *    grid [-z s, (3 - z) s] covers its residual range with the smallest step (lower z on ties); sigma
 *    is the smallest power of two with 255 sigma >= the tile's largest such step; s8 = ceil(step /
 *    sigma); q = clamp(rint(r (1/s) + z), 0, 3).  |r - r_hat| <= s/2. */
typedef enum { QWM_STORAGE_FP16 = 0, QWM_STORAGE_COMPACT = 1 } qwm_storage;

typedef struct qwm_ctx qwm_ctx;

/* Kind of a chunk descriptor.  A chunk is quantised once it is complete; the chunk still being
 * generated stays in bf16 and attends beside the packed history (English v2 summary §5.1, §D.1). */
typedef enum {
  QWM_CHUNK_PACKED = 0, /* written by qwm_quantize_kv */
  QWM_CHUNK_BF16 = 1    /* k_raw / v_raw only (qwm_attend) */
} qwm_chunk_kind;

/* Layout of a packed chunk's PSAC coefficients (c and c_scale).
 *  QWM_C_DENSE: c int8 [H][N][r] and c_scale fp16 [H][N], r = rank_eff, as qwm_quantize_kv writes them.
 *  QWM_C_PER_HEAD: what qwm_psac_pack writes: each head h has its own rank r_h <= rank_eff (columns
 *    past r_h of its basis are zero, so its coefficients there are zero and not stored) and its own
 *    layout, dense (a row of r_h bytes and a scale per token) or sparse (rows only for the tokens
 *    whose scale is not zero, found through a 128-token-tile bitmap and per-tile counts), the smaller
 *    of the two (English v2 summary §D.1: the smaller dense or sparse coefficient layout, with
 *    sparse-index storage; Chinese summary step (4): C kept only where it lowers the Query-weighted
 *    error).  c_heads[h] locates head h's rows in c and scales in c_scale. */
typedef enum { QWM_C_DENSE = 0, QWM_C_PER_HEAD = 1 } qwm_c_layout;

typedef struct {
  int64_t c_off;   /* byte offset of the head's first row in chunk.c */
  int64_t s_off;   /* element offset of the head's first scale in chunk.c_scale */
  int32_t rank;    /* r_h: bytes per row (0: the head stores nothing and has no PSAC term) */
  int32_t sparse;  /* 0: a row per token; 1: rows of the kept tokens only (c_mask, c_tile_rank) */
} qwm_psac_head;

/* One compressed chunk of the cache, all heads.  Every pointer is caller-owned
 * device memory; N = n_tokens, H = heads, d = head_dim, G = d / group, r = rank. */
typedef struct {
  int64_t n_tokens;      /* N >= 0 */
  int32_t rank_eff;      /* r used for this chunk: 0 (cold start, PSAC off) or config.rank; 0 for bf16 */
  int32_t kind;          /* qwm_chunk_kind */
  uint8_t *k_codes;      /* [H][N][d/4]: channel 4j+t -> bits 2t..2t+1 of byte j */
  uint8_t *v_codes;      /* [H][N][d/4] */
  void *k_idx;           /* [H][N] Key centroid index: uint8 when C <= 256, uint16 when C = 1024 */
  void *v_idx;           /* [H][N] Value centroid index, likewise */
  uint16_t *k_scale;     /* fp16 [H][N][G]: INT2 step s */
  uint16_t *k_min;       /* fp16 [H][N][G]: INT2 offset m (r_hat = m + s q) */
  uint16_t *v_scale;     /* fp16 [H][N][G] */
  uint16_t *v_min;       /* fp16 [H][N][G] */
  uint16_t *cent_k;      /* bf16 [H][C][d] Key codebook the chunk is packed with (qwm_fit_centroids'
                            output); read by qwm_quantize_kv only: the caller may release it after */
  uint16_t *cent_v;      /* bf16 [H][C][d] Value codebook, likewise */
  int8_t *c;             /* [H][N][r] PSAC coefficients (unused when rank_eff == 0) */
  uint16_t *c_scale;     /* fp16 [H][N]: C_hat = c_scale * c */
  uint16_t *u_r;         /* bf16 [H][d][r]: the basis C was built with (snapshot per chunk) */
  uint16_t *cent_k16;    /* fp16 [H][C][d]: the chunk's stored Key codebook, written by qwm_quantize_kv
                            as the fp16 value of every bf16 centroid element (the same value for
                            magnitudes in [2^-17, 65504] and for 0; an element beyond 65504 records
                            QWM_ERR_RANGE); qwm_attend (as tensor-core operands) and qwm_dequantize
                            read it */
  uint16_t *cent_v16;    /* fp16 [H][C][d]: the stored Value codebook, likewise */
  /* QWM_CHUNK_BF16 only (every packed field above is then unused): */
  const uint16_t *k_raw; /* bf16 [H][N][d] Keys of the chunk being generated */
  const uint16_t *v_raw; /* bf16 [H][N][d] */
  int64_t causal_tpf;    /* > 0: block-causal mask over frames of causal_tpf tokens: Query row i (the
                            i-th row of qwm_attend's q, taken as token i of this chunk) sees key j of
                            this chunk only when j / causal_tpf <= i / causal_tpf; 0: no mask */
  /* QWM_STORAGE_COMPACT contexts only (k_scale, k_min, v_scale, v_min are then unused): */
  uint8_t *k_s8;         /* [H][N][G] 8-bit steps */
  uint8_t *v_s8;         /* [H][N][G] */
  uint8_t *k_zp;         /* [H][N] zero-points: group g in bits 2g..2g+1 */
  uint8_t *v_zp;         /* [H][N] */
  uint16_t *k_sigma;     /* fp16 [H][ceil(N/128)][G] second-level scales */
  uint16_t *v_sigma;     /* fp16 [H][ceil(N/128)][G] */
  /* PSAC coefficient layout (packed chunks with rank_eff > 0): */
  int32_t c_layout;      /* qwm_c_layout */
  const qwm_psac_head *c_heads; /* QWM_C_PER_HEAD: device [H] */
  const uint32_t *c_mask;       /* QWM_C_PER_HEAD: device [H][ceil(N/128)][4]: bit b of word w of tile t
                                   set when token 128 t + 32 w + b has a row (sparse heads) */
  const int32_t *c_tile_rank;   /* QWM_C_PER_HEAD: device [H][ceil(N/128)]: rows of the head stored
                                   for the tokens before tile t (sparse heads) */
} qwm_chunk;

/* Optional stage outputs of qwm_quantize_kv for parity checks (NULL members are skipped). */
typedef struct {
  float *c_f32;          /* [H][N][r] PSAC coefficients before INT8 */
  int32_t *cand;         /* [H][N][M] QSAC candidates (any order) */
  float *score;          /* [H][N] QSAC score S of the chosen Key centroid */
  float *gate_err;       /* [H][N][2] sum_c w_c e_c^2 without and with the decoded PSAC correction */
} qwm_debug;

QWM_API const char *qwm_status_string(qwm_status s);

/* Bytes of device workspace qwm_create allocates for this configuration. */
QWM_API size_t qwm_workspace_bytes(const qwm_config *cfg);

/* Validate cfg and allocate a context (host struct + device workspace) on the
 * current device.  *out is NULL on failure. */
QWM_API qwm_status qwm_create(const qwm_config *cfg, qwm_ctx **out);
QWM_API qwm_status qwm_destroy(qwm_ctx *ctx);

/* Step 1 -- Query statistics (Chinese summary "二阶Query统计与低秩分解" and step (1);
 * English v2 summary §D.1: statistics kept incrementally, no Query tensor kept;
 * principal basis recomputed at each chunk boundary).
 *   q        bf16 [H][nq][d]      Queries to fold in (nq >= 0; nq == 0 only recomputes)
 *   S        fp32 [H][d][d] inout running sum of q q^T
 *   n        int64 [H]     inout  running Query count
 *   w        fp32 [H][d]   out    w_c = S_cc / n, or 1 when n == 0 (cold start, §C.3)
 *   eigvals  fp32 [H][d]   out    eigenvalues of M = S / n, descending (0 when n == 0)
 *   u_r      bf16 [H][d][r] out   top-r eigenvectors of M (column k = k-th), rounded to
 *                                 nearest-even; each column's largest-magnitude component
 *                                 is positive.  May be NULL when config.rank == 0.
 * The eigensolver (fp32, one thread block per head) reduces M to tridiagonal form by Householder
 * reflections, finds every eigenvalue by bisection on Sturm counts and the top-r eigenvectors by
 * inverse iteration; an eigenvector whose solve overflowed or vanished records
 * QWM_ERR_NOT_CONVERGED in the status word. */
QWM_API qwm_status qwm_update_query_stats(qwm_ctx *ctx, const uint16_t *q, int64_t nq, float *S, int64_t *n,
                                  float *w, float *eigvals, uint16_t *u_r, qwm_stream stream);

/* Step 2a -- codebook (QVG summary §2A: k-means of the tokens along the sequence
 * axis; §2C: each chunk's k-means starts from the previous chunk's centroids).
 *   x     bf16 [H][n][d]  tokens of one chunk (n >= config.n_centroids)
 *   init  bf16 [H][C][d]  starting centroids, or NULL: centroid j starts at token floor(j n / C)
 *   cent  bf16 [H][C][d]  out: centroids after config.kmeans_iters Lloyd iterations
 *                          (Euclidean assignment, lower index on ties; a cluster left
 *                          empty keeps its centroid), rounded to nearest-even. */
QWM_API qwm_status qwm_fit_centroids(qwm_ctx *ctx, const uint16_t *x, int64_t n, const uint16_t *init, uint16_t *cent,
                             qwm_stream stream);

/* Step 2a for the Keys and the Values of one chunk in one call: the same two fits as
 * qwm_fit_centroids(ctx, k, n, init_k, cent_k) and qwm_fit_centroids(ctx, v, n, init_v, cent_v),
 * with bit-identical results, run side by side.  The Key fit runs on `stream`, the Value fit on
 * the context's second stream with a k-means workspace of its own (the two fits read and write
 * disjoint data); the second stream starts after the work `stream` already holds and `stream`
 * waits for it at the end, so the call is ordered on `stream` like any other.  Each fit uses
 * about 120 of the GPU's SMs at 40 heads, so side by side they fill the SMs one fit leaves idle.
 *   k, v           bf16 [H][n][d]  the chunk's Keys and Values (n >= config.n_centroids)
 *   init_k, init_v bf16 [H][C][d]  starting centroids of each, or NULL (as qwm_fit_centroids)
 *   cent_k, cent_v bf16 [H][C][d]  out: the two codebooks (distinct buffers: the two fits write them
 *                                  at the same time)
 * Errors as qwm_fit_centroids; on an error nothing is launched. */
QWM_API qwm_status qwm_fit_centroids_kv(qwm_ctx *ctx, const uint16_t *k, const uint16_t *v, int64_t n,
                                const uint16_t *init_k, const uint16_t *init_v, uint16_t *cent_k,
                                uint16_t *cent_v, qwm_stream stream);

/* Steps 2-4 -- QSAC assignment, INT2 residual codes and PSAC coefficients for one chunk
 * (Chinese summary "核心方法" and steps (2)-(4); Korean summary "무엇과 다른가", "어떻게 쓰나").
 *   k, v  bf16 [H][n][d]   the chunk's Keys and Values
 *   w     fp32 [H][d]      channel weights, or NULL for uniform weights (cold start)
 *   u_r   bf16 [H][d][r]   PSAC basis, or NULL to switch PSAC off (cold start)
 *   out   chunk to fill: out->n_tokens must equal n, out->cent_k / out->cent_v must hold the
 *         chunk's codebooks; the codes, indices, scales, the stored fp16 codebooks
 *         out->cent_k16 / out->cent_v16 and (when u_r) c, c_scale (QWM_C_DENSE) are written,
 *         out->rank_eff is set on the host (r or 0) and, when u_r is given, out->u_r must
 *         point at a caller-owned copy of the basis (the library does not copy it).
 *   dbg   optional stage outputs, or NULL.
 * INT2 per (token, group): m = fp16 round-down of min r, s = fp16 round-up of
 * (max r - m)/3 (s = 0 when max r == m), q = clamp(rint((r - m)/s), 0, 3); so |r - r_hat| <= s/2.
 * INT8 per token: sC = fp16 round-up of max|C|/127, c = clamp(rint(C/sC), -127, 127).
 * The Value pass runs on a second stream of the context beside the Key pass (forked from and joined
 * back into `stream` with events), so work issued on `stream` afterwards sees both. */
QWM_API qwm_status qwm_quantize_kv(qwm_ctx *ctx, const uint16_t *k, const uint16_t *v, int64_t n, const float *w,
                           const uint16_t *u_r, qwm_chunk *out, const qwm_debug *dbg, qwm_stream stream);

/* qwm_quantize_kv with the QSAC candidates ranked by the full quadratic form (k - mu)^T M (k - mu)
 * instead of its diagonal (English v2 summary §C.4: the ablation of QSAC's diagonal approximation;
 * the pages report no consistent gain).  The rest is unchanged, with w = diag(M) for the range score.
 *   S       fp32 [H][d][d] running sum of q q^T and
 *   n_seen  int64 [H]      running Query count, both as qwm_update_query_stats leaves them: the
 *                          library forms M = S / n (fp32, IEEE division) in its workspace, or the
 *                          identity for a head with n == 0 (uniform weights, as at a cold start). */
QWM_API qwm_status qwm_quantize_kv_full(qwm_ctx *ctx, const uint16_t *k, const uint16_t *v, int64_t n,
                                        const float *S, const int64_t *n_seen, const uint16_t *u_r, qwm_chunk *out,
                                        const qwm_debug *dbg, qwm_stream stream);

/* PSAC rank per (chunk, head) (Chinese summary "独立分析的弱点", weakness three: the Query energy's
 * concentration differs by model and layer, so one global r is a compromise; English v2 summary §C.2:
 * a larger r still helps).  For each head, the smallest r_h in 0..config.rank whose r_h largest
 * eigenvalues hold at least `energy` of their sum (tr M; the sum taken in descending order in double
 * precision; r_h = config.rank when no smaller one does, 0 when the sum is not positive), then
 * columns r_h.. of that head's basis set to zero, so that qwm_quantize_kv with this basis writes zero
 * coefficients past r_h (and its INT8 scale and gate see only the first r_h).
 *   eigvals    fp32 [H][d] descending (qwm_update_query_stats' output)
 *   energy     share of tr M to reach, in [0, 1]
 *   u_r        bf16 [H][d][config.rank] inout: the chunk's basis snapshot
 *   head_rank  int32 [H] out: r_h */
QWM_API qwm_status qwm_select_rank(qwm_ctx *ctx, const float *eigvals, float energy, uint16_t *u_r,
                                   int32_t *head_rank, qwm_stream stream);

/* Tokens per head whose PSAC scale is not zero (the tokens that keep a coefficient row in the sparse
 * layout) of a QWM_C_DENSE packed chunk.  kept: device int32 [H] out. */
QWM_API qwm_status qwm_psac_kept(qwm_ctx *ctx, const qwm_chunk *chunk, int32_t *kept, qwm_stream stream);

/* Host-only: the per-head layout of a QWM_C_PER_HEAD chunk of n tokens from each head's rank and kept
 * count: the dense layout takes n (r_h + 2) bytes, the sparse one kept (r_h + 2) + 20 ceil(n/128) bytes
 * (16-byte bitmap and 4-byte count per tile); each head takes the smaller (dense on a tie; a head with
 * r_h = 0 stores nothing).  Heads are laid out one after the other in c and c_scale.
 *   head_rank, kept  HOST int32 [H]
 *   plan             HOST [H] out (copy it to device memory for qwm_psac_pack and the chunk)
 *   c_bytes          out: bytes of c; n_scales: out: fp16 elements of c_scale (either may be NULL) */
QWM_API qwm_status qwm_psac_plan(const qwm_config *cfg, int64_t n, const int32_t *head_rank, const int32_t *kept,
                                 qwm_psac_head *plan, int64_t *c_bytes, int64_t *n_scales);

/* Repack a QWM_C_DENSE chunk's coefficients into the QWM_C_PER_HEAD layout of `plan`.
 *   dense        the packed chunk (c_layout QWM_C_DENSE, rank_eff > 0)
 *   plan         device [H], as qwm_psac_plan computed it for this chunk
 *   c            int8 [c_bytes] out; c_scale fp16 [n_scales] out
 *   c_mask       uint32 [H][ceil(N/128)][4] out; c_tile_rank int32 [H][ceil(N/128)] out
 * The caller then describes the chunk with c_layout = QWM_C_PER_HEAD and these buffers (the dense
 * c and c_scale may be released). */
QWM_API qwm_status qwm_psac_pack(qwm_ctx *ctx, const qwm_chunk *dense, const qwm_psac_head *plan, int8_t *c,
                                 uint16_t *c_scale, uint32_t *c_mask, int32_t *c_tile_rank, qwm_stream stream);

/* Step 5 -- attention over the compressed cache (Chinese summary "注意力logits与时空token
 * 选择": L = Q K^T / sqrt(d); "核心方法": PSAC logits Q K_hat_0^T + Q U_r C^T).
 *   q        bf16 [H][nq][d]
 *   chunks   HOST array of 1 <= n_chunks <= 128 chunk descriptors (device pointers inside);
 *            chunks with n_tokens == 0 are skipped.  QWM_CHUNK_BF16 chunks (the chunk still being
 *            generated) attend with their bf16 Keys and Values (converted to the kernel's fp16
 *            operands: exact for magnitudes in [2^-14, 65504]) in the same softmax, optionally
 *            under their block-causal mask; a Query row must see at least one key
 *   softmax_scale  multiplies both logit terms (usually 1/sqrt(d))
 *   out      fp32 [H][nq][d] = softmax(l) V_hat over every token of every chunk (no mask); fp32
 *            because the output averages thousands of values and its largest entries are many
 *            times its RMS, so a bf16 result would carry a rounding error larger than the
 *            computation's
 * The INT2/centroid/PSAC decode happens inside the kernel's tile loads; no decoded
 * K or V is written to memory. */
QWM_API qwm_status qwm_attend(qwm_ctx *ctx, const uint16_t *q, int64_t nq, const qwm_chunk *chunks, int32_t n_chunks,
                      float softmax_scale, float *out, qwm_stream stream);

/* qwm_attend over a subset of a cache's chunks, in two parts that merge: the softmax over a union of
 * chunk sets is the weighted mean of the softmaxes over its parts, each weighted by its share of the
 * exponential sum.  So the attention over the chunks already packed can run while the newest chunk is
 * still being fitted and packed, and the newest chunk's attention then merges into it.
 *   q, nq, chunks, n_chunks, softmax_scale  as qwm_attend
 *   out      fp32 [H][nq][d]   merge == 0: out; merge == 1: inout
 *   lse      fp32 [H][nq]      merge == 0: out; merge == 1: inout: log2 of the sum over the call's keys
 *                              of 2^(softmax_scale * log2(e) * l_ij), l_ij the logit as in qwm_attend
 *   merge    0: out and lse are this call's softmax output and log-sum-exp;
 *            1: out and lse hold a result over other keys of the same Queries (a merge == 0 call, or
 *               earlier merges) and become the result over those keys and this call's together
 * The merged output equals one qwm_attend over the union of the chunks up to rounding (the parts'
 * weights 2^(lse_part - lse_union) are computed in fp32 with CUDA's exp2f and log2f).  A Query row must
 * see at least one key in a merge == 0 call. */
QWM_API qwm_status qwm_attend_merge(qwm_ctx *ctx, const uint16_t *q, int64_t nq, const qwm_chunk *chunks,
                            int32_t n_chunks, float softmax_scale, float *out, float *lse, int32_t merge,
                            qwm_stream stream);

/* Step 5' -- BF16 reconstruction of one packed chunk (the pages' fused decoder, English v2 §D.1;
 * QWM_ERR_UNSUPPORTED for a QWM_CHUNK_BF16 descriptor):
 * K_hat = mu^K_idx + r_hat + C_hat U_r^T and V_hat = mu^V_idx + r_hat, rounded to nearest-even.
 *   k_hat, v_hat  bf16 [H][N][d] out (either may be NULL). */
QWM_API qwm_status qwm_dequantize(qwm_ctx *ctx, const qwm_chunk *chunk, uint16_t *k_hat, uint16_t *v_hat,
                          qwm_stream stream);

/* qwm_dequantize of several packed chunks in one launch, written one after the other along the
 * token axis: the decoded cache [H][sum N][d] in the order of `chunks` (the layout a bf16 attention
 * over the whole cache takes).  chunks: HOST array of 1 <= n_chunks <= 128 packed descriptors
 * (n_tokens == 0 ones skipped); k_hat, v_hat bf16 [H][sum of n_tokens][d] out (either may be NULL). */
QWM_API qwm_status qwm_dequantize_chunks(qwm_ctx *ctx, const qwm_chunk *chunks, int32_t n_chunks, uint16_t *k_hat,
                                         uint16_t *v_hat, qwm_stream stream);

/* Wait for `stream`, return (and clear) the first error recorded on the device since
 * the last call, else QWM_OK. */
QWM_API qwm_status qwm_sync_status(qwm_ctx *ctx, qwm_stream stream);

/* qwm_update_query_stats for callers that cannot allocate device memory.
 * (This entry point has no counterpart in the paper; it is a deployment convenience.)
 * Some callers cannot call cudaMalloc: an application whose device memory is handed out by its
 * own pool or by a host framework that owns every allocation, or a service whose memory budget is
 * fixed at start-up and must not grow.  Such callers cannot create a qwm_ctx, because
 * qwm_create allocates the context's workspace.  This call needs no context: it computes
 * exactly what qwm_update_query_stats computes (same arguments, layouts and meaning, with the
 * configuration passed directly) and allocates nothing -- no cudaMalloc, no cudaFree, no
 * allocating library routine.  Its scratch memory (the partial sums of q q^T) is
 * one fixed array inside the library, 8 MiB, that every GPU which loads the library
 * keeps until the process exits.
 *   cfg          only heads (1..64), head_dim (128) and rank (0..16) are used; heads > 64 is
 *                rejected with QWM_ERR_SHAPE
 *   dev_status   device int32 where a device-side error (QWM_ERR_NOT_CONVERGED, ...) is recorded
 *                if the word is still 0, or NULL
 * The first call in each CUDA context (a device's primary context, or a context the caller made
 * current itself) looks up the array's device address in that context (cudaGetSymbolAddress);
 * make that first call before any stream capture.  With lazy module loading (the CUDA default)
 * the array is reserved on the device when the library's module loads, which is that first
 * call: a caller whose memory budget is fixed at start-up should make one call at start-up (with
 * nq == 0 and its own S, n, w, eigvals, u_r buffers, which that call recomputes from S and n).
 * All calls share the one array and each call leaves its contents behind: calls that can run on
 * the GPU at the same time (on different streams) race on it and must be ordered by the caller. */
QWM_API qwm_status qwm_update_query_stats_noalloc(const qwm_config *cfg, const uint16_t *q, int64_t nq, float *S,
                                                  int64_t *n, float *w, float *eigvals, uint16_t *u_r,
                                                  int32_t *dev_status, qwm_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* QWM_H_ */
