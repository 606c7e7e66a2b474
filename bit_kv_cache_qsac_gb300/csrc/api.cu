// C ABI entry points of libqwm.so: argument checks, context, workspace, dispatch.
#include <stdlib.h>
#include <string.h>

#include "qwm_internal.cuh"

namespace {

constexpr int kStatsSplits = 8;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  size_t status, stats_part, q_img, q_bfull, q_mfull, total;
  size_t km_sum[2], km_cnt[2], km_cent[2], km_img[2], km_prev[2];  // two k-means workspaces (Keys, Values)
};

Layout layout_of(const qwm_config &c) {
  Layout L{};
  size_t off = 0;
  L.status = off; off = align_up(off + 256, 256);
  L.stats_part = off; off = align_up(off + (size_t)kStatsSplits * c.heads * QWM_D * QWM_D * sizeof(float), 256);
  const size_t G = (size_t)kmeans_ctas_per_head(c.heads, QWM_MAX_SMS);
  for (int i = 0; i < 2; i++) {
    L.km_sum[i] = off; off = align_up(off + G * c.heads * c.n_centroids * QWM_D * sizeof(float), 256);
    L.km_cnt[i] = off; off = align_up(off + G * c.heads * c.n_centroids * sizeof(int32_t), 256);
    L.km_cent[i] = off; off = align_up(off + (size_t)c.heads * c.n_centroids * QWM_D * sizeof(float), 256);
    off = align_up(off, 1024);
    L.km_img[i] = off; off = align_up(off + kmeans_image_bytes(c.heads, c.n_centroids), 1024);
    L.km_prev[i] = off;  // resident codebooks only (uint8 assignments)
    off = align_up(off + (c.n_centroids <= QWM_MAX_RESIDENT_CENTROIDS ? (size_t)c.heads * kKmPrevTokens : 0), 256);
  }
  L.q_img = off; off = align_up(off + quantize_image_bytes(c.heads, c.n_centroids), 1024);
  L.q_bfull = off; off = align_up(off + (size_t)c.heads * c.n_centroids * QWM_D * sizeof(float), 256);
  L.q_mfull = off; off = align_up(off + (size_t)c.heads * QWM_D * QWM_D * sizeof(float), 256);
  L.total = off;
  return L;
}

qwm_status check_config(const qwm_config *c) {
  if (!c) return QWM_ERR_ARG;
  if (c->heads < 1 || c->head_dim < 1 || c->n_centroids < 1 || c->group < 1 || c->top_m < 1 || c->rank < 0 ||
      c->bits < 1 || c->kmeans_iters < 1)
    return QWM_ERR_ARG;
  if (c->head_dim != QWM_D || c->group != QWM_GROUP) return QWM_ERR_SHAPE;
  if (c->bits != 2) return QWM_ERR_UNSUPPORTED;
  if (!(c->n_centroids == 64 || c->n_centroids == 128 || c->n_centroids == 256 || c->n_centroids == 1024))
    return QWM_ERR_SHAPE;
  if (c->top_m > QWM_MAX_TOPM || c->top_m > c->n_centroids) return QWM_ERR_SHAPE;
  if (c->rank > QWM_MAX_RANK) return QWM_ERR_SHAPE;
  if (c->kmeans_iters > 100) return QWM_ERR_SHAPE;
  if ((int64_t)c->heads > 4096) return QWM_ERR_SHAPE;
  if (c->storage != QWM_STORAGE_FP16 && c->storage != QWM_STORAGE_COMPACT) return QWM_ERR_ARG;
  if (c->psac_gate != 0 && c->psac_gate != 1) return QWM_ERR_ARG;
  if (c->test_flags & ~QWM_TEST_EXPIRE_WAIT) return QWM_ERR_ARG;
  return QWM_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

qwm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QWM_OK : QWM_ERR_CUDA; }

// A chunk descriptor is usable when every pointer it needs is set and aligned.
// A chunk descriptor is usable when every pointer it needs is set and aligned.  `packing`: for
// qwm_quantize_kv (the bf16 codebooks are read, the stored fp16 ones written); otherwise for
// qwm_attend / qwm_dequantize (the stored codebooks and the coefficient layout are read).
qwm_status check_chunk(const qwm_config &c, const qwm_chunk *ch, bool packing) {
  if (!ch) return QWM_ERR_ARG;
  if (ch->n_tokens < 0) return QWM_ERR_ARG;
  if (ch->kind == QWM_CHUNK_BF16) {
    if (ch->rank_eff != 0 || ch->causal_tpf < 0) return QWM_ERR_ARG;
    if (!ch->k_raw || !ch->v_raw) return QWM_ERR_ARG;
    if (!aligned16(ch->k_raw) || !aligned16(ch->v_raw)) return QWM_ERR_ALIGN;
    return QWM_OK;
  }
  if (ch->kind != QWM_CHUNK_PACKED) return QWM_ERR_ARG;
  if (ch->rank_eff != 0 && ch->rank_eff != c.rank) return QWM_ERR_SHAPE;
  if (ch->c_layout != QWM_C_DENSE && ch->c_layout != QWM_C_PER_HEAD) return QWM_ERR_ARG;
  if (packing && ch->c_layout != QWM_C_DENSE) return QWM_ERR_ARG;
  const bool compact = c.storage == QWM_STORAGE_COMPACT;
  const void *req[] = {ch->k_codes, ch->v_codes, ch->k_idx, ch->v_idx, ch->cent_k16, ch->cent_v16,
                       compact ? (const void *)ch->k_s8 : ch->k_scale, compact ? (const void *)ch->k_zp : ch->k_min,
                       compact ? (const void *)ch->v_s8 : ch->v_scale, compact ? (const void *)ch->v_zp : ch->v_min,
                       compact ? (const void *)ch->k_sigma : ch->k_codes, compact ? (const void *)ch->v_sigma : ch->v_codes,
                       packing ? (const void *)ch->cent_k : ch->k_codes, packing ? (const void *)ch->cent_v : ch->k_codes};
  for (const void *p : req) {
    if (!p) return QWM_ERR_ARG;
    if (!aligned16(p)) return QWM_ERR_ALIGN;
  }
  if (ch->rank_eff > 0) {
    const void *psac[] = {ch->c, ch->c_scale, ch->u_r};
    for (const void *p : psac) {
      if (!p) return QWM_ERR_ARG;
      if (ch->c_layout == QWM_C_DENSE && !aligned16(p)) return QWM_ERR_ALIGN;
    }
    if (ch->c_layout == QWM_C_PER_HEAD) {  // rows of r_h bytes: c and c_scale need no 16-byte alignment
      if (!ch->c_heads || !ch->c_mask || !ch->c_tile_rank) return QWM_ERR_ARG;
      if (!aligned16(ch->c_heads) || !aligned16(ch->c_mask) || !aligned16(ch->c_tile_rank) || !aligned16(ch->u_r) ||
          ((uintptr_t)ch->c_scale & 1u))
        return QWM_ERR_ALIGN;
    }
  }
  return QWM_OK;
}

}  // namespace

extern "C" {

const char *qwm_status_string(qwm_status s) {
  switch (s) {
    case QWM_OK: return "ok";
    case QWM_ERR_ARG: return "invalid argument";
    case QWM_ERR_SHAPE: return "unsupported shape";
    case QWM_ERR_ALIGN: return "pointer not 16-byte aligned";
    case QWM_ERR_CUDA: return "CUDA error";
    case QWM_ERR_NOT_CONVERGED: return "eigensolver did not converge within its sweep limit";
    case QWM_ERR_UNSUPPORTED: return "unsupported configuration";
    case QWM_ERR_RANGE: return "value outside the fp16 range";
    case QWM_ERR_DEVICE_TIMEOUT: return "a kernel gave up after its internal wait limit";
  }
  return "unknown status";
}

size_t qwm_workspace_bytes(const qwm_config *cfg) {
  if (check_config(cfg) != QWM_OK) return 0;
  return layout_of(*cfg).total;
}

qwm_status qwm_create(const qwm_config *cfg, qwm_ctx **out) {
  if (!out) return QWM_ERR_ARG;
  *out = nullptr;
  qwm_status s = check_config(cfg);
  if (s != QWM_OK) return s;
  qwm_ctx *ctx = (qwm_ctx *)calloc(1, sizeof(qwm_ctx));
  if (!ctx) return QWM_ERR_ARG;
  ctx->cfg = *cfg;
  if (cudaGetDevice(&ctx->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess) {
    free(ctx);
    return QWM_ERR_CUDA;
  }
  Layout L = layout_of(*cfg);
  if (cudaMalloc(&ctx->ws, L.total) != cudaSuccess) {
    free(ctx);
    return QWM_ERR_CUDA;
  }
  if (cudaMemset(ctx->ws, 0, L.total) != cudaSuccess) {
    cudaFree(ctx->ws);
    free(ctx);
    return QWM_ERR_CUDA;
  }
  char *base = (char *)ctx->ws;
  ctx->ws_bytes = L.total;
  ctx->status = (int32_t *)(base + L.status);
  ctx->stats_part = (float *)(base + L.stats_part);
  ctx->stats_splits = kStatsSplits;
  for (int i = 0; i < 2; i++) {
    ctx->km[i].sum = (float *)(base + L.km_sum[i]);
    ctx->km[i].cnt = (int32_t *)(base + L.km_cnt[i]);
    ctx->km[i].cent = (float *)(base + L.km_cent[i]);
    ctx->km[i].img = (unsigned char *)(base + L.km_img[i]);
    ctx->km[i].prev =
        ctx->cfg.n_centroids <= QWM_MAX_RESIDENT_CENTROIDS ? (uint8_t *)(base + L.km_prev[i]) : nullptr;
  }
  ctx->q_img = (unsigned char *)(base + L.q_img);
  ctx->q_bfull = (float *)(base + L.q_bfull);
  ctx->q_mfull = (float *)(base + L.q_mfull);
  if (cudaStreamCreateWithFlags(&ctx->side, cudaStreamNonBlocking) != cudaSuccess) {
    cudaFree(ctx->ws);
    free(ctx);
    return QWM_ERR_CUDA;
  }
  if (cudaEventCreateWithFlags(&ctx->fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->join, cudaEventDisableTiming) != cudaSuccess) {
    if (ctx->fork) cudaEventDestroy(ctx->fork);
    cudaStreamDestroy(ctx->side);
    cudaFree(ctx->ws);
    free(ctx);
    return QWM_ERR_CUDA;
  }
  *out = ctx;
  return QWM_OK;
}

qwm_status qwm_destroy(qwm_ctx *ctx) {
  if (!ctx) return QWM_ERR_ARG;
  cudaError_t e = cudaStreamSynchronize(ctx->side);
  if (cudaEventDestroy(ctx->fork) != cudaSuccess) e = cudaErrorUnknown;
  if (cudaEventDestroy(ctx->join) != cudaSuccess) e = cudaErrorUnknown;
  if (cudaStreamDestroy(ctx->side) != cudaSuccess) e = cudaErrorUnknown;
  if (cudaFree(ctx->ws) != cudaSuccess) e = cudaErrorUnknown;
  free(ctx);
  return cuda_status(e);
}

qwm_status qwm_update_query_stats(qwm_ctx *ctx, const uint16_t *q, int64_t nq, float *S, int64_t *n, float *w,
                                  float *eigvals, uint16_t *u_r, qwm_stream stream) {
  if (!ctx || !S || !n || !w || !eigvals || nq < 0) return QWM_ERR_ARG;
  if (nq > 0 && !q) return QWM_ERR_ARG;
  if (ctx->cfg.rank > 0 && !u_r) return QWM_ERR_ARG;
  if ((q && !aligned16(q)) || !aligned16(S) || !aligned16(n) || !aligned16(w) || !aligned16(eigvals) ||
      (u_r && !aligned16(u_r)))
    return QWM_ERR_ALIGN;
  cudaStream_t st = (cudaStream_t)stream;
  const int H = ctx->cfg.heads;
  cudaError_t e = cudaSuccess;
  // splits: enough CTAs to cover the SMs, at most the workspace's partial slots
  int splits = (ctx->num_sms + H - 1) / H;
  if (splits > ctx->stats_splits) splits = ctx->stats_splits;
  if (splits < 1) splits = 1;
  if (nq > 0) e = launch_stats_partial(q, nq, H, ctx->stats_part, splits, ctx->status, st);
  if (e == cudaSuccess) e = launch_stats_finish(ctx->stats_part, nq > 0 ? splits : 0, nq, H, S, n, w, st);
  if (e == cudaSuccess)
    e = launch_eig(S, n, nq, H, ctx->cfg.rank, eigvals, u_r, ctx->status, st);
  return cuda_status(e);
}

static qwm_status check_fit(const qwm_ctx *ctx, const uint16_t *x, int64_t n, const uint16_t *init,
                            const uint16_t *cent) {
  if (!ctx || !x || !cent || n < 0) return QWM_ERR_ARG;
  if (n < ctx->cfg.n_centroids) return QWM_ERR_SHAPE;
  if (n * ctx->cfg.heads >= ((int64_t)1 << 31)) return QWM_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(cent) || (init && !aligned16(init))) return QWM_ERR_ALIGN;
  return QWM_OK;
}

// One fit with k-means workspace `ws` on stream st.
static cudaError_t fit_on(qwm_ctx *ctx, int ws, const uint16_t *x, int64_t n, const uint16_t *init, uint16_t *cent,
                          cudaStream_t st) {
  const int sms = ctx->num_sms < QWM_MAX_SMS ? ctx->num_sms : QWM_MAX_SMS;
  const KmWorkspace &w = ctx->km[ws];
  return launch_kmeans(x, n, ctx->cfg.heads, ctx->cfg.n_centroids, init, ctx->cfg.kmeans_iters, cent, w.cent, w.sum,
                       w.cnt, sms, ctx->status, w.img, w.prev, kKmPrevTokens, st);
}

qwm_status qwm_fit_centroids(qwm_ctx *ctx, const uint16_t *x, int64_t n, const uint16_t *init, uint16_t *cent,
                             qwm_stream stream) {
  qwm_status s = check_fit(ctx, x, n, init, cent);
  if (s != QWM_OK) return s;
  return cuda_status(fit_on(ctx, 0, x, n, init, cent, (cudaStream_t)stream));
}

qwm_status qwm_fit_centroids_kv(qwm_ctx *ctx, const uint16_t *k, const uint16_t *v, int64_t n, const uint16_t *init_k,
                                const uint16_t *init_v, uint16_t *cent_k, uint16_t *cent_v, qwm_stream stream) {
  qwm_status s = check_fit(ctx, k, n, init_k, cent_k);
  if (s == QWM_OK) s = check_fit(ctx, v, n, init_v, cent_v);
  if (s != QWM_OK) return s;
  const size_t cb = (size_t)ctx->cfg.heads * ctx->cfg.n_centroids * QWM_D * sizeof(uint16_t);
  const uintptr_t a0 = (uintptr_t)cent_k, b0 = (uintptr_t)cent_v;
  if (a0 < b0 + cb && b0 < a0 + cb) return QWM_ERR_ARG;  // the two outputs overlap
  const cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaEventRecord(ctx->fork, st);  // the Value fit starts after the work st holds
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->side, ctx->fork, 0);
  if (e == cudaSuccess) e = fit_on(ctx, 0, k, n, init_k, cent_k, st);
  if (e == cudaSuccess) e = fit_on(ctx, 1, v, n, init_v, cent_v, ctx->side);
  if (e == cudaSuccess) e = cudaEventRecord(ctx->join, ctx->side);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ctx->join, 0);
  return cuda_status(e);
}

static qwm_status quantize_impl(qwm_ctx *ctx, const uint16_t *k, const uint16_t *v, int64_t n, const float *w,
                                const float *S, const int64_t *n_seen, const uint16_t *u_r, qwm_chunk *out,
                                const qwm_debug *dbg, qwm_stream stream) {
  if (!ctx || !out || n < 0) return QWM_ERR_ARG;
  if (out->n_tokens != n) return QWM_ERR_SHAPE;
  if (out->kind != QWM_CHUNK_PACKED) return QWM_ERR_ARG;
  if (n == 0) {  // nothing to read or write: the chunk's pointers may be NULL
    out->rank_eff = (u_r != nullptr && ctx->cfg.rank > 0) ? ctx->cfg.rank : 0;
    return QWM_OK;
  }
  if (!k || !v) return QWM_ERR_ARG;
  if (n > ((int64_t)1 << 31) / QWM_D) return QWM_ERR_SHAPE;
  if (!aligned16(k) || !aligned16(v) || (w && !aligned16(w)) || (S && !aligned16(S)) ||
      (n_seen && !aligned16(n_seen)) || (u_r && !aligned16(u_r)))
    return QWM_ERR_ALIGN;
  if (out->kind != QWM_CHUNK_PACKED) return QWM_ERR_ARG;
  const bool psac = (u_r != nullptr) && ctx->cfg.rank > 0;
  out->rank_eff = psac ? ctx->cfg.rank : 0;
  qwm_status s = check_chunk(ctx->cfg, out, true);
  if (s != QWM_OK) return s;
  if (dbg) {
    if ((dbg->c_f32 && !aligned16(dbg->c_f32)) || (dbg->cand && !aligned16(dbg->cand)) ||
        (dbg->score && !aligned16(dbg->score)))
      return QWM_ERR_ALIGN;
  }
  if (n == 0) return QWM_OK;
  cudaError_t e = launch_quantize(ctx->cfg, k, v, n, w, S, n_seen, ctx->q_mfull, ctx->q_bfull, psac ? u_r : nullptr,
                                  *out, dbg, ctx->status, ctx->num_sms, ctx->q_img, (cudaStream_t)stream, ctx->side,
                                  ctx->fork, ctx->join);
  return cuda_status(e);
}

qwm_status qwm_quantize_kv(qwm_ctx *ctx, const uint16_t *k, const uint16_t *v, int64_t n, const float *w,
                           const uint16_t *u_r, qwm_chunk *out, const qwm_debug *dbg, qwm_stream stream) {
  return quantize_impl(ctx, k, v, n, w, nullptr, nullptr, u_r, out, dbg, stream);
}

qwm_status qwm_quantize_kv_full(qwm_ctx *ctx, const uint16_t *k, const uint16_t *v, int64_t n, const float *S,
                                const int64_t *n_seen, const uint16_t *u_r, qwm_chunk *out, const qwm_debug *dbg,
                                qwm_stream stream) {
  if (!S || !n_seen) return QWM_ERR_ARG;
  return quantize_impl(ctx, k, v, n, nullptr, S, n_seen, u_r, out, dbg, stream);
}

static qwm_status attend_impl(qwm_ctx *ctx, const uint16_t *q, int64_t nq, const qwm_chunk *chunks,
                              int32_t n_chunks, float softmax_scale, float *out, float *lse, int merge,
                              qwm_stream stream) {
  if (!ctx || !chunks || nq < 0 || n_chunks < 1) return QWM_ERR_ARG;
  if (nq > 0 && !out) return QWM_ERR_ARG;
  if (nq > 0 && !q) return QWM_ERR_ARG;
  if ((q && !aligned16(q)) || !aligned16(out)) return QWM_ERR_ALIGN;
  if (nq > ((int64_t)1 << 31) / QWM_D) return QWM_ERR_SHAPE;
  if (n_chunks > 128) return QWM_ERR_SHAPE;
  int64_t total = 0;
  for (int i = 0; i < n_chunks; i++) {
    if (chunks[i].n_tokens < 0) return QWM_ERR_ARG;
    if (chunks[i].n_tokens == 0) continue;  // skipped: its pointers may be NULL
    qwm_status s = check_chunk(ctx->cfg, &chunks[i], false);
    if (s != QWM_OK) return s;
    total += chunks[i].n_tokens;
  }
  if (total < 1) return QWM_ERR_SHAPE;
  if (nq == 0) return QWM_OK;
  cudaError_t e = launch_attend(ctx->cfg, q, nq, chunks, n_chunks, softmax_scale, out, lse, merge, ctx->num_sms,
                                ctx->status, (cudaStream_t)stream);
  return cuda_status(e);
}

qwm_status qwm_attend(qwm_ctx *ctx, const uint16_t *q, int64_t nq, const qwm_chunk *chunks, int32_t n_chunks,
                      float softmax_scale, float *out, qwm_stream stream) {
  return attend_impl(ctx, q, nq, chunks, n_chunks, softmax_scale, out, nullptr, 0, stream);
}

qwm_status qwm_attend_merge(qwm_ctx *ctx, const uint16_t *q, int64_t nq, const qwm_chunk *chunks, int32_t n_chunks,
                            float softmax_scale, float *out, float *lse, int32_t merge, qwm_stream stream) {
  if (merge != 0 && merge != 1) return QWM_ERR_ARG;
  if (nq > 0 && !lse) return QWM_ERR_ARG;
  if (lse && !aligned16(lse)) return QWM_ERR_ALIGN;
  return attend_impl(ctx, q, nq, chunks, n_chunks, softmax_scale, out, lse, merge, stream);
}

qwm_status qwm_dequantize(qwm_ctx *ctx, const qwm_chunk *chunk, uint16_t *k_hat, uint16_t *v_hat,
                          qwm_stream stream) {
  if (!ctx || !chunk || chunk->n_tokens < 0) return QWM_ERR_ARG;
  if (chunk->kind == QWM_CHUNK_BF16) return QWM_ERR_UNSUPPORTED;
  if (chunk->n_tokens == 0) return QWM_OK;
  qwm_status s = check_chunk(ctx->cfg, chunk, false);
  if (s != QWM_OK) return s;
  if ((k_hat && !aligned16(k_hat)) || (v_hat && !aligned16(v_hat))) return QWM_ERR_ALIGN;
  if (chunk->n_tokens == 0 || (!k_hat && !v_hat)) return QWM_OK;
  cudaError_t e = launch_dequantize(ctx->cfg, chunk, 1, k_hat, v_hat, (cudaStream_t)stream);
  return cuda_status(e);
}

qwm_status qwm_dequantize_chunks(qwm_ctx *ctx, const qwm_chunk *chunks, int32_t n_chunks, uint16_t *k_hat,
                                 uint16_t *v_hat, qwm_stream stream) {
  if (!ctx || !chunks || n_chunks < 1) return QWM_ERR_ARG;
  if (n_chunks > 128) return QWM_ERR_SHAPE;
  for (int i = 0; i < n_chunks; i++) {
    if (chunks[i].n_tokens < 0) return QWM_ERR_ARG;
    if (chunks[i].kind == QWM_CHUNK_BF16) return QWM_ERR_UNSUPPORTED;
    if (chunks[i].n_tokens == 0) continue;  // skipped: its pointers may be NULL
    qwm_status s = check_chunk(ctx->cfg, &chunks[i], false);
    if (s != QWM_OK) return s;
  }
  if ((k_hat && !aligned16(k_hat)) || (v_hat && !aligned16(v_hat))) return QWM_ERR_ALIGN;
  cudaError_t e = launch_dequantize(ctx->cfg, chunks, n_chunks, k_hat, v_hat, (cudaStream_t)stream);
  return cuda_status(e);
}

qwm_status qwm_select_rank(qwm_ctx *ctx, const float *eigvals, float energy, uint16_t *u_r, int32_t *head_rank,
                           qwm_stream stream) {
  if (!ctx || !eigvals || !head_rank) return QWM_ERR_ARG;
  if (!(energy >= 0.f && energy <= 1.f)) return QWM_ERR_ARG;
  if (ctx->cfg.rank > 0 && !u_r) return QWM_ERR_ARG;
  if (!aligned16(eigvals) || !aligned16(head_rank) || (u_r && !aligned16(u_r))) return QWM_ERR_ALIGN;
  return cuda_status(launch_select_rank(eigvals, energy, ctx->cfg.heads, ctx->cfg.rank, u_r, head_rank,
                                        (cudaStream_t)stream));
}

qwm_status qwm_psac_kept(qwm_ctx *ctx, const qwm_chunk *chunk, int32_t *kept, qwm_stream stream) {
  if (!ctx || !chunk || !kept) return QWM_ERR_ARG;
  if (chunk->kind != QWM_CHUNK_PACKED || chunk->c_layout != QWM_C_DENSE || chunk->rank_eff < 1) return QWM_ERR_ARG;
  if (chunk->n_tokens < 0 || !chunk->c_scale) return QWM_ERR_ARG;
  if (!aligned16(kept) || !aligned16(chunk->c_scale)) return QWM_ERR_ALIGN;
  return cuda_status(launch_psac_kept(chunk->c_scale, chunk->n_tokens, ctx->cfg.heads, kept, (cudaStream_t)stream));
}

qwm_status qwm_psac_plan(const qwm_config *cfg, int64_t n, const int32_t *head_rank, const int32_t *kept,
                         qwm_psac_head *plan, int64_t *c_bytes, int64_t *n_scales) {
  qwm_status s = check_config(cfg);
  if (s != QWM_OK) return s;
  if (n < 0 || !head_rank || !kept || !plan) return QWM_ERR_ARG;
  for (int h = 0; h < cfg->heads; h++)
    if (head_rank[h] < 0 || head_rank[h] > cfg->rank || kept[h] < 0 || kept[h] > n) return QWM_ERR_ARG;
  psac_plan_host(cfg->heads, n, head_rank, kept, plan, c_bytes, n_scales);
  return QWM_OK;
}

qwm_status qwm_psac_pack(qwm_ctx *ctx, const qwm_chunk *dense, const qwm_psac_head *plan, int8_t *c,
                         uint16_t *c_scale, uint32_t *c_mask, int32_t *c_tile_rank, qwm_stream stream) {
  if (!ctx || !dense || !plan || !c_mask || !c_tile_rank) return QWM_ERR_ARG;
  if (dense->kind != QWM_CHUNK_PACKED || dense->c_layout != QWM_C_DENSE || dense->rank_eff < 1) return QWM_ERR_ARG;
  if (dense->n_tokens < 1 || !dense->c || !dense->c_scale) return QWM_ERR_ARG;
  if (!aligned16(plan) || !aligned16(c_mask) || !aligned16(c_tile_rank) || ((uintptr_t)c_scale & 1u))
    return QWM_ERR_ALIGN;
  return cuda_status(launch_psac_pack(dense->c, dense->c_scale, dense->n_tokens, ctx->cfg.heads, dense->rank_eff, plan,
                                      c, c_scale, c_mask, c_tile_rank, (cudaStream_t)stream));
}

qwm_status qwm_sync_status(qwm_ctx *ctx, qwm_stream stream) {
  if (!ctx) return QWM_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, ctx->status, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return QWM_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return QWM_ERR_CUDA;
  if (h != 0 && cudaMemsetAsync(ctx->status, 0, sizeof(int32_t), st) != cudaSuccess) return QWM_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return QWM_ERR_CUDA;
  return (qwm_status)h;
}

}  // extern "C"
