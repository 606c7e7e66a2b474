// Comparison baselines of the ablation workload (not the QuantWM path):
//   QVG progressive residual quantisation (Quant VideoGen summary §2B): the stage residual and the
//     fused decoder of a two-stage chunk;
//   KIVI-style INT2: Keys per channel over groups of 32 tokens, Values per token over groups of 32
//     channels, with the QuantWM INT2 encoder.
// All HBM-bound elementwise kernels: 16-byte (or 8-byte) vector accesses, grid-stride loops.
#include "../../include/qwm_baselines.h"
#include "qwm_internal.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int KG = QWM_KIVI_GROUP;

__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ int load_idx(const void *idx, int64_t i, bool wide) {
  return wide ? (int)((const uint16_t *)idx)[i] : (int)((const uint8_t *)idx)[i];
}

// out = bf16(x - mu_idx), one thread per (row, 8 channels)
__global__ void prq_residual_kernel(const uint16_t *__restrict__ x, int64_t n, int H, int C,
                                    const uint16_t *__restrict__ cent, const void *__restrict__ idx,
                                    uint16_t *__restrict__ out) {
  const int64_t total = (int64_t)H * n * (D / 8);
  const bool wide = C > 256;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = e / (D / 8);
    const int cb = (int)(e % (D / 8)), h = (int)(row / n);
    const int j = min(load_idx(idx, row, wide), C - 1);
    const uint4 xv = *(const uint4 *)(x + row * D + 8 * cb);
    const uint4 mv = *(const uint4 *)(cent + ((int64_t)h * C + j) * D + 8 * cb);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, mw[4] = {mv.x, mv.y, mv.z, mv.w};
    uint32_t o[4];
#pragma unroll
    for (int u = 0; u < 4; u++)
      o[u] = (uint32_t)f32_to_bf16_rn(__fsub_rn(lo16(xw[u]), lo16(mw[u]))) |
             ((uint32_t)f32_to_bf16_rn(__fsub_rn(hi16(xw[u]), hi16(mw[u]))) << 16);
    *(uint4 *)(out + row * D + 8 * cb) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// x_hat = bf16(mu1 + (mu2 + (m + s q))), one thread per (row, 8 channels), Keys then Values
__global__ void prq_dequant_kernel(qwm_chunk ch, int H, int C, const uint16_t *__restrict__ c1k,
                                   const void *__restrict__ i1k, const uint16_t *__restrict__ c1v,
                                   const void *__restrict__ i1v, uint16_t *__restrict__ k_hat,
                                   uint16_t *__restrict__ v_hat) {
  const int64_t N = ch.n_tokens, total = (int64_t)H * N * (D / 8);
  const bool wide = C > 256;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = e / (D / 8);
    const int cb = (int)(e % (D / 8)), h = (int)(row / N), c0 = 8 * cb, g = c0 / QWM_GROUP;
    for (int pass = 0; pass < 2; pass++) {
      uint16_t *dst = pass ? v_hat : k_hat;
      if (!dst) continue;
      const float s = f16_to_f32((pass ? ch.v_scale : ch.k_scale)[row * 2 + g]);
      const float m = f16_to_f32((pass ? ch.v_min : ch.k_min)[row * 2 + g]);
      const uint32_t b2 = *(const uint16_t *)((pass ? ch.v_codes : ch.k_codes) + row * (D / 4) + 2 * cb);
      const int j2 = min(load_idx(pass ? ch.v_idx : ch.k_idx, row, wide), C - 1);
      const int j1 = min(load_idx(pass ? i1v : i1k, row, wide), C - 1);
      const uint4 m2 = *(const uint4 *)((pass ? ch.cent_v : ch.cent_k) + ((int64_t)h * C + j2) * D + c0);
      const uint4 m1 = *(const uint4 *)((pass ? c1v : c1k) + ((int64_t)h * C + j1) * D + c0);
      const uint32_t w2[4] = {m2.x, m2.y, m2.z, m2.w}, w1[4] = {m1.x, m1.y, m1.z, m1.w};
      float xo[8];
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const float q = (float)((b2 >> (2 * u)) & 3u);
        const float mu2 = (u & 1) ? hi16(w2[u / 2]) : lo16(w2[u / 2]);
        const float mu1 = (u & 1) ? hi16(w1[u / 2]) : lo16(w1[u / 2]);
        xo[u] = __fadd_rn(mu1, __fadd_rn(mu2, __fmaf_rn(s, q, m)));
      }
      uint32_t o[4];
#pragma unroll
      for (int u = 0; u < 4; u++)
        o[u] = (uint32_t)f32_to_bf16_rn(xo[2 * u]) | ((uint32_t)f32_to_bf16_rn(xo[2 * u + 1]) << 16);
      *(uint4 *)(dst + row * D + c0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// KIVI Keys: one thread per (head, 32-token group, 4 channels); a warp covers a whole token row
__global__ void kivi_keys_kernel(const uint16_t *__restrict__ k, int64_t n, int H, uint8_t *__restrict__ codes,
                                 uint16_t *__restrict__ scale, uint16_t *__restrict__ minv, int32_t *status) {
  const int64_t ng = (n + KG - 1) / KG, total = (int64_t)H * ng * (D / 4);
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int c4 = (int)(e % (D / 4));
    const int64_t hg = e / (D / 4), h = hg / ng, tg = hg % ng;
    const int64_t t0 = tg * KG;
    const int len = (int)((n - t0) < KG ? (n - t0) : KG);
    const uint16_t *src = k + (h * n + t0) * D + 4 * c4;
    float mn[4], mx[4];
#pragma unroll
    for (int u = 0; u < 4; u++) { mn[u] = INFINITY; mx[u] = -INFINITY; }
    for (int t = 0; t < len; t++) {
      const uint2 v = *(const uint2 *)(src + (int64_t)t * D);
      const float f[4] = {lo16(v.x), hi16(v.x), lo16(v.y), hi16(v.y)};
#pragma unroll
      for (int u = 0; u < 4; u++) { mn[u] = fminf(mn[u], f[u]); mx[u] = fmaxf(mx[u], f[u]); }
    }
    float m[4], s[4], inv[4];
    uint16_t mb[4], sb[4];
#pragma unroll
    for (int u = 0; u < 4; u++) int2_params(mn[u], mx[u], m[u], s[u], inv[u], mb[u], sb[u], status);
    const int64_t pg = (h * ng + tg) * D + 4 * c4;
    *(uint2 *)(scale + pg) = make_uint2((uint32_t)sb[0] | ((uint32_t)sb[1] << 16), (uint32_t)sb[2] | ((uint32_t)sb[3] << 16));
    *(uint2 *)(minv + pg) = make_uint2((uint32_t)mb[0] | ((uint32_t)mb[1] << 16), (uint32_t)mb[2] | ((uint32_t)mb[3] << 16));
    for (int t = 0; t < len; t++) {
      const uint2 v = *(const uint2 *)(src + (int64_t)t * D);
      const float f[4] = {lo16(v.x), hi16(v.x), lo16(v.y), hi16(v.y)};
      uint32_t b = 0;
#pragma unroll
      for (int u = 0; u < 4; u++) b |= int2_code(f[u], m[u], s[u], inv[u]) << (2 * u);
      codes[(h * n + t0 + t) * (D / 4) + c4] = (uint8_t)b;
    }
  }
}

// KIVI Values: one thread per (head, token, 32-channel group)
__global__ void kivi_values_kernel(const uint16_t *__restrict__ v, int64_t n, int H, uint8_t *__restrict__ codes,
                                   uint16_t *__restrict__ scale, uint16_t *__restrict__ minv, int32_t *status) {
  const int64_t total = (int64_t)H * n * (D / KG);
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = e / (D / KG);
    const int cg = (int)(e % (D / KG));
    const uint4 *src = (const uint4 *)(v + row * D + KG * cg);
    float f[KG];
#pragma unroll
    for (int i = 0; i < KG / 8; i++) {
      const uint4 w = src[i];
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int u = 0; u < 4; u++) { f[8 * i + 2 * u] = lo16(ww[u]); f[8 * i + 2 * u + 1] = hi16(ww[u]); }
    }
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < KG; i++) { mn = fminf(mn, f[i]); mx = fmaxf(mx, f[i]); }
    float m, s, inv;
    uint16_t mb, sb;
    int2_params(mn, mx, m, s, inv, mb, sb, status);
    scale[row * (D / KG) + cg] = sb;
    minv[row * (D / KG) + cg] = mb;
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < KG; i++) w[i / 16] |= int2_code(f[i], m, s, inv) << (2 * (i % 16));
    *(uint2 *)(codes + row * (D / 4) + (KG / 4) * cg) = make_uint2(w[0], w[1]);
  }
}

// KIVI decode: x_hat = bf16(m + s q), one thread per (row, 8 channels), Keys then Values
__global__ void kivi_dequant_kernel(qwm_kivi_chunk ch, int H, uint16_t *__restrict__ k_hat,
                                    uint16_t *__restrict__ v_hat) {
  const int64_t N = ch.n_tokens, ng = (N + KG - 1) / KG, total = (int64_t)H * N * (D / 8);
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = e / (D / 8);
    const int cb = (int)(e % (D / 8)), c0 = 8 * cb;
    const int64_t h = row / N, t = row % N;
    for (int pass = 0; pass < 2; pass++) {
      uint16_t *dst = pass ? v_hat : k_hat;
      if (!dst) continue;
      const uint32_t b2 = *(const uint16_t *)((pass ? ch.v_codes : ch.k_codes) + row * (D / 4) + 2 * cb);
      float xo[8];
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const int c = c0 + u;
        const int64_t pg = pass ? row * (D / KG) + c / KG : (h * ng + t / KG) * D + c;
        const float s = f16_to_f32((pass ? ch.v_scale : ch.k_scale)[pg]);
        const float m = f16_to_f32((pass ? ch.v_min : ch.k_min)[pg]);
        xo[u] = __fmaf_rn(s, (float)((b2 >> (2 * u)) & 3u), m);
      }
      uint32_t o[4];
#pragma unroll
      for (int u = 0; u < 4; u++)
        o[u] = (uint32_t)f32_to_bf16_rn(xo[2 * u]) | ((uint32_t)f32_to_bf16_rn(xo[2 * u + 1]) << 16);
      *(uint4 *)(dst + row * D + c0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

int grid_for(int64_t total) {
  int64_t b = (total + 255) / 256;
  if (b > 152 * 32) b = 152 * 32;
  return b < 1 ? 1 : (int)b;
}

bool al16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" {

qwm_status qwm_kivi_quantize(qwm_ctx *ctx, const uint16_t *k, const uint16_t *v, int64_t n, qwm_kivi_chunk *out,
                             qwm_stream stream) {
  if (!ctx || !k || !v || !out || n < 0) return QWM_ERR_ARG;
  if (out->n_tokens != n) return QWM_ERR_SHAPE;
  const void *req[] = {out->k_codes, out->v_codes, out->k_scale, out->k_min, out->v_scale, out->v_min};
  for (const void *p : req)
    if (!p) return QWM_ERR_ARG;
  if (!al16(k) || !al16(v) || !al16(out->k_codes) || !al16(out->v_codes)) return QWM_ERR_ALIGN;
  if (n == 0) return QWM_OK;
  const int H = ctx->cfg.heads;
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t ng = (n + KG - 1) / KG;
  kivi_keys_kernel<<<grid_for((int64_t)H * ng * (D / 4)), 256, 0, st>>>(k, n, H, out->k_codes, out->k_scale,
                                                                         out->k_min, ctx->status);
  kivi_values_kernel<<<grid_for((int64_t)H * n * (D / KG)), 256, 0, st>>>(v, n, H, out->v_codes, out->v_scale,
                                                                          out->v_min, ctx->status);
  return cudaGetLastError() == cudaSuccess ? QWM_OK : QWM_ERR_CUDA;
}

qwm_status qwm_kivi_dequantize(qwm_ctx *ctx, const qwm_kivi_chunk *chunk, uint16_t *k_hat, uint16_t *v_hat,
                               qwm_stream stream) {
  if (!ctx || !chunk || chunk->n_tokens < 0) return QWM_ERR_ARG;
  if ((k_hat && !al16(k_hat)) || (v_hat && !al16(v_hat))) return QWM_ERR_ALIGN;
  if (chunk->n_tokens == 0 || (!k_hat && !v_hat)) return QWM_OK;
  const int H = ctx->cfg.heads;
  kivi_dequant_kernel<<<grid_for((int64_t)H * chunk->n_tokens * (D / 8)), 256, 0, (cudaStream_t)stream>>>(
      *chunk, H, k_hat, v_hat);
  return cudaGetLastError() == cudaSuccess ? QWM_OK : QWM_ERR_CUDA;
}

qwm_status qwm_prq_residual(qwm_ctx *ctx, const uint16_t *x, int64_t n, const uint16_t *cent, const void *idx,
                            uint16_t *out, qwm_stream stream) {
  if (!ctx || !x || !cent || !idx || !out || n < 0) return QWM_ERR_ARG;
  if (!al16(x) || !al16(cent) || !al16(out)) return QWM_ERR_ALIGN;
  if (n == 0) return QWM_OK;
  const int H = ctx->cfg.heads;
  prq_residual_kernel<<<grid_for((int64_t)H * n * (D / 8)), 256, 0, (cudaStream_t)stream>>>(
      x, n, H, ctx->cfg.n_centroids, cent, idx, out);
  return cudaGetLastError() == cudaSuccess ? QWM_OK : QWM_ERR_CUDA;
}

qwm_status qwm_prq_dequantize(qwm_ctx *ctx, const qwm_chunk *last, const uint16_t *cent1_k, const void *idx1_k,
                              const uint16_t *cent1_v, const void *idx1_v, uint16_t *k_hat, uint16_t *v_hat,
                              qwm_stream stream) {
  if (!ctx || !last || !cent1_k || !idx1_k || !cent1_v || !idx1_v || last->n_tokens < 0) return QWM_ERR_ARG;
  if (last->rank_eff != 0) return QWM_ERR_UNSUPPORTED;
  const void *req[] = {last->k_codes, last->v_codes, last->k_idx, last->v_idx, last->k_scale,
                       last->k_min,   last->v_scale, last->v_min, last->cent_k, last->cent_v};
  for (const void *p : req)
    if (!p) return QWM_ERR_ARG;
  if (!al16(cent1_k) || !al16(cent1_v) || (k_hat && !al16(k_hat)) || (v_hat && !al16(v_hat))) return QWM_ERR_ALIGN;
  if (last->n_tokens == 0 || (!k_hat && !v_hat)) return QWM_OK;
  const int H = ctx->cfg.heads;
  prq_dequant_kernel<<<grid_for((int64_t)H * last->n_tokens * (D / 8)), 256, 0, (cudaStream_t)stream>>>(
      *last, H, ctx->cfg.n_centroids, cent1_k, idx1_k, cent1_v, idx1_v, k_hat, v_hat);
  return cudaGetLastError() == cudaSuccess ? QWM_OK : QWM_ERR_CUDA;
}

}  // extern "C"
