// Step 5': BF16 reconstruction of one packed chunk (QuantWM English v2 summary §D.1:
// the fused decoder unpacks the INT2 residuals, rebuilds the affine parameters,
// gathers the centroids and adds the PSAC term; Chinese summary step (5)).
//   K_hat = (mu^K_idx + m + s q) + sum_k (sC c_k) U_r[:, k],   V_hat = mu^V_idx + m + s q.
// One thread per (head, token, 8-channel block): 16-byte centroid loads and stores.
#include "qwm_internal.cuh"

namespace {

constexpr int D = QWM_D;

__global__ void dequant_kernel(qwm_chunk ch, int H, int C, int R, int compact, uint16_t *__restrict__ k_hat,
                               uint16_t *__restrict__ v_hat) {
  const int64_t N = ch.n_tokens;
  const int64_t total = (int64_t)H * N * (D / 8);
  const int G = D / QWM_GROUP;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int cb = (int)(e % (D / 8));
    const int64_t row = e / (D / 8);  // h * N + token
    const int h = (int)(row / N);
    const int c0 = 8 * cb, g = c0 / QWM_GROUP;
    for (int pass = 0; pass < 2; pass++) {
      uint16_t *dst = pass ? v_hat : k_hat;
      if (!dst) continue;
      const uint8_t *codes = pass ? ch.v_codes : ch.k_codes;
      const void *idx = pass ? ch.v_idx : ch.k_idx;  // uint16 for 1024-centroid codebooks
      const uint16_t *sc = pass ? ch.v_scale : ch.k_scale;
      const uint16_t *mn = pass ? ch.v_min : ch.k_min;
      const uint16_t *cent = pass ? ch.cent_v : ch.cent_k;
      float s, m;
      if (compact) {  // s = sigma s8 (sigma a power of two), m = -z s: exact
        const int64_t tiles = (N + 127) / 128;
        const float sg = f16_to_f32((pass ? ch.v_sigma : ch.k_sigma)[((int64_t)h * tiles + (row - (int64_t)h * N) / 128) * G + g]);
        s = sg * (float)(pass ? ch.v_s8 : ch.k_s8)[row * G + g];
        m = -(float)(((pass ? ch.v_zp : ch.k_zp)[row] >> (2 * g)) & 3u) * s;
      } else {
        s = f16_to_f32(sc[row * G + g]);
        m = f16_to_f32(mn[row * G + g]);
      }
      const uint32_t b2 = *(const uint16_t *)(codes + row * (D / 4) + 2 * cb);  // 8 codes
      const int j = min(C > 256 ? (int)((const uint16_t *)idx)[row] : (int)((const uint8_t *)idx)[row],
                        C - 1);  // never read past the codebook
      const uint4 mu = *(const uint4 *)(cent + ((int64_t)h * C + j) * D + c0);
      const uint32_t muw[4] = {mu.x, mu.y, mu.z, mu.w};
      float x[8];
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const float q = (float)((b2 >> (2 * u)) & 3u);
        const float rhat = __fmaf_rn(s, q, m);
        const float muf = __uint_as_float((u & 1) ? (muw[u / 2] & 0xFFFF0000u) : (muw[u / 2] << 16));
        x[u] = __fadd_rn(muf, rhat);
      }
      if (pass == 0 && R > 0) {
        const float sC = f16_to_f32(ch.c_scale[row]);
        const int8_t *cc = ch.c + row * R;
        const uint16_t *U = ch.u_r + (int64_t)h * D * R;
#pragma unroll 4
        for (int kk = 0; kk < R; kk++) {
          const float chat = sC * (float)cc[kk];
#pragma unroll
          for (int u = 0; u < 8; u++) x[u] = fmaf(chat, bf16_to_f32(U[(c0 + u) * R + kk]), x[u]);
        }
      }
      uint32_t o[4];
#pragma unroll
      for (int u = 0; u < 4; u++)
        o[u] = (uint32_t)f32_to_bf16_rn(x[2 * u]) | ((uint32_t)f32_to_bf16_rn(x[2 * u + 1]) << 16);
      *(uint4 *)(dst + row * D + c0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

cudaError_t launch_dequantize(const qwm_config &cfg, const qwm_chunk &ch, uint16_t *k_hat, uint16_t *v_hat,
                              cudaStream_t st) {
  const int64_t total = (int64_t)cfg.heads * ch.n_tokens * (D / 8);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 64) blocks = 152 * 64;
  dequant_kernel<<<(int)blocks, threads, 0, st>>>(ch, cfg.heads, cfg.n_centroids, ch.rank_eff,
                                                  cfg.storage == QWM_STORAGE_COMPACT ? 1 : 0, k_hat, v_hat);
  return cudaGetLastError();
}
