// Steps 2-4: QSAC centroid assignment, INT2 residual codes and PSAC coefficients.
//
// QuantWM (Chinese summary "核心方法" and steps (2)-(4); Korean summary "무엇과 다른가",
// "어떻게 쓰나"):
//   Keys:   the top-M centroids by d_Q(k, mu) = sum_c w_c (k_c - mu_c)^2, then the one
//           minimising S(k, mu) = sum_g W_g R_g(k - mu)^2, W_g = sum_{c in G_g} w_c,
//           R_g = max - min of the residual over group g (64 channels).
//   Values: the nearest centroid (QVG's k-means assignment).
//   INT2:   per (token, group) m = fp16 round-down of min r, s = fp16 round-up of
//           (max r - m)/3, q = clamp(rint((r - m) * (1/s)), 0, 3); channel 4j+t of a token
//           goes to bits 2t..2t+1 of byte j.
//   PSAC:   K_hat_0 = mu + m + s q, E = K - K_hat_0, C = E U_r, INT8 per token with
//           sC = fp16 round-up of max|C|/127.
// The exactness-critical arithmetic (residual, range, scale, code) uses explicitly rounded
// intrinsics so that indices and codes match a plain IEEE implementation bit for bit.
//
// Layout: one warp per token.  Lane l holds channels 4l..4l+3, so lanes 0-15 cover group 0
// and lanes 16-31 group 1, and lane l writes byte l of the token's packed codes.  The Key
// and Value codebooks of the head sit transposed in shared memory ([channel][centroid]) so
// that the 32 lanes scoring 32 different centroids read consecutive words.
#include "qwm_internal.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct QuantParams {
  const uint16_t *k, *v;
  int64_t n;
  const float *w;
  const uint16_t *u_r;
  int C, top_m, rank;
  qwm_chunk out;
  float *dbg_c;
  int32_t *dbg_cand;
  float *dbg_score;
  int32_t *status;
};

__device__ __forceinline__ void load4_bf16(const uint16_t *p, float x[4]) {
  const uint2 raw = *(const uint2 *)p;
  x[0] = __uint_as_float(raw.x << 16); x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
  x[2] = __uint_as_float(raw.y << 16); x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
}

// min and max of v over the 16 lanes of this half-warp
__device__ __forceinline__ void group_minmax(float &mn, float &mx) {
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
}

// INT2 encode of the lane's 4 residuals (its group's min/max already reduced).
// Returns the packed byte; writes s and m (fp16 bits) and the decoded r_hat.
__device__ __forceinline__ uint32_t int2_encode(const float r[4], float mn, float mx, uint16_t &s_bits,
                                                uint16_t &m_bits, float rhat[4], int32_t *status) {
  const __half mh = __float2half_rd(mn);
  const float m = __half2float(mh);
  const float range = __fsub_ru(mx, m);
  __half sh = __float2half_ru(__fdiv_ru(range, 3.0f));
  if (range == 0.f) sh = __float2half_rn(0.f);
  const float s = __half2float(sh);
  if (!isfinite(m) || !isfinite(s)) qwm_dev_error(status, QWM_ERR_RANGE);
  s_bits = __half_as_ushort(sh);
  m_bits = __half_as_ushort(mh);
  uint32_t byte = 0;
  if (s == 0.f) {
#pragma unroll
    for (int u = 0; u < 4; u++) rhat[u] = m;
    return 0;
  }
  const float inv = __frcp_rn(s);
#pragma unroll
  for (int u = 0; u < 4; u++) {
    float qf = rintf(__fmul_rn(__fsub_rn(r[u], m), inv));
    qf = fminf(fmaxf(qf, 0.f), 3.f);
    byte |= ((uint32_t)qf) << (2 * u);
    rhat[u] = __fmaf_rn(s, qf, m);  // s * q is exact: one rounding, as m + s q
  }
  return byte;
}

// dynamic smem: cT_k [D][C] bf16, cT_v [D][C] bf16, u [D][r] fp32
__global__ void __launch_bounds__(kThreads) quantize_kernel(QuantParams p, int tok_per_cta) {
  extern __shared__ __align__(16) unsigned char qsm[];
  const int C = p.C, R = p.rank, M = p.top_m;
  uint16_t *cTk = (uint16_t *)qsm;
  uint16_t *cTv = cTk + D * C;
  float *us = (float *)(cTv + D * C);
  __shared__ float tk[kWarps][D], wsh[D];
  __shared__ float Wg[2];
  const int h = blockIdx.y, tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const uint16_t *ck = p.out.cent_k + (int64_t)h * C * D;
  const uint16_t *cv = p.out.cent_v + (int64_t)h * C * D;
  // transpose the codebooks: each thread reads 8 channels of one centroid (16 bytes) and
  // the lanes of a warp write consecutive centroids of one channel row
  for (int e = tid; e < C * (D / 8); e += kThreads) {
    const int j = e % C, cb = e / C;
    const uint4 a = *(const uint4 *)(ck + (int64_t)j * D + 8 * cb);
    const uint4 b = *(const uint4 *)(cv + (int64_t)j * D + 8 * cb);
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int u = 0; u < 4; u++) {
      cTk[(8 * cb + 2 * u) * C + j] = (uint16_t)(wa[u] & 0xFFFFu);
      cTk[(8 * cb + 2 * u + 1) * C + j] = (uint16_t)(wa[u] >> 16);
      cTv[(8 * cb + 2 * u) * C + j] = (uint16_t)(wb[u] & 0xFFFFu);
      cTv[(8 * cb + 2 * u + 1) * C + j] = (uint16_t)(wb[u] >> 16);
    }
  }
  for (int e = tid; e < D * R; e += kThreads) us[e] = bf16_to_f32(p.u_r[(int64_t)h * D * R + e]);
  for (int c = tid; c < D; c += kThreads) wsh[c] = p.w ? p.w[(int64_t)h * D + c] : 1.0f;
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, b = 0.f;
    for (int c = 0; c < 64; c++) a += wsh[c];
    for (int c = 64; c < 128; c++) b += wsh[c];
    Wg[0] = a; Wg[1] = b;
  }
  __syncthreads();
  const float Wmine = Wg[lane >> 4];
  const int per_lane = C / 32;
  const int G = D / QWM_GROUP;
  const int64_t t_begin = (int64_t)blockIdx.x * tok_per_cta;
  const int64_t t_end = min(p.n, t_begin + tok_per_cta);
  for (int64_t i = t_begin + warp; i < t_end; i += kWarps) {
    const int64_t row = (int64_t)h * p.n + i;
    float kx[4], vx[4];
    load4_bf16(p.k + row * D + 4 * lane, kx);
    load4_bf16(p.v + row * D + 4 * lane, vx);
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 4; u++) tk[warp][4 * lane + u] = kx[u];
    __syncwarp();
    // ---- d_Q to every centroid (lane scores centroids lane + 32 t) ----
    float dq[8];
#pragma unroll
    for (int t = 0; t < 8; t++) dq[t] = 0.f;
    for (int c = 0; c < D; c++) {
      const float kc = tk[warp][c], wc = wsh[c];
#pragma unroll
      for (int t = 0; t < 8; t++) {
        if (t < per_lane) {
          const float df = __fsub_rn(kc, bf16_to_f32(cTk[c * C + lane + 32 * t]));
          dq[t] = __fmaf_rn(wc, __fmul_rn(df, df), dq[t]);
        }
      }
    }
    // ---- top-M by repeated warp argmin (lower index on ties) and QSAC score ----
    float best_S = INFINITY;
    int best_j = 0x7fffffff;
    for (int m = 0; m < M; m++) {
      float bv = INFINITY;
      int bj = 0x7fffffff;
#pragma unroll
      for (int t = 0; t < 8; t++)
        if (t < per_lane && dq[t] < bv) { bv = dq[t]; bj = lane + 32 * t; }
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oj = __shfl_xor_sync(0xffffffffu, bj, off);
        if (ov < bv || (ov == bv && oj < bj)) { bv = ov; bj = oj; }
      }
      if (bj >= C) {  // only when every score is NaN (non-finite inputs)
        bj = 0;
        qwm_dev_error(p.status, QWM_ERR_RANGE);
      }
      if ((bj & 31) == lane) {
#pragma unroll
        for (int t = 0; t < 8; t++)
          if (t == (bj >> 5)) dq[t] = INFINITY;
      }
      if (p.dbg_cand && lane == 0) p.dbg_cand[row * M + m] = bj;
      // residual range of candidate bj over each group
      float mu[4];
      load4_bf16(ck + (int64_t)bj * D + 4 * lane, mu);
      float mn = INFINITY, mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const float r = __fsub_rn(kx[u], mu[u]);
        mn = fminf(mn, r);
        mx = fmaxf(mx, r);
      }
      group_minmax(mn, mx);
      const float Rg = __fsub_rn(mx, mn);
      const float mine = __fmul_rn(Wmine, __fmul_rn(Rg, Rg));
      const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
      const float S = (lane < 16) ? __fadd_rn(mine, other) : __fadd_rn(other, mine);
      if (S < best_S || (S == best_S && bj < best_j)) { best_S = S; best_j = bj; }
    }
    // ---- Values: nearest centroid ----
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 4; u++) tk[warp][4 * lane + u] = vx[u];
    __syncwarp();
    float dv[8];
#pragma unroll
    for (int t = 0; t < 8; t++) dv[t] = 0.f;
    for (int c = 0; c < D; c++) {
      const float vc = tk[warp][c];
#pragma unroll
      for (int t = 0; t < 8; t++) {
        if (t < per_lane) {
          const float df = __fsub_rn(vc, bf16_to_f32(cTv[c * C + lane + 32 * t]));
          dv[t] = __fmaf_rn(df, df, dv[t]);
        }
      }
    }
    float bv = INFINITY;
    int jv = 0x7fffffff;
#pragma unroll
    for (int t = 0; t < 8; t++)
      if (t < per_lane && dv[t] < bv) { bv = dv[t]; jv = lane + 32 * t; }
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oj = __shfl_xor_sync(0xffffffffu, jv, off);
      if (ov < bv || (ov == bv && oj < jv)) { bv = ov; jv = oj; }
    }
    if (jv >= C) {
      jv = 0;
      qwm_dev_error(p.status, QWM_ERR_RANGE);
    }
    if (best_j >= C) best_j = 0;
    // ---- INT2 of the Key and Value residuals ----
    const int g = lane >> 4;
    float muk[4], muv[4], rk[4], rv[4], rhk[4], rhv[4];
    load4_bf16(ck + (int64_t)best_j * D + 4 * lane, muk);
    load4_bf16(cv + (int64_t)jv * D + 4 * lane, muv);
    float mnk = INFINITY, mxk = -INFINITY, mnv = INFINITY, mxv = -INFINITY;
#pragma unroll
    for (int u = 0; u < 4; u++) {
      rk[u] = __fsub_rn(kx[u], muk[u]);
      rv[u] = __fsub_rn(vx[u], muv[u]);
      mnk = fminf(mnk, rk[u]); mxk = fmaxf(mxk, rk[u]);
      mnv = fminf(mnv, rv[u]); mxv = fmaxf(mxv, rv[u]);
    }
    group_minmax(mnk, mxk);
    group_minmax(mnv, mxv);
    uint16_t sk, mk, sv, mv;
    const uint32_t bk = int2_encode(rk, mnk, mxk, sk, mk, rhk, p.status);
    const uint32_t bvb = int2_encode(rv, mnv, mxv, sv, mv, rhv, p.status);
    p.out.k_codes[row * (D / 4) + lane] = (uint8_t)bk;
    p.out.v_codes[row * (D / 4) + lane] = (uint8_t)bvb;
    if ((lane & 15) == 0) {
      p.out.k_scale[row * G + g] = sk; p.out.k_min[row * G + g] = mk;
      p.out.v_scale[row * G + g] = sv; p.out.v_min[row * G + g] = mv;
    }
    if (lane == 0) {
      p.out.k_idx[row] = (uint8_t)best_j;
      p.out.v_idx[row] = (uint8_t)jv;
      if (p.dbg_score) p.dbg_score[row] = best_S;
    }
    // ---- PSAC: C = (K - K_hat_0) U_r, INT8 per token ----
    if (R > 0) {
      float e[4];
#pragma unroll
      for (int u = 0; u < 4; u++) e[u] = __fsub_rn(kx[u], __fadd_rn(muk[u], rhk[u]));
      float Cv[QWM_MAX_RANK];
#pragma unroll
      for (int kk = 0; kk < QWM_MAX_RANK; kk++) {
        float acc = 0.f;
        if (kk < R) {
#pragma unroll
          for (int u = 0; u < 4; u++) acc = fmaf(e[u], us[(4 * lane + u) * R + kk], acc);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        }
        Cv[kk] = acc;
      }
      float a = 0.f;
#pragma unroll
      for (int kk = 0; kk < QWM_MAX_RANK; kk++)
        if (kk < R) a = fmaxf(a, fabsf(Cv[kk]));
      __half sch = __float2half_ru(__fdiv_ru(a, 127.0f));
      if (a == 0.f) sch = __float2half_rn(0.f);
      const float sc = __half2float(sch);
      if (!isfinite(sc)) qwm_dev_error(p.status, QWM_ERR_RANGE);
      const float inv = sc > 0.f ? __frcp_rn(sc) : 0.f;
#pragma unroll
      for (int kk = 0; kk < QWM_MAX_RANK; kk++) {
        if (kk < R && lane == kk) {
          float qf = sc > 0.f ? rintf(__fmul_rn(Cv[kk], inv)) : 0.f;
          qf = fminf(fmaxf(qf, -127.f), 127.f);
          p.out.c[row * R + kk] = (int8_t)qf;
          if (p.dbg_c) p.dbg_c[row * R + kk] = Cv[kk];
        }
      }
      if (lane == 0) p.out.c_scale[row] = __half_as_ushort(sch);
    }
  }
}

}  // namespace

cudaError_t launch_quantize(const qwm_config &cfg, const uint16_t *k, const uint16_t *v, int64_t n, const float *w,
                            const uint16_t *u_r, const qwm_chunk &out, const qwm_debug *dbg, int32_t *status,
                            int num_sms, cudaStream_t st) {
  QuantParams p;
  p.k = k; p.v = v; p.n = n; p.w = w; p.u_r = u_r;
  p.C = cfg.n_centroids; p.top_m = cfg.top_m; p.rank = u_r ? cfg.rank : 0;
  p.out = out;
  p.dbg_c = dbg ? dbg->c_f32 : nullptr;
  p.dbg_cand = dbg ? dbg->cand : nullptr;
  p.dbg_score = dbg ? dbg->score : nullptr;
  p.status = status;
  const size_t smem = 2 * (size_t)D * p.C * sizeof(uint16_t) + (size_t)D * (p.rank > 0 ? p.rank : 1) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // about two CTAs per SM in total: the codebook transpose is paid once per CTA
  const int64_t blocks_per_head = (2LL * num_sms + cfg.heads - 1) / cfg.heads;
  int tok_per_cta = (int)((n + blocks_per_head - 1) / blocks_per_head);
  if (tok_per_cta < 32) tok_per_cta = 32;
  const int gx = (int)((n + tok_per_cta - 1) / tok_per_cta);
  quantize_kernel<<<dim3(gx, cfg.heads), kThreads, smem, st>>>(p, tok_per_cta);
  return cudaGetLastError();
}
