// Steps 2-4: QSAC centroid assignment, INT2 residual codes and PSAC coefficients, with the
// centroid distances computed on the tensor cores.
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
//
// Distance GEMM.  d_Q(k, mu_j) = sum_c w_c k_c^2 - 2 k.(w . mu_j) + sum_c w_c mu_jc^2; the first
// term is the same for every j, so the ranking uses score_j = nw_j - 2 k.b_j with b_j = w . mu_j
// split as b = hi + lo (bf16 each): two bf16 MMAs per 128-token tile (M = 128, N = C, K = 128)
// accumulate k.b_j in TMEM.  Values use b_j = mu_j (exact in bf16, one MMA) and nw_j = |mu_j|^2.
// The approximate scores pick the candidates; whenever the gap at the candidate boundary (Keys:
// between the M-th and (M+1)-th score; Values: between the best and the runner-up) is not
// larger than twice an error bound of the scores, the token falls back to exact fp32 distances
// against every centroid, so the candidate set is the exact one.  The range score S, the INT2
// codes and the PSAC coefficients are computed exactly in fp32 with explicitly rounded
// intrinsics, so that indices and codes match a plain IEEE implementation bit for bit.
//
// One CTA = one head x a contiguous range of 128-token tiles; 320 threads:
//   warp 0     TMA producer: K (or V) tiles as two [128][64] bf16 blocks, 128-byte swizzle, 2 stages
//   warp 1     TMEM owner and MMA issuer: tile g into TMEM buffer g % 2
//   warps 2-9  two epilogue warpgroups; group e owns the tiles g with g % 2 == e, thread = token
// All waits are bounded; on expiry the kernel records QWM_ERR_DEVICE_TIMEOUT and stops.
#include "qwm_internal.cuh"
#include "tc.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int TILE = 128;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int MAXM = QWM_MAX_TOPM + 1;
constexpr uint64_t kWaitNs = 1000000000ull;
// error bound of an approximate score: |err| <= kRel |k| max_j |b_j| + kRelN max_j |nw_j|
constexpr float kRel = 1.0f / 16384.0f;   // 2^-14
constexpr float kRelN = 1.0f / 65536.0f;  // 2^-16

struct QSmem {
  int bh, bl, x, nw, wv, U, total;
  __host__ __device__ QSmem(int C, bool key) {
    bh = 0;                             // 2 blocks of [C][64] bf16: hi of b (or mu for Values)
    bl = bh + 2 * C * 128;              // lo of b (Keys only)
    x = bl + (key ? 2 * C * 128 : 0);   // 2 stages x 2 blocks of [128][64]
    nw = x + 2 * 2 * TILE * 128;        // nw[C], then |b_j|[C]
    wv = nw + 8 * C;                    // w[D]
    U = wv + 4 * D;                     // U_r as fp32 [D][16], zero past the rank
    total = U + 4 * D * 16;
  }
};

struct QParams {
  int64_t n;
  const float *w;           // [H][D] or NULL
  const uint16_t *u_r;      // [H][D][R] or NULL
  const uint16_t *cent;     // [H][C][D] bf16 codebook
  int C, top_m, rank, G;
  uint8_t *codes, *idx;
  uint16_t *scale, *minv;
  int8_t *c;
  uint16_t *c_scale;
  float *dbg_c;
  int32_t *dbg_cand;
  float *dbg_score;
  int32_t *status;
};

__device__ __forceinline__ void bf16x8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int u = 0; u < 4; u++) {
    f[2 * u] = __uint_as_float(w[u] << 16);
    f[2 * u + 1] = __uint_as_float(w[u] & 0xFFFF0000u);
  }
}

// Insert (v, j) into the ascending list tv[0..m] of the m+1 smallest seen so far (thr == tv[m]).
// Indices arrive in increasing order, so the strict comparison keeps the lower index first on
// ties.  Only compile-time indices are used, so the lists stay in registers.
__device__ __forceinline__ void topk_insert(float (&tv)[MAXM], int (&ti)[MAXM], float &thr, int m, float v, int j) {
  if (!(v < thr)) return;
  bool placed = false;
#pragma unroll
  for (int k = MAXM - 1; k >= 1; k--) {
    if (k <= m && !placed) {
      if (tv[k - 1] > v) { tv[k] = tv[k - 1]; ti[k] = ti[k - 1]; }
      else { tv[k] = v; ti[k] = j; placed = true; }
    }
  }
  if (!placed) { tv[0] = v; ti[0] = j; }
  thr = tv[0];
#pragma unroll
  for (int k = 1; k < MAXM; k++)
    if (k == m) thr = tv[k];
}

// INT2 parameters of one group from its fp32 residual min and max.
__device__ __forceinline__ void int2_params(float mn, float mx, float &m, float &s, float &inv, uint16_t &m_bits,
                                            uint16_t &s_bits, int32_t *status) {
  const __half mh = __float2half_rd(mn);
  m = __half2float(mh);
  const float range = __fsub_ru(mx, m);
  __half sh = __float2half_ru(__fdiv_ru(range, 3.0f));
  if (range == 0.f) sh = __float2half_rn(0.f);
  s = __half2float(sh);
  if (!isfinite(m) || !isfinite(s)) qwm_dev_error(status, QWM_ERR_RANGE);
  inv = s > 0.f ? __frcp_rn(s) : 0.f;
  m_bits = __half_as_ushort(mh);
  s_bits = __half_as_ushort(sh);
}
__device__ __forceinline__ uint32_t int2_code(float r, float m, float s, float inv) {
  if (s == 0.f) return 0u;
  float qf = rintf(__fmul_rn(__fsub_rn(r, m), inv));
  qf = fminf(fmaxf(qf, 0.f), 3.f);
  return (uint32_t)qf;
}

// KEY: Keys (QSAC + PSAC) or Values (nearest centroid).  RMAX: 8 or 16, bound on the PSAC rank.
template <bool KEY, int RMAX>
__global__ void __launch_bounds__(kThreads, 1) quant_kernel(const __grid_constant__ TensorMap128 tmap,
                                                             const QParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char *sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t x_full[2], x_empty[2], t_full[2], t_empty[2], drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ float Wg[2], bmax_sh, nwmax_sh;
  const int C = p.C, M = KEY ? p.top_m : 1, R = KEY ? p.rank : 0;
  const QSmem L(C, KEY);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, cta = blockIdx.x;
  const int64_t tiles = (p.n + TILE - 1) / TILE;
  const int64_t per = (tiles + p.G - 1) / p.G;
  const int64_t tile0 = (int64_t)cta * per;
  const int64_t tile1 = tile0 + per < tiles ? tile0 + per : tiles;
  const int nt = tile1 > tile0 ? (int)(tile1 - tile0) : 0;
  float *nw = (float *)(sm + L.nw);
  float *bn = nw + C;
  float *wv = (float *)(sm + L.wv);
  float *Us = (float *)(sm + L.U);
  volatile int *abort_v = &abort_flag;
  const uint16_t *cent = p.cent + (int64_t)h * C * D;

  if (tid == 0) {
    for (int i = 0; i < 2; i++) {
      tc::mbar_init(&x_full[i], 1);
      tc::mbar_init(&x_empty[i], 4);
      tc::mbar_init(&t_full[i], 1);
      tc::mbar_init(&t_empty[i], 4);
    }
    tc::mbar_init(&drain, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&tmem_base_sh, 512);
    tc::tmem_relinquish();
  }
  // ---- per-head constants: weights, basis, distance operand (b = w . mu as hi/lo), nw, |b| ----
  for (int c = tid; c < D; c += kThreads) wv[c] = (KEY && p.w) ? p.w[(int64_t)h * D + c] : 1.0f;
  for (int e = tid; e < D * 16; e += kThreads) {
    const int c = e / 16, k = e % 16;
    Us[e] = (k < R) ? bf16_to_f32(p.u_r[((int64_t)h * D + c) * R + k]) : 0.f;
  }
  __syncthreads();
  for (int e = tid; e < C * (D / 8); e += kThreads) {
    const int j = e / (D / 8), ci = e % (D / 8);
    float mu[8];
    bf16x8(*(const uint4 *)(cent + (int64_t)j * D + 8 * ci), mu);
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const float b0 = KEY ? __fmul_rn(wv[8 * ci + 2 * u], mu[2 * u]) : mu[2 * u];
      const float b1 = KEY ? __fmul_rn(wv[8 * ci + 2 * u + 1], mu[2 * u + 1]) : mu[2 * u + 1];
      const float h0 = __bfloat162float(__float2bfloat16_rn(b0)), h1 = __bfloat162float(__float2bfloat16_rn(b1));
      hw[u] = (uint32_t)f32_to_bf16_rn(h0) | ((uint32_t)f32_to_bf16_rn(h1) << 16);
      lw[u] = (uint32_t)f32_to_bf16_rn(b0 - h0) | ((uint32_t)f32_to_bf16_rn(b1 - h1) << 16);
    }
    const uint32_t off = (ci / 8) * C * 128 + tc::sw128_offset(j, 8 * (ci % 8));
    *(uint4 *)(sm + L.bh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    if (KEY) *(uint4 *)(sm + L.bl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  for (int j = tid; j < C; j += kThreads) {
    float s = 0.f, bb = 0.f;
    for (int ci = 0; ci < D / 8; ci++) {
      float mu[8];
      bf16x8(*(const uint4 *)(cent + (int64_t)j * D + 8 * ci), mu);
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const float wm = __fmul_rn(wv[8 * ci + u], mu[u]);
        s = fmaf(wm, mu[u], s);
        bb = fmaf(wm, wm, bb);
      }
    }
    nw[j] = s;
    bn[j] = sqrtf(bb);
  }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, b = 0.f, bm = 0.f, nm = 0.f;
    for (int c = 0; c < 64; c++) a += wv[c];
    for (int c = 64; c < 128; c++) b += wv[c];
    for (int j = 0; j < C; j++) { bm = fmaxf(bm, bn[j]); nm = fmaxf(nm, fabsf(nw[j])); }
    Wg[0] = a; Wg[1] = b; bmax_sh = bm; nwmax_sh = nm;
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      for (int g = 0; g < nt && !*abort_v; g++) {
        const int s = g & 1;
        if (g >= 2 && !tc::mbar_wait(&x_empty[s], ((g >> 1) - 1) & 1, kWaitNs)) { *abort_v = 1; break; }
        tc::mbar_arrive_expect_tx(&x_full[s], 2 * TILE * 128);
        const int row = (int)((int64_t)h * p.n + (tile0 + g) * TILE);
        unsigned char *dst = sm + L.x + s * 2 * TILE * 128;
        tc::tma_load_2d(dst, &tmap, 0, row, &x_full[s]);
        tc::tma_load_2d(dst + TILE * 128, &tmap, 64, row, &x_full[s]);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(TILE, C);
      const uint32_t sx = tc::smem_u32(sm + L.x), sbh = tc::smem_u32(sm + L.bh), sbl = tc::smem_u32(sm + L.bl);
      for (int g = 0; g < nt && !*abort_v; g++) {
        const int s = g & 1;
        if (!tc::mbar_wait(&x_full[s], (g >> 1) & 1, kWaitNs) ||
            (g >= 2 && !tc::mbar_wait(&t_empty[s], ((g >> 1) - 1) & 1, kWaitNs))) {
          *abort_v = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + 256u * s;
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
          const uint32_t xo = sx + s * 2 * TILE * 128 + (kk / 4) * TILE * 128 + 32 * (kk % 4);
          tc::mma_ss(d, tc::desc_sw128(xo), tc::desc_sw128(sbh + (kk / 4) * C * 128 + 32 * (kk % 4)), idesc, kk > 0);
        }
        if (KEY) {
#pragma unroll
          for (int kk = 0; kk < D / 16; kk++) {
            const uint32_t xo = sx + s * 2 * TILE * 128 + (kk / 4) * TILE * 128 + 32 * (kk % 4);
            tc::mma_ss(d, tc::desc_sw128(xo), tc::desc_sw128(sbl + (kk / 4) * C * 128 + 32 * (kk % 4)), idesc, 1);
          }
        }
        tc::mma_commit(&t_full[s]);
      }
      tc::mma_commit(&drain);
      if (!tc::mbar_wait(&drain, 0, kWaitNs)) *abort_v = 1;
    }
  } else {
    // ======================= epilogue: thread = token =======================
    const int e = (warp - 2) >> 2, sub = warp & 3, row = 32 * sub + lane;
    const uint32_t lane_addr = (uint32_t)(32 * sub) << 16;
    const float W0 = Wg[0], W1 = Wg[1];
    const float knorm_coef = kRel * bmax_sh, nw_err = kRelN * nwmax_sh;
    for (int g = e; g < nt; g += 2) {
      const int s = g & 1;
      if (!tc::mbar_wait(&t_full[s], (g >> 1) & 1, kWaitNs) || !tc::mbar_wait(&x_full[s], (g >> 1) & 1, kWaitNs))
        *abort_v = 1;
      if (*abort_v) break;
      tc::fence_after_sync();
      const unsigned char *xt = sm + L.x + s * 2 * TILE * 128;
      // the token's values (bf16, exact in fp32) are read back from the swizzled tile
      auto xchunk = [&](int ci, float (&f)[8]) {
        bf16x8(*(const uint4 *)(xt + (ci / 8) * TILE * 128 + tc::sw128_offset(row, 8 * (ci % 8))), f);
      };
      // ---- approximate scores -> the M+1 smallest ----
      float tv[MAXM], thr = INFINITY;
      int ti[MAXM];
#pragma unroll
      for (int k = 0; k < MAXM; k++) { tv[k] = INFINITY; ti[k] = C; }
      uint32_t r[32];
      for (int c0 = 0; c0 < C; c0 += 32) {
        tc::tmem_ld32(tmem + lane_addr + 256u * s + c0, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 32; k++)
          topk_insert(tv, ti, thr, M, fmaf(-2.f, __uint_as_float(r[k]), nw[c0 + k]), c0 + k);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&t_empty[s]);
      const int64_t tok = (tile0 + g) * TILE + row;
      const bool valid = tok < p.n;
      const int64_t grow = (int64_t)h * p.n + tok;
      // ---- exact fallback when the candidate boundary lies within the error bound ----
      float kn2 = 0.f;
      for (int ci = 0; ci < D / 8; ci++) {
        float f[8];
        xchunk(ci, f);
#pragma unroll
        for (int u = 0; u < 8; u++) kn2 = fmaf(f[u], f[u], kn2);
      }
      const float delta = knorm_coef * sqrtf(kn2) + nw_err;
      float vM = tv[0], vM1 = tv[0];  // the M-th and (M+1)-th smallest (compile-time indexing)
#pragma unroll
      for (int k = 1; k < MAXM; k++) {
        if (k == M - 1) vM = tv[k];
        if (k == M) vM1 = tv[k];
      }
      const bool amb = valid && (M < C) && !(vM1 - vM > 2.f * delta);
      if (amb) {
        thr = INFINITY;
#pragma unroll
        for (int k = 0; k < MAXM; k++) { tv[k] = INFINITY; ti[k] = C; }
        for (int j = 0; j < C; j++) {
          float dq = 0.f;
          for (int ci = 0; ci < D / 8; ci++) {
            float f[8], mu[8];
            xchunk(ci, f);
            bf16x8(*(const uint4 *)(cent + (int64_t)j * D + 8 * ci), mu);
#pragma unroll
            for (int u = 0; u < 8; u++) {
              const float df = __fsub_rn(f[u], mu[u]);
              dq = __fmaf_rn(wv[8 * ci + u], __fmul_rn(df, df), dq);
            }
          }
          topk_insert(tv, ti, thr, M, dq, j);
        }
      }
      // ---- QSAC: exact range score of each candidate (Values: the single nearest) ----
      int best = 0;
      float best_S = INFINITY, bmn0 = 0.f, bmx0 = 0.f, bmn1 = 0.f, bmx1 = 0.f;
#pragma unroll 1
      for (int m = 0; m < MAXM - 1; m++) {
        if (m >= M) break;
        int j = ti[0];
#pragma unroll
        for (int k = 1; k < MAXM; k++)
          if (k == m) j = ti[k];
        if (j >= C) j = 0;
        float mn0 = INFINITY, mx0 = -INFINITY, mn1 = INFINITY, mx1 = -INFINITY;
        for (int ci = 0; ci < D / 8; ci++) {
          float f[8], mu[8];
          xchunk(ci, f);
          bf16x8(*(const uint4 *)(cent + (int64_t)j * D + 8 * ci), mu);
#pragma unroll
          for (int u = 0; u < 8; u++) {
            const float rr = __fsub_rn(f[u], mu[u]);
            if (ci < 8) { mn0 = fminf(mn0, rr); mx0 = fmaxf(mx0, rr); }
            else { mn1 = fminf(mn1, rr); mx1 = fmaxf(mx1, rr); }
          }
        }
        float S = 0.f;
        if (KEY) {
          const float R0 = __fsub_rn(mx0, mn0), R1 = __fsub_rn(mx1, mn1);
          S = __fadd_rn(__fmul_rn(W0, __fmul_rn(R0, R0)), __fmul_rn(W1, __fmul_rn(R1, R1)));
          if (p.dbg_cand && valid) p.dbg_cand[grow * M + m] = j;
        }
        if (m == 0 || S < best_S || (S == best_S && j < best)) {
          best_S = S; best = j; bmn0 = mn0; bmx0 = mx0; bmn1 = mn1; bmx1 = mx1;
        }
      }
      // ---- INT2 codes of the chosen centroid's residual; PSAC coefficients ----
      float m0, s0, i0, m1, s1, i1;
      uint16_t mb0, sb0, mb1, sb1;
      int2_params(bmn0, bmx0, m0, s0, i0, mb0, sb0, p.status);
      int2_params(bmn1, bmx1, m1, s1, i1, mb1, sb1, p.status);
      uint32_t packed[8];
      float Cv[RMAX];
#pragma unroll
      for (int k = 0; k < RMAX; k++) Cv[k] = 0.f;
#pragma unroll
      for (int ci = 0; ci < D / 8; ci++) {
        float f[8], mu[8];
        xchunk(ci, f);
        bf16x8(*(const uint4 *)(cent + (int64_t)best * D + 8 * ci), mu);
        const bool g1 = ci >= 8;
        const float mm = g1 ? m1 : m0, ss = g1 ? s1 : s0, ii = g1 ? i1 : i0;
        uint32_t bits = 0;
#pragma unroll
        for (int u = 0; u < 8; u++) {
          const uint32_t q = int2_code(__fsub_rn(f[u], mu[u]), mm, ss, ii);
          bits |= q << (2 * u);
          if (KEY && R > 0) {
            const float ev = __fsub_rn(f[u], __fadd_rn(mu[u], __fmaf_rn(ss, (float)q, mm)));
            const float *Uc = Us + (8 * ci + u) * 16;
#pragma unroll
            for (int k = 0; k < RMAX; k++) Cv[k] = fmaf(ev, Uc[k], Cv[k]);
          }
        }
        if (ci & 1) packed[ci >> 1] |= bits << 16;
        else packed[ci >> 1] = bits;
      }
      if (valid) {
        uint4 *cdst = (uint4 *)(p.codes + grow * (D / 4));
        cdst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        cdst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        p.idx[grow] = (uint8_t)best;
        *(uint32_t *)(p.scale + grow * 2) = (uint32_t)sb0 | ((uint32_t)sb1 << 16);
        *(uint32_t *)(p.minv + grow * 2) = (uint32_t)mb0 | ((uint32_t)mb1 << 16);
        if (KEY && p.dbg_score) p.dbg_score[grow] = best_S;
        if (KEY && R > 0) {
          float a = 0.f;
#pragma unroll
          for (int k = 0; k < RMAX; k++)
            if (k < R) a = fmaxf(a, fabsf(Cv[k]));
          __half sch = __float2half_ru(__fdiv_ru(a, 127.0f));
          if (a == 0.f) sch = __float2half_rn(0.f);
          const float sc = __half2float(sch);
          if (!isfinite(sc)) qwm_dev_error(p.status, QWM_ERR_RANGE);
          const float inv = sc > 0.f ? __frcp_rn(sc) : 0.f;
#pragma unroll
          for (int k = 0; k < RMAX; k++) {
            if (k < R) {
              float qf = sc > 0.f ? rintf(__fmul_rn(Cv[k], inv)) : 0.f;
              qf = fminf(fmaxf(qf, -127.f), 127.f);
              p.c[grow * R + k] = (int8_t)qf;
              if (p.dbg_c) p.dbg_c[grow * R + k] = Cv[k];
            }
          }
          p.c_scale[grow] = __half_as_ushort(sch);
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&x_empty[s]);
    }
  }
  __syncthreads();
  if (*abort_v && tid == 0) qwm_dev_error(p.status, QWM_ERR_DEVICE_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <bool KEY, int RMAX>
cudaError_t launch_one(const TensorMap128 &tmap, const QParams &p, int H, int smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(quant_kernel<KEY, RMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  quant_kernel<KEY, RMAX><<<dim3(p.G, H), kThreads, smem, st>>>(tmap, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const qwm_config &cfg, const uint16_t *k, const uint16_t *v, int64_t n, const float *w,
                            const uint16_t *u_r, const qwm_chunk &out, const qwm_debug *dbg, int32_t *status,
                            int num_sms, cudaStream_t st) {
  const int H = cfg.heads, C = cfg.n_centroids;
  const int64_t tiles = (n + TILE - 1) / TILE;
  int G = (num_sms + H - 1) / H;
  if (G > tiles) G = (int)tiles;
  if (G < 1) G = 1;
  for (int pass = 0; pass < 2; pass++) {
    const bool key = pass == 0;
    TensorMap128 tmap;
    if (!make_tmap_rows128_bf16(&tmap, key ? k : v, (uint64_t)H * n, TILE)) return cudaErrorInvalidValue;
    QParams p;
    p.n = n; p.w = key ? w : nullptr; p.u_r = key ? u_r : nullptr;
    p.cent = key ? out.cent_k : out.cent_v;
    p.C = C; p.top_m = cfg.top_m; p.rank = (key && u_r) ? cfg.rank : 0; p.G = G;
    p.codes = key ? out.k_codes : out.v_codes; p.idx = key ? out.k_idx : out.v_idx;
    p.scale = key ? out.k_scale : out.v_scale; p.minv = key ? out.k_min : out.v_min;
    p.c = out.c; p.c_scale = out.c_scale;
    p.dbg_c = (key && dbg) ? dbg->c_f32 : nullptr;
    p.dbg_cand = (key && dbg) ? dbg->cand : nullptr;
    p.dbg_score = (key && dbg) ? dbg->score : nullptr;
    p.status = status;
    const int smem = QSmem(C, key).total + 1024;
    cudaError_t e;
    if (!key) e = launch_one<false, 8>(tmap, p, H, smem, st);
    else if (p.rank <= 8) e = launch_one<true, 8>(tmap, p, H, smem, st);
    else e = launch_one<true, 16>(tmap, p, H, smem, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
