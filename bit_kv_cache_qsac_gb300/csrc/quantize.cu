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
// term is the same for every j, so the ranking uses T_j = k.b_j - nw_j / 2 (the largest T is the
// nearest centroid) with b_j = w . mu_j and nw_j = sum_c w_c mu_jc^2.  The tensor cores produce T
// directly in TMEM: two bf16 MMAs against b = hi + lo (each bf16; Values use b = mu, exact, one
// MMA) and a third, K = 16 MMA of a constant [1 1 0 ...] row block against [-nw/2 hi, lo, 0 ...].
// The approximate T pick the candidates: with |T_approx - T| <= delta, every centroid outside
// the window T_approx >= T_M - 2 delta (T_M = the M-th largest) is outside the exact top-M.  When
// the window holds exactly M centroids (almost always) it is the exact candidate set; otherwise
// the warp computes exact fp32 distances for the window and keeps the M nearest (lower index on
// ties).  The range score S, the INT2 codes and the PSAC coefficients are exact fp32 with
// explicitly rounded intrinsics, so indices and codes match a plain IEEE implementation bit for
// bit.
//
// One CTA = one head x a contiguous range of 128-token tiles; 320 threads:
//   warp 0     TMA producer: K (or V) tiles as two [128][64] bf16 blocks, 128-byte swizzle, 2 stages
//   warp 1     TMEM owner and MMA issuer: tile g into TMEM buffer g % 2
//   warps 2-9  two epilogue warpgroups; group e owns the tiles g with g % 2 == e.  Per tile:
//     (1) thread = token: the M+1 largest T from TMEM (branch-free insertion network), then the
//         window as a bit mask per token in shared memory; TMEM is released;
//     (2) warp-cooperative (lane = 4 channels), for the rare tokens whose window holds more than
//         M centroids: exact distances to the window's centroids, the M nearest kept;
//     (3) Keys, warp-cooperative: S of every (token, candidate) pair, with the centroid row read
//         coalesced from global memory and the group ranges reduced across half-warps;
//     (4) thread = token: INT2 codes of the chosen centroid's residual, PSAC coefficients.
// Codebooks of 1024 centroids (WIDE) do not fit in shared memory: a small kernel writes each head's
// distance operands as an image of 128-centroid slices in global memory, and the producer streams
// the slices (bulk copies) through one shared-memory slice buffer, each tile's MMAs running slice by
// slice into two 128-column TMEM halves per epilogue group.  Phase (1) then keeps the M+3 largest T
// with their indices while the slices go by; when the window reaches past that list, the token's
// window becomes the whole codebook and phase (2) finds its exact M nearest.  Indices are uint16.
// All waits are bounded; on expiry the kernel records QWM_ERR_DEVICE_TIMEOUT and stops.
#include <cuda_fp16.h>

#include "qwm_internal.cuh"
#include "tc.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int TILE = 128;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr uint64_t kWaitNs = 1000000000ull;
// error bound of an approximate T: |err| <= kRel |k| max_j |b_j| + kRelN max_j |nw_j|
constexpr float kRel = 1.0f / 32768.0f;    // 2^-15
constexpr float kRelN = 1.0f / 131072.0f;  // 2^-17
constexpr int kSlice = 128;                // centroids per streamed slice (WIDE)
constexpr float kRint = 8388608.0f;        // 2^23: x + 2^23 - 2^23 = rint(x) for 0 <= x < 2^22

struct QSmem {
  int bh, bl, bn, an, x, msk, wv, U, ef, total;
  // CB = centroids held in shared memory at once: the whole codebook, or one slice (WIDE).  The
  // range [0, an) is also the layout of one slice of the global operand image.
  __host__ __device__ QSmem(int C, bool key, bool wide) {
    const int CB = wide ? kSlice : C;
    bh = 0;                               // 2 blocks of [CB][64] bf16: hi of b (or mu for Values)
    bl = bh + 2 * CB * 128;               // lo of b (Keys only)
    bn = bl + (key ? 2 * CB * 128 : 0);   // [CB][16] bf16 no-swizzle: -nw/2 as hi, lo, then zeros
    an = bn + CB * 32;                    // [128][16] bf16 no-swizzle: 1, 1, then zeros
    x = an + TILE * 32;                 // 2 stages x 2 blocks of [128][64]
    msk = x + 2 * 2 * TILE * 128;       // window masks: [8 warps][C/32 words][32 tokens]
    wv = msk + kEpiWarps * (C / 32) * 32 * 4;  // w[D]
    U = wv + 4 * D;                     // U_r as fp32 [D][16], zero past the rank (Keys)
    ef = U + (key ? 4 * D * 16 : 0);    // Keys: per epilogue warp, one residual row (full-form fallback)
    total = ef + (key ? kEpiWarps * D * 4 : 0);
  }
};

struct QParams {
  int64_t n;
  const float *w;           // [H][D] or NULL
  const uint16_t *u_r;      // [H][D][R] or NULL
  const uint16_t *cent;     // [H][C][D] bf16 codebook
  int C, top_m, rank, G;
  const unsigned char *img;  // WIDE: [H][C / kSlice] operand slices
  const float *img_max;      // WIDE: [H][2] max_j |b_j|, max_j |nw_j|
  uint8_t *codes;
  void *idx;                 // uint8 [H][n], or uint16 [H][n] (WIDE)
  uint16_t *scale, *minv;    // fp16 storage: [H][n][2]
  int compact, gate;         // compact metadata; PSAC keep-if-better
  uint8_t *s8, *zp;          // compact: [H][n][2] steps, [H][n] zero-points (group g in bits 2g..2g+1)
  uint16_t *sigma;           // compact: fp16 [H][ceil(n/128)][2] second-level scales
  const float *wk;           // [H][D] channel weights of the gate (NULL: uniform)
  const float *Mq;           // full-form ranking: [H][D][D] Query second moment (NULL: diagonal w)
  const float *Bq;           // full-form ranking: [H][C][D] b_j = M mu_j (the distance GEMM's operand)
  float *dbg_gate;           // [H][n][2] w-weighted error without / with C, or NULL
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

// Eight bf16 values (channels 2u, 2u + 1 in word u) as four fp32 pairs {channel 2u, channel 2u + 1}
// for the packed f32x2 instructions.
__device__ __forceinline__ void bf16x8_pairs(const uint4 v, uint64_t (&f)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int u = 0; u < 4; u++) f[u] = ((uint64_t)(w[u] & 0xFFFF0000u) << 32) | (uint64_t)(w[u] << 16);
}
__device__ __forceinline__ uint64_t u2(uint32_t lo, uint32_t hi) { return ((uint64_t)hi << 32) | (uint64_t)lo; }

// byte offset of (row, column k) in a [rows][16] bf16 K-major operand without swizzle
__host__ __device__ constexpr uint32_t noswz16(uint32_t row, uint32_t k) {
  return (row >> 3) * 256u + (k >> 3) * 128u + (row & 7u) * 16u + (k & 7u) * 2u;
}

// The lane's share (channels 4 lane .. 4 lane + 3) of e^T M e for a residual row e in shared memory
// (the rare exact pass of the full-form ranking; kept out of line so that it does not weigh on the
// register allocation of the common path).
__device__ __forceinline__ float quad_form_lane(const float *__restrict__ Mh, const float *er, int lane) {
  float dq = 0.f;
#pragma unroll 1
  for (int u = 0; u < 4; u++) {
    const int c = 4 * lane + u;
    const float *row = Mh + (int64_t)c * D;
    float t = 0.f;
#pragma unroll 1
    for (int c2 = 0; c2 < D; c2++) t = __fmaf_rn(row[c2], er[c2], t);
    dq = __fmaf_rn(er[c], t, dq);
  }
  return dq;
}

// Compact metadata (the paper's packed form): the smallest step whose grid [-z s, (3 - z) s] covers
// [a, b] over the four integer zero-points (lower z on ties), rounded up.
__device__ __forceinline__ void zp_range(float a, float b, float &need, int &z) {
  need = 0.f;
  z = 0;
  if (a == 0.f && b == 0.f) return;
  float best = INFINITY;
#pragma unroll
  for (int zz = 0; zz < 4; zz++) {
    const float lo = (a >= 0.f) ? 0.f : (zz > 0 ? __fdiv_ru(-a, (float)zz) : INFINITY);
    const float hi = (b <= 0.f) ? 0.f : (zz < 3 ? __fdiv_ru(b, (float)(3 - zz)) : INFINITY);
    const float sz = fmaxf(lo, hi);
    if (sz < best) { best = sz; z = zz; }
  }
  need = best;
}
// The second-level scale: the smallest power of two sigma with 255 sigma >= smax (>= 2^-24).
__device__ __forceinline__ float pow2_sigma(float smax) {
  if (smax == 0.f) return 0.f;
  const uint32_t t = __float_as_uint(__fdiv_ru(smax, 255.0f));
  const uint32_t e = t >> 23, m = t & 0x7FFFFFu;
  float sg = (m == 0u && e != 0u) ? __uint_as_float(t) : __uint_as_float((e + 1u) << 23);
  if (e == 0u) sg = __uint_as_float(1u << 23);  // t subnormal: the smallest normal power of two
  return fmaxf(sg, 5.9604644775390625e-08f);
}

// Byte offset, inside a [128][64] x 2 swizzled tile, of this lane's 4 channels (4 lane .. 4 lane + 3)
// of token row t.
__device__ __forceinline__ uint32_t lane4_offset(int t, int lane) {
  return (uint32_t)(lane >> 4) * TILE * 128u + (uint32_t)t * 128u +
         ((((uint32_t)(lane & 15) >> 1) ^ ((uint32_t)t & 7u)) << 4) + 8u * (uint32_t)(lane & 1);
}
__device__ __forceinline__ void unpack4(uint2 v, float (&f)[4]) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// KEY: Keys (QSAC + PSAC) or Values (nearest centroid).  RMAX: 8 or 16, bound on the PSAC rank.
// MP1: length of the largest-T list, at least top_m + 1 (5 serves top_m 1..4; QWM_MAX_TOPM + 1
// covers every M, with the list's tail unused).  WIDE: the codebook streams through in slices.
template <bool KEY, int RMAX, int MP1, bool WIDE>
__global__ void __launch_bounds__(kThreads, 1) quant_kernel(const __grid_constant__ TensorMap128 tmap,
                                                             const QParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char *sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t x_full[2], x_empty[2], t_full[2], t_empty[2], drain;
  __shared__ uint64_t tw_full[4], tw_empty[4], sl_full, sl_empty;  // WIDE: TMEM halves, slice buffer
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ float Wg[2], bmax_sh, nwmax_sh;
  __shared__ float red_sg[2][2][4][2];  // compact: [group][tile parity][warp][channel group] step maxima
  __shared__ uint64_t sg_bar[2];        // compact: the 4 warps of epilogue group e per tile
  const int C = p.C, M = KEY ? p.top_m : 1, R = KEY ? p.rank : 0;
  const int NW = C / 32;  // mask words per token
  const int NSL = WIDE ? C / kSlice : 1;
  const QSmem L(C, KEY, WIDE);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, cta = blockIdx.x;
  const int64_t tiles = (p.n + TILE - 1) / TILE;
  const int64_t per = (tiles + p.G - 1) / p.G;
  const int64_t tile0 = (int64_t)cta * per;
  const int64_t tile1 = tile0 + per < tiles ? tile0 + per : tiles;
  const int nt = tile1 > tile0 ? (int)(tile1 - tile0) : 0;
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
    for (int i = 0; i < 4; i++) {
      tc::mbar_init(&tw_full[i], 1);
      tc::mbar_init(&tw_empty[i], 4);
    }
    tc::mbar_init(&sl_full, 1);
    tc::mbar_init(&sl_empty, 1);
    tc::mbar_init(&sg_bar[0], 4);
    tc::mbar_init(&sg_bar[1], 4);
    tc::mbar_init(&drain, 1);
    abort_flag = 0;
    bmax_sh = WIDE ? p.img_max[2 * h] : 0.f;
    nwmax_sh = WIDE ? p.img_max[2 * h + 1] : 0.f;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&tmem_base_sh, 512);
    tc::tmem_relinquish();
  }
  // ---- per-head constants: weights, basis, distance operands ----
  for (int c = tid; c < D; c += kThreads)
    wv[c] = (KEY && p.Mq) ? p.Mq[((int64_t)h * D + c) * D + c] : ((KEY && p.w) ? p.w[(int64_t)h * D + c] : 1.0f);
  if (KEY) {
    for (int e = tid; e < D * 16; e += kThreads) {
      const int c = e / 16, k = e % 16;
      Us[e] = (k < R) ? bf16_to_f32(p.u_r[((int64_t)h * D + c) * R + k]) : 0.f;
    }
  }
  for (int e = tid; e < TILE * 8; e += kThreads) {  // constant A block of the nw MMA
    const int row = e >> 3, kw = e & 7;           // 8 words of 2 bf16 per row
    *(uint32_t *)(sm + L.an + noswz16(row, 2 * kw)) = kw == 0 ? 0x3F803F80u : 0u;
  }
  __syncthreads();
  // b = w . mu split into bf16 hi + lo (Keys) or mu itself (Values), 128-byte swizzled K-major
  // (WIDE: the operand image already holds them)
  for (int e = tid; e < (WIDE ? 0 : C) * (D / 8); e += kThreads) {
    const int j = e / (D / 8), ci = e % (D / 8);
    float mu[8];
    bf16x8(*(const uint4 *)(cent + (int64_t)j * D + 8 * ci), mu);
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const float *bq = (KEY && p.Bq) ? p.Bq + ((int64_t)h * C + j) * D + 8 * ci : nullptr;
      const float b0 = bq ? bq[2 * u] : (KEY ? __fmul_rn(wv[8 * ci + 2 * u], mu[2 * u]) : mu[2 * u]);
      const float b1 = bq ? bq[2 * u + 1] : (KEY ? __fmul_rn(wv[8 * ci + 2 * u + 1], mu[2 * u + 1]) : mu[2 * u + 1]);
      const float h0 = __bfloat162float(__float2bfloat16_rn(b0)), h1 = __bfloat162float(__float2bfloat16_rn(b1));
      hw[u] = (uint32_t)f32_to_bf16_rn(h0) | ((uint32_t)f32_to_bf16_rn(h1) << 16);
      lw[u] = (uint32_t)f32_to_bf16_rn(b0 - h0) | ((uint32_t)f32_to_bf16_rn(b1 - h1) << 16);
    }
    const uint32_t off = (ci / 8) * C * 128 + tc::sw128_offset(j, 8 * (ci % 8));
    *(uint4 *)(sm + L.bh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    if (KEY) *(uint4 *)(sm + L.bl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  // nw_j and |b_j| (one warp per centroid, lane = 4 channels), the nw operand, the maxima
  for (int j = warp; j < (WIDE ? 0 : C); j += kThreads / 32) {
    float mu[4];
    unpack4(*(const uint2 *)(cent + (int64_t)j * D + 4 * lane), mu);
    float s = 0.f, bb = 0.f;
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const float wm = (KEY && p.Bq) ? p.Bq[((int64_t)h * C + j) * D + 4 * lane + u] : __fmul_rn(wv[4 * lane + u], mu[u]);
      s = fmaf(wm, mu[u], s);
      bb = fmaf(wm, wm, bb);
    }
    s = warp_sum(s);
    bb = warp_sum(bb);
    if (lane < 8) {  // row j of the nw operand: [-nw/2 hi, lo, 0 ...]
      uint32_t wd = 0u;
      if (lane == 0) {
        const float t = -0.5f * s, th = __bfloat162float(__float2bfloat16_rn(t));
        wd = (uint32_t)f32_to_bf16_rn(th) | ((uint32_t)f32_to_bf16_rn(t - th) << 16);
      }
      *(uint32_t *)(sm + L.bn + noswz16(j, 2 * lane)) = wd;
    }
    if (lane == 0) {
      atomicMax((int *)&bmax_sh, __float_as_int(sqrtf(bb)));  // non-negative floats order as ints
      atomicMax((int *)&nwmax_sh, __float_as_int(fabsf(s)));
    }
  }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, b = 0.f;
    for (int c = 0; c < 64; c++) a += wv[c];
    for (int c = 64; c < 128; c++) b += wv[c];
    Wg[0] = a;
    Wg[1] = b;
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
        if (WIDE) {  // this tile's pass over the codebook, one slice at a time
          const uint32_t ib = (uint32_t)L.an;
          const unsigned char *img = p.img + (int64_t)h * NSL * ib;
          for (int sl = 0; sl < NSL; sl++) {
            const int u = g * NSL + sl;
            if (u >= 1 && !tc::mbar_wait(&sl_empty, (u - 1) & 1, kWaitNs)) { *abort_v = 1; break; }
            tc::mbar_arrive_expect_tx(&sl_full, ib);
            tc::bulk_load(tc::smem_u32(sm), img + (int64_t)sl * ib, ib, &sl_full);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const int CB = WIDE ? kSlice : C;  // centroids per MMA
      const uint32_t idesc = tc::idesc_bf16_f32(TILE, CB);
      const uint32_t sx = tc::smem_u32(sm + L.x), sbh = tc::smem_u32(sm + L.bh), sbl = tc::smem_u32(sm + L.bl);
      const uint32_t sbn = tc::smem_u32(sm + L.bn), san = tc::smem_u32(sm + L.an);
      auto issue = [&](uint32_t d, int s) {  // T of one tile against the centroids in shared memory
        tc::mma_ss(d, tc::desc_noswz(san, 128, 256), tc::desc_noswz(sbn, 128, 256), idesc, 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
          const uint32_t xo = sx + s * 2 * TILE * 128 + (kk / 4) * TILE * 128 + 32 * (kk % 4);
          tc::mma_ss(d, tc::desc_sw128(xo), tc::desc_sw128(sbh + (kk / 4) * CB * 128 + 32 * (kk % 4)), idesc, 1);
        }
        if (KEY) {
#pragma unroll
          for (int kk = 0; kk < D / 16; kk++) {
            const uint32_t xo = sx + s * 2 * TILE * 128 + (kk / 4) * TILE * 128 + 32 * (kk % 4);
            tc::mma_ss(d, tc::desc_sw128(xo), tc::desc_sw128(sbl + (kk / 4) * CB * 128 + 32 * (kk % 4)), idesc, 1);
          }
        }
      };
      for (int g = 0; g < nt && !*abort_v; g++) {
        const int s = g & 1;
        if (WIDE) {
          if (!tc::mbar_wait(&x_full[s], (g >> 1) & 1, kWaitNs)) { *abort_v = 1; break; }
          for (int sl = 0; sl < NSL; sl++) {
            // slice sl of tile g -> TMEM half (sl & 1) of group s; that half's k-th use
            const int u = g * NSL + sl, hb = 2 * s + (sl & 1), k = (g >> 1) * (NSL / 2) + (sl >> 1);
            if (!tc::mbar_wait(&sl_full, u & 1, kWaitNs) ||
                (k >= 1 && !tc::mbar_wait(&tw_empty[hb], (k - 1) & 1, kWaitNs))) {
              *abort_v = 1;
              break;
            }
            tc::fence_after_sync();
            issue(tmem + 256u * s + 128u * (sl & 1), s);
            tc::mma_commit(&tw_full[hb]);
            tc::mma_commit(&sl_empty);
          }
          continue;
        }
        if (!tc::mbar_wait(&x_full[s], (g >> 1) & 1, kWaitNs) ||
            (g >= 2 && !tc::mbar_wait(&t_empty[s], ((g >> 1) - 1) & 1, kWaitNs))) {
          *abort_v = 1;
          break;
        }
        tc::fence_after_sync();
        issue(tmem + 256u * s, s);
        tc::mma_commit(&t_full[s]);
      }
      tc::mma_commit(&drain);
      if (!tc::mbar_wait(&drain, 0, kWaitNs)) *abort_v = 1;
    }
  } else {
    // ======================= epilogue =======================
    const int ew = warp - 2, e = ew >> 2, sub = warp & 3, row = 32 * sub + lane;
    const uint32_t lane_addr = (uint32_t)(32 * sub) << 16;
    const float W0 = Wg[0], W1 = Wg[1];
    const float dcoef = kRel * bmax_sh, dconst = kRelN * nwmax_sh;
    uint32_t *msk = (uint32_t *)(sm + L.msk) + ew * NW * 32;  // [word][token] for this warp
    float wl[4];  // this lane's 4 channel weights (cooperative phases)
#pragma unroll
    for (int u = 0; u < 4; u++) wl[u] = wv[4 * lane + u];
    for (int g = e; g < nt; g += 2) {
      const int s = g & 1;
      if ((!WIDE && !tc::mbar_wait(&t_full[s], (g >> 1) & 1, kWaitNs)) ||
          !tc::mbar_wait(&x_full[s], (g >> 1) & 1, kWaitNs))
        *abort_v = 1;
      if (*abort_v) break;
      tc::fence_after_sync();
      const unsigned char *xt = sm + L.x + s * 2 * TILE * 128;
      const uint32_t xts = tc::smem_u32(xt);
      const int64_t tok0 = (tile0 + g) * TILE + 32 * sub;  // token of lane 0 of this warp
      const int64_t tok = tok0 + lane;
      const bool valid = tok < p.n;
      // ---- (1) the M+1 largest T, then the window mask (thread = token) ----
      uint64_t kn2p = 0ull;  // ||k||^2 as two interleaved partial sums (it only sizes the window)
#pragma unroll
      for (int ci = 0; ci < D / 8; ci++) {
        uint64_t f2[4];
        bf16x8_pairs(tc::lds128(xts + (ci / 8) * TILE * 128 + tc::sw128_offset(row, 8 * (ci % 8))), f2);
#pragma unroll
        for (int u = 0; u < 4; u++) kn2p = tc::fma2(f2[u], f2[u], kn2p);
      }
      const float kn2 = tc::f2lo(kn2p) + tc::f2hi(kn2p);
      const float delta2 = 2.f * (dcoef * sqrtf(kn2) + dconst);
      uint32_t r[32];
      bool amb;
      if constexpr (WIDE) {
        // the KL largest T with their indices (descending; equal T keep the lower index first),
        // fed slice by slice from the two TMEM halves of this group
        constexpr int KL = MP1 + 2;
        float tv[KL];
        int ti[KL];
#pragma unroll
        for (int k = 0; k < KL; k++) { tv[k] = -INFINITY; ti[k] = C; }
        bool bad = false;
#pragma unroll 1
        for (int sl = 0; sl < NSL; sl++) {
          const int hb = 2 * s + (sl & 1), k = (g >> 1) * (NSL / 2) + (sl >> 1);
          const bool ok = tc::mbar_wait(&tw_full[hb], k & 1, kWaitNs);
          if (__any_sync(0xffffffffu, !ok || *abort_v != 0)) { bad = true; break; }  // warp-uniform
          tc::fence_after_sync();
#pragma unroll 1
          for (int c0 = 0; c0 < kSlice; c0 += 32) {
            tc::tmem_ld16(tmem + lane_addr + 256u * s + 128u * (sl & 1) + c0, r);
            tc::tmem_ld16(tmem + lane_addr + 256u * s + 128u * (sl & 1) + c0 + 16, r + 16);
            tc::tmem_ld_wait();
#pragma unroll
            for (int kk = 0; kk < 32; kk++) {
              const float v = __uint_as_float(r[kk]);
              if (v > tv[KL - 1]) {
                const int j = sl * kSlice + c0 + kk;
#pragma unroll
                for (int i = KL - 1; i >= 1; i--) {
                  const bool up = v > tv[i - 1], in = v > tv[i];
                  tv[i] = up ? tv[i - 1] : (in ? v : tv[i]);
                  ti[i] = up ? ti[i - 1] : (in ? j : ti[i]);
                }
                if (v > tv[0]) { tv[0] = v; ti[0] = j; }
              }
            }
          }
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&tw_empty[hb]);
        }
        if (bad) { *abort_v = 1; break; }
        float tM = tv[0], tM1 = tv[0];
#pragma unroll
        for (int k = 1; k < KL; k++) {
          if (k == M - 1) tM = tv[k];
          if (k == M) tM1 = tv[k];
        }
        const float thr = tM - delta2;
        amb = valid && (M < C) && !(tM1 < thr);
        // a window that may reach past the list: every centroid goes to the exact pass
        const bool over = amb && !(tv[KL - 1] < thr);
        for (int wi = 0; wi < NW; wi++) msk[wi * 32 + lane] = (valid && over) ? 0xFFFFFFFFu : 0u;
        if (valid && !over) {
#pragma unroll
          for (int k = 0; k < KL; k++)
            if (tv[k] >= thr && ti[k] < C) msk[(ti[k] >> 5) * 32 + lane] |= 1u << (ti[k] & 31);
        }
        __syncwarp();
      } else {
        float tv[MP1];
#pragma unroll
        for (int k = 0; k < MP1; k++) tv[k] = -INFINITY;
#pragma unroll 1
        for (int c0 = 0; c0 < C; c0 += 32) {
          tc::tmem_ld16(tmem + lane_addr + 256u * s + c0, r);
          tc::tmem_ld16(tmem + lane_addr + 256u * s + c0 + 16, r + 16);
          tc::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            // two values at a time: the sorted pair a >= b merged into the descending list,
            // new tv[i] = max(tv[i], min(tv[i-1], a), min(tv[i-2], b)), updated from the bottom up
            const float v0 = __uint_as_float(r[k]), v1 = __uint_as_float(r[k + 1]);
            const float a = fmaxf(v0, v1), b = fminf(v0, v1);
#pragma unroll
            for (int i = MP1 - 1; i >= 2; i--) tv[i] = tc::max3(tv[i], fminf(tv[i - 1], a), fminf(tv[i - 2], b));
            tv[1] = tc::max3(tv[1], fminf(tv[0], a), b);
            tv[0] = fmaxf(tv[0], a);
          }
        }
        float tM = tv[0], tM1 = tv[0];  // the M-th and (M+1)-th largest (compile-time indexing)
#pragma unroll
        for (int k = 1; k < MP1; k++) {
          if (k == M - 1) tM = tv[k];
          if (k == M) tM1 = tv[k];
        }
        const float thr = tM - delta2;
        amb = valid && (M < C) && !(tM1 < thr);
#pragma unroll 1
        for (int c0 = 0; c0 < C; c0 += 32) {
          tc::tmem_ld16(tmem + lane_addr + 256u * s + c0, r);
          tc::tmem_ld16(tmem + lane_addr + 256u * s + c0 + 16, r + 16);
          tc::tmem_ld_wait();
          uint32_t word = 0u;
#pragma unroll
          for (int k = 0; k < 32; k++) word |= (__uint_as_float(r[k]) >= thr ? 1u : 0u) << k;
          msk[(c0 >> 5) * 32 + lane] = valid ? word : 0u;
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&t_empty[s]);
      }
      // ---- (2) exact candidate set for tokens whose window holds more than M centroids ----
      uint32_t ambs = __ballot_sync(0xffffffffu, amb);
      while (ambs) {
        const int t = __ffs(ambs) - 1;
        ambs &= ambs - 1;
        float xf[4];
        unpack4(*(const uint2 *)(xt + lane4_offset(32 * sub + t, lane)), xf);
        float ev[17];
        int ei[17];
#pragma unroll
        for (int k = 0; k < 17; k++) { ev[k] = INFINITY; ei[k] = C; }
        for (int wi = 0; wi < NW; wi++) {
          uint32_t m = msk[wi * 32 + t];
          while (m) {
            const int j = 32 * wi + __ffs(m) - 1;
            m &= m - 1;
            float mu[4];
            unpack4(*(const uint2 *)(cent + (int64_t)j * D + 4 * lane), mu);
            float dq = 0.f;
            if (KEY && p.Mq) {  // (x - mu)^T M (x - mu): the residual row through shared memory
              float *er = (float *)(sm + L.ef) + ew * D;
#pragma unroll
              for (int u = 0; u < 4; u++) er[4 * lane + u] = __fsub_rn(xf[u], mu[u]);
              __syncwarp();
              dq = quad_form_lane(p.Mq + (int64_t)h * D * D, er, lane);
              __syncwarp();
            } else {
#pragma unroll
              for (int u = 0; u < 4; u++) {
                const float df = __fsub_rn(xf[u], mu[u]);
                dq = __fmaf_rn(wl[u], __fmul_rn(df, df), dq);
              }
            }
            dq = warp_sum(dq);  // identical on every lane
            // insert (dq, j) into the ascending exact list (j increasing: a strict comparison
            // keeps the lower index first on ties)
            if (dq < ev[16]) {
              float cv = dq;
              int cj = j;
#pragma unroll
              for (int k = 0; k < 17; k++) {
                const bool sw = cv < ev[k];
                const float tvv = ev[k];
                const int tj = ei[k];
                ev[k] = sw ? cv : ev[k];
                ei[k] = sw ? cj : ei[k];
                cv = sw ? tvv : cv;
                cj = sw ? tj : cj;
              }
            }
          }
        }
        __syncwarp();
        // the token's candidate mask := the M nearest
        if (lane < NW) {
          uint32_t word = 0u;
#pragma unroll
          for (int k = 0; k < 17; k++)
            if (k < M && (ei[k] >> 5) == lane) word |= 1u << (ei[k] & 31);
          msk[lane * 32 + t] = word;
        }
        __syncwarp();
      }
      // ---- (3) Keys: range score S of every candidate (thread = token), best per token ----
      int best = 0;
      float best_S = 0.f;
      float bmn0 = INFINITY, bmx0 = -INFINITY, bmn1 = INFINITY, bmx1 = -INFINITY;  // the best one's ranges
      bool have_range = false;
      if (KEY) {
        // The token's candidates from its window mask (newest first), then one pass over its 16
        // eight-channel chunks: the chunk of x from shared memory once, the same chunk of every
        // candidate row from global memory (independent loads: their latencies overlap), and the
        // per-group min / max of each candidate's residual.  Ties in S go to the lower index.
        constexpr int KM = MP1 - 1;
        int cj[KM];
        int cnt = 0;
#pragma unroll
        for (int k = 0; k < KM; k++) cj[k] = 0;
        for (int wi = 0; wi < NW; wi++) {
          uint32_t m = msk[wi * 32 + lane];
          while (m) {
            const int j = 32 * wi + __ffs(m) - 1;
            m &= m - 1;
#pragma unroll
            for (int k = KM - 1; k >= 1; k--) cj[k] = cj[k - 1];
            cj[0] = j;
            cnt++;
          }
        }
        cnt = valid ? (cnt < KM ? cnt : KM) : 0;
        float mnv[KM][2], mxv[KM][2];
#pragma unroll
        for (int k = 0; k < KM; k++) {
          mnv[k][0] = mnv[k][1] = INFINITY;
          mxv[k][0] = mxv[k][1] = -INFINITY;
        }
        if (cnt > 0) {
#pragma unroll
          for (int gi = 0; gi < 2; gi++) {  // the two groups of 64 channels
#pragma unroll
          for (int cc = 0; cc < 8; cc++) {
            const int ci = 8 * gi + cc;
            uint64_t f2[4];
            bf16x8_pairs(tc::lds128(xts + gi * TILE * 128 + tc::sw128_offset(row, 8 * cc)), f2);
#pragma unroll
            for (int k = 0; k < KM; k++) {
              if (k < cnt) {
                uint64_t m2[4];
                bf16x8_pairs(*(const uint4 *)(cent + (int64_t)cj[k] * D + 8 * ci), m2);
#pragma unroll
                for (int u = 0; u < 4; u++) {  // two channels per packed subtraction
                  const uint64_t rr = tc::sub2(f2[u], m2[u]);
                  mnv[k][gi] = tc::min3(mnv[k][gi], tc::f2lo(rr), tc::f2hi(rr));
                  mxv[k][gi] = tc::max3(mxv[k][gi], tc::f2lo(rr), tc::f2hi(rr));
                }
              }
            }
          }
          }
        }
        float bS = INFINITY;
        int bj = C;
#pragma unroll
        for (int k = 0; k < KM; k++) {
          if (k < cnt) {
            const float R0 = __fsub_rn(mxv[k][0], mnv[k][0]), R1 = __fsub_rn(mxv[k][1], mnv[k][1]);
            const float S = __fadd_rn(__fmul_rn(W0, __fmul_rn(R0, R0)), __fmul_rn(W1, __fmul_rn(R1, R1)));
            if (S < bS || (S == bS && cj[k] < bj)) {
              bS = S; bj = cj[k];
              bmn0 = mnv[k][0]; bmx0 = mxv[k][0]; bmn1 = mnv[k][1]; bmx1 = mxv[k][1];
            }
            if (p.dbg_cand && k < M) p.dbg_cand[((int64_t)h * p.n + tok) * M + k] = cj[k];
          }
        }
        best = bj;
        best_S = bS;
        have_range = cnt > 0;
      } else {
        for (int wi = 0; wi < NW; wi++) {
          const uint32_t m = msk[wi * 32 + lane];
          if (m) best = 32 * wi + __ffs(m) - 1;
        }
      }
      if (best >= C) best = 0;
      // ---- (4) INT2 codes of the chosen centroid's residual; PSAC coefficients (thread = token) ----
      const int64_t grow = (int64_t)h * p.n + tok;
      const uint16_t *mub = cent + (int64_t)best * D;
      float mn0 = bmn0, mx0 = bmx0, mn1 = bmn1, mx1 = bmx1;  // Keys: the ranges of the scoring pass
      if (valid && !have_range) {
#pragma unroll
        for (int gi = 0; gi < 2; gi++) {
          uint4 mv[8];
#pragma unroll
          for (int cc = 0; cc < 8; cc++) mv[cc] = *(const uint4 *)(mub + 64 * gi + 8 * cc);
#pragma unroll
          for (int cc = 0; cc < 8; cc++) {
            uint64_t f2[4], m2[4];
            bf16x8_pairs(tc::lds128(xts + gi * TILE * 128 + tc::sw128_offset(row, 8 * cc)), f2);
            bf16x8_pairs(mv[cc], m2);
#pragma unroll
            for (int u = 0; u < 4; u++) {
              const uint64_t rr = tc::sub2(f2[u], m2[u]);
              if (gi == 0) {
                mn0 = tc::min3(mn0, tc::f2lo(rr), tc::f2hi(rr));
                mx0 = tc::max3(mx0, tc::f2lo(rr), tc::f2hi(rr));
              } else {
                mn1 = tc::min3(mn1, tc::f2lo(rr), tc::f2hi(rr));
                mx1 = tc::max3(mx1, tc::f2lo(rr), tc::f2hi(rr));
              }
            }
          }
        }
      }
      // per group: r_hat = mm + ss q with q = clamp(rint(r ii + zz), 0, 3); fp16 storage: mm = offset,
      // zz = 0; compact: mm = -z s (exact), zz = z
      float m0, s0, i0, m1, s1, i1, z0f = 0.f, z1f = 0.f;
      uint16_t mb0 = 0, sb0 = 0, mb1 = 0, sb1 = 0;
      uint32_t s8w = 0, zbits = 0;
      if (p.compact) {
        float need0 = 0.f, need1 = 0.f;
        int z0 = 0, z1 = 0;
        if (valid) {
          zp_range(mn0, mx0, need0, z0);
          zp_range(mn1, mx1, need1, z1);
        }
        // the tile's largest step per group (the epilogue group's 4 warps meet on sg_bar[e])
        float r0 = need0, r1 = need1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          r0 = fmaxf(r0, __shfl_xor_sync(0xffffffffu, r0, o));
          r1 = fmaxf(r1, __shfl_xor_sync(0xffffffffu, r1, o));
        }
        const int rb = (g >> 1) & 1;  // alternate buffers on alternate tiles of this group
        if (lane == 0) {
          red_sg[e][rb][sub][0] = r0;
          red_sg[e][rb][sub][1] = r1;
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sg_bar[e]);
        const bool ok = tc::mbar_wait(&sg_bar[e], (g >> 1) & 1, kWaitNs);
        if (__any_sync(0xffffffffu, !ok)) { *abort_v = 1; break; }
        float smax0 = 0.f, smax1 = 0.f;
#pragma unroll
        for (int w4 = 0; w4 < 4; w4++) {
          smax0 = fmaxf(smax0, red_sg[e][rb][w4][0]);
          smax1 = fmaxf(smax1, red_sg[e][rb][w4][1]);
        }
        const float sg0 = pow2_sigma(smax0), sg1 = pow2_sigma(smax1);
        if (sub == 0 && lane == 0)
          *(uint32_t *)(p.sigma + ((int64_t)h * ((p.n + TILE - 1) / TILE) + tile0 + g) * 2) =
              (uint32_t)__half_as_ushort(__float2half_rn(sg0)) | ((uint32_t)__half_as_ushort(__float2half_rn(sg1)) << 16);
        // s8 = ceil(need / sigma): exact quotient (sigma is a power of two); s = sigma s8 exact
        const float q0 = need0 == 0.f ? 0.f : ceilf(need0 * (1.0f / sg0));
        const float q1 = need1 == 0.f ? 0.f : ceilf(need1 * (1.0f / sg1));
        s0 = sg0 * q0;
        s1 = sg1 * q1;
        if (!(3.f * fmaxf(s0, s1) <= 65504.f)) qwm_dev_error(p.status, QWM_ERR_RANGE);  // z s must fit fp16
        i0 = s0 > 0.f ? __frcp_rn(s0) : 0.f;
        i1 = s1 > 0.f ? __frcp_rn(s1) : 0.f;
        z0f = (float)z0;
        z1f = (float)z1;
        m0 = -z0f * s0;
        m1 = -z1f * s1;
        s8w = (uint32_t)q0 | ((uint32_t)q1 << 8);
        zbits = (uint32_t)z0 | ((uint32_t)z1 << 2);
      } else if (valid) {
        int2_params(mn0, mx0, m0, s0, i0, mb0, sb0, p.status);
        int2_params(mn1, mx1, m1, s1, i1, mb1, sb1, p.status);
      }
      if (valid) {
        uint32_t packed[8];
        uint64_t Cv2[RMAX / 2];  // the PSAC coefficients as fp32 pairs {k, k + 1}
#pragma unroll
        for (int k = 0; k < RMAX / 2; k++) Cv2[k] = 0ull;
#pragma unroll
        for (int gi = 0; gi < 2; gi++) {
        uint4 mv[8];  // the group's half of the centroid row, loaded at once (one L2 latency per group)
#pragma unroll
        for (int cc = 0; cc < 8; cc++) mv[cc] = *(const uint4 *)(mub + 64 * gi + 8 * cc);
#pragma unroll
        for (int cc = 0; cc < 8; cc++) {
          const int ci = 8 * gi + cc;
          uint64_t f2[4], m2[4];
          bf16x8_pairs(tc::lds128(xts + gi * TILE * 128 + tc::sw128_offset(row, 8 * cc)), f2);
          bf16x8_pairs(mv[cc], m2);
          const bool g1 = gi == 1;
          const float mm = g1 ? m1 : m0, ss = g1 ? s1 : s0, ii = g1 ? i1 : i0, zz = g1 ? z1f : z0f;
          const uint64_t mm2 = tc::f2(mm, mm), ss2 = tc::f2(ss, ss), ii2 = tc::f2(ii, ii);
          const uint64_t mg2 = tc::f2(kRint, kRint);
          uint32_t bits = 0;
#pragma unroll
          for (int u = 0; u < 4; u++) {  // channels 8 ci + 2u, 8 ci + 2u + 1 as one fp32 pair
            const uint64_t rr2 = tc::sub2(f2[u], m2[u]);
            uint32_t q0, q1;
            uint64_t qf2;
            if (p.compact) {
              const float r0 = tc::f2lo(rr2), r1 = tc::f2hi(rr2);
              const float a0 = ss > 0.f ? rintf(__fadd_rn(__fmul_rn(r0, ii), zz)) : 0.f;
              const float a1 = ss > 0.f ? rintf(__fadd_rn(__fmul_rn(r1, ii), zz)) : 0.f;
              q0 = (uint32_t)fminf(fmaxf(a0, 0.f), 3.f);
              q1 = (uint32_t)fminf(fmaxf(a1, 0.f), 3.f);
              qf2 = tc::f2((float)q0, (float)q1);
            } else {
              // q = rint((r - m) * (1/s)): the rounded product lies in [0, 3] up to rounding (m <= r
              // and s >= (max r - m) / 3), so adding 2^23 rounds it to the integer q (ties to even)
              // in the low bits; with s = 0 (1/s taken as 0) the product is 0.  The max with 0 (a
              // no-op here) keeps the assembler from contracting the packed multiply and add into
              // one FMA, whose unrounded product would round the ties differently.
              const uint64_t y2 = tc::mul2(tc::sub2(rr2, mm2), ii2);
              const uint64_t z2 = tc::add2(tc::f2(fmaxf(tc::f2lo(y2), 0.f), fmaxf(tc::f2hi(y2), 0.f)), mg2);
              q0 = (uint32_t)z2 & 3u;
              q1 = (uint32_t)(z2 >> 32) & 3u;
              qf2 = tc::sub2(z2, mg2);
            }
            bits |= (q0 | (q1 << 2)) << (4 * u);
            if (KEY && R > 0) {
              // E = K - (mu + (m + s q)), then C += E_c U_r[c][:] channel by channel
              const uint64_t ev2 = tc::sub2(f2[u], tc::add2(m2[u], tc::fma2(ss2, qf2, mm2)));
#pragma unroll
              for (int hc = 0; hc < 2; hc++) {
                const float ev = hc ? tc::f2hi(ev2) : tc::f2lo(ev2);
                const uint64_t evd = tc::f2(ev, ev);
                const float *Uc = Us + (8 * ci + 2 * u + hc) * 16;
#pragma unroll
                for (int k4 = 0; k4 < RMAX / 4; k4++) {
                  const uint4 uv = *(const uint4 *)(Uc + 4 * k4);
                  Cv2[2 * k4] = tc::fma2(evd, u2(uv.x, uv.y), Cv2[2 * k4]);
                  Cv2[2 * k4 + 1] = tc::fma2(evd, u2(uv.z, uv.w), Cv2[2 * k4 + 1]);
                }
              }
            }
          }
          if (ci & 1) packed[ci >> 1] |= bits << 16;
          else packed[ci >> 1] = bits;
        }
        }
        uint4 *cdst = (uint4 *)(p.codes + grow * (D / 4));
        cdst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        cdst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        if (WIDE) ((uint16_t *)p.idx)[grow] = (uint16_t)best;
        else ((uint8_t *)p.idx)[grow] = (uint8_t)best;
        if (p.compact) {
          *(uint16_t *)(p.s8 + grow * 2) = (uint16_t)s8w;
          p.zp[grow] = (uint8_t)zbits;
        } else {
          *(uint32_t *)(p.scale + grow * 2) = (uint32_t)sb0 | ((uint32_t)sb1 << 16);
          *(uint32_t *)(p.minv + grow * 2) = (uint32_t)mb0 | ((uint32_t)mb1 << 16);
        }
        if (KEY && p.dbg_score) p.dbg_score[grow] = best_S;
        float Cv[RMAX];
#pragma unroll
        for (int k = 0; k < RMAX / 2; k++) {
          Cv[2 * k] = tc::f2lo(Cv2[k]);
          Cv[2 * k + 1] = tc::f2hi(Cv2[k]);
        }
        if (KEY && R > 0) {
          float a = 0.f;
#pragma unroll
          for (int k = 0; k < RMAX; k++)
            if (k < R) a = fmaxf(a, fabsf(Cv[k]));
          __half sch = __float2half_ru(__fdiv_ru(a, 127.0f));
          if (a == 0.f) sch = __float2half_rn(0.f);
          float sc = __half2float(sch);
          if (!isfinite(sc)) qwm_dev_error(p.status, QWM_ERR_RANGE);
          const float inv = sc > 0.f ? __frcp_rn(sc) : 0.f;
          int8_t c8[RMAX];
#pragma unroll
          for (int k = 0; k < RMAX; k++) {
            float qf = (k < R && sc > 0.f) ? rintf(__fmul_rn(Cv[k], inv)) : 0.f;
            c8[k] = (int8_t)fminf(fmaxf(qf, -127.f), 127.f);
          }
          if (p.gate || p.dbg_gate) {
            // w-weighted error of the token without and with the decoded correction C_hat U_r^T
            float e0 = 0.f, e1 = 0.f;
#pragma unroll 2
            for (int ci = 0; ci < D / 8; ci++) {
              float f[8], mu[8];
              bf16x8(tc::lds128(xts + (ci / 8) * TILE * 128 + tc::sw128_offset(row, 8 * (ci % 8))), f);
              bf16x8(*(const uint4 *)(mub + 8 * ci), mu);
              const bool g1 = ci >= 8;
              const float mm = g1 ? m1 : m0, ss = g1 ? s1 : s0;
              const uint32_t bits = packed[ci >> 1] >> (16 * (ci & 1));
#pragma unroll
              for (int u = 0; u < 8; u++) {
                const int c = 8 * ci + u;
                const float ev = __fsub_rn(f[u], __fadd_rn(mu[u], __fmaf_rn(ss, (float)((bits >> (2 * u)) & 3u), mm)));
                float corr = 0.f;
                const float *Uc = Us + c * 16;
#pragma unroll
                for (int k = 0; k < RMAX; k++) corr = fmaf(sc * (float)c8[k], Uc[k], corr);
                const float wc = wv[c], d1 = ev - corr;
                e0 = fmaf(wc, ev * ev, e0);
                e1 = fmaf(wc, d1 * d1, e1);
              }
            }
            if (p.dbg_gate) {
              p.dbg_gate[grow * 2] = e0;
              p.dbg_gate[grow * 2 + 1] = e1;
            }
            if (p.gate && !(e1 < e0)) {  // the correction does not help this token: drop it
#pragma unroll
              for (int k = 0; k < RMAX; k++) c8[k] = 0;
              sch = __float2half_rn(0.f);
            }
          }
#pragma unroll
          for (int k = 0; k < RMAX; k++) {
            if (k < R) {
              p.c[grow * R + k] = c8[k];
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
  __syncwarp();  // idle lanes of the TMA and MMA warps wait for lane 0 here
  __syncthreads();
  if (*abort_v && tid == 0) qwm_dev_error(p.status, QWM_ERR_DEVICE_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// The chunk's stored codebooks: the fp16 value of every bf16 centroid element (exact for magnitudes
// in [2^-17, 65504] and for 0; an element beyond the fp16 range records QWM_ERR_RANGE).  The
// attention's tensor cores take them as fp16 operands and the decoder reads them.
__global__ void codebook_f16_kernel(const uint16_t *__restrict__ ck, const uint16_t *__restrict__ cv, uint16_t *ok,
                                    uint16_t *ov, int64_t n8, int32_t *status) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * n8; i += (int64_t)gridDim.x * blockDim.x) {
    const bool key = i < n8;
    const int64_t e = key ? i : i - n8;
    const uint4 v = ((const uint4 *)(key ? ck : cv))[e];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
    bool bad = false;
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const float lo = __uint_as_float(w[u] << 16), hi = __uint_as_float(w[u] & 0xFFFF0000u);
      const __half hl = __float2half_rn(lo), hh = __float2half_rn(hi);
      bad |= (__hisinf(hl) != 0 && !isinf(lo)) || (__hisinf(hh) != 0 && !isinf(hi));
      o[u] = (uint32_t)__half_as_ushort(hl) | ((uint32_t)__half_as_ushort(hh) << 16);
    }
    if (bad) qwm_dev_error(status, QWM_ERR_RANGE);
    ((uint4 *)(key ? ok : ov))[e] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// WIDE operand image: block (slice, head) writes the slice's distance operands exactly as quant_kernel
// lays them out in shared memory (b = w . mu as bf16 hi + lo for Keys, mu for Values, 128-byte
// swizzled; the [-nw/2 hi, lo, 0 ...] rows), and raises the head's max |b_j| and max |nw_j| (img_max
// zeroed beforehand; non-negative floats order as integers).
__global__ void __launch_bounds__(256) quant_image_kernel(const uint16_t *__restrict__ cent_all,
                                                          const float *__restrict__ w, const float *__restrict__ Bq,
                                                          int C, int key, unsigned char *__restrict__ img_all,
                                                          float *img_max) {
  __shared__ float wv[D];
  const int sl = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const QSmem L(C, key != 0, true);
  const int NSL = C / kSlice;
  unsigned char *img = img_all + ((int64_t)h * NSL + sl) * L.an;
  const uint16_t *cent = cent_all + ((int64_t)h * C + (int64_t)sl * kSlice) * D;
  for (int c = tid; c < D; c += 256) wv[c] = (key && w) ? w[(int64_t)h * D + c] : 1.0f;
  __syncthreads();
  for (int e = tid; e < kSlice * (D / 8); e += 256) {
    const int j = e / (D / 8), ci = e % (D / 8);
    float mu[8];
    bf16x8(*(const uint4 *)(cent + (int64_t)j * D + 8 * ci), mu);
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const float *bq = (key && Bq) ? Bq + ((int64_t)h * C + (int64_t)sl * kSlice + j) * D + 8 * ci : nullptr;
      const float b0 = bq ? bq[2 * u] : (key ? __fmul_rn(wv[8 * ci + 2 * u], mu[2 * u]) : mu[2 * u]);
      const float b1 = bq ? bq[2 * u + 1] : (key ? __fmul_rn(wv[8 * ci + 2 * u + 1], mu[2 * u + 1]) : mu[2 * u + 1]);
      const float h0 = __bfloat162float(__float2bfloat16_rn(b0)), h1 = __bfloat162float(__float2bfloat16_rn(b1));
      hw[u] = (uint32_t)f32_to_bf16_rn(h0) | ((uint32_t)f32_to_bf16_rn(h1) << 16);
      lw[u] = (uint32_t)f32_to_bf16_rn(b0 - h0) | ((uint32_t)f32_to_bf16_rn(b1 - h1) << 16);
    }
    const uint32_t off = (ci / 8) * kSlice * 128 + tc::sw128_offset(j, 8 * (ci % 8));
    *(uint4 *)(img + L.bh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    if (key) *(uint4 *)(img + L.bl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  float bmax = 0.f, nwmax = 0.f;
  for (int j = warp; j < kSlice; j += 8) {
    float mu[4];
    unpack4(*(const uint2 *)(cent + (int64_t)j * D + 4 * lane), mu);
    float s = 0.f, bb = 0.f;
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const float wm = (key && Bq) ? Bq[((int64_t)h * C + (int64_t)sl * kSlice + j) * D + 4 * lane + u]
                                   : __fmul_rn(wv[4 * lane + u], mu[u]);
      s = fmaf(wm, mu[u], s);
      bb = fmaf(wm, wm, bb);
    }
    s = warp_sum(s);
    bb = warp_sum(bb);
    if (lane < 8) {
      uint32_t wd = 0u;
      if (lane == 0) {
        const float t = -0.5f * s, th = __bfloat162float(__float2bfloat16_rn(t));
        wd = (uint32_t)f32_to_bf16_rn(th) | ((uint32_t)f32_to_bf16_rn(t - th) << 16);
      }
      *(uint32_t *)(img + L.bn + noswz16(j, 2 * lane)) = wd;
    }
    bmax = fmaxf(bmax, sqrtf(bb));
    nwmax = fmaxf(nwmax, fabsf(s));
  }
  if (lane == 0) {
    atomicMax((int *)&img_max[2 * h], __float_as_int(bmax));
    atomicMax((int *)&img_max[2 * h + 1], __float_as_int(nwmax));
  }
}

// The Query second moment M = S / n of every head (IEEE division in fp32); the identity while no Query
// has been seen (n = 0: uniform weights, as at a cold start).
__global__ void __launch_bounds__(256) mfull_kernel(const float *__restrict__ S, const int64_t *__restrict__ n_seen,
                                                    float *__restrict__ M) {
  const int h = blockIdx.y, e = blockIdx.x * 256 + threadIdx.x;
  const int64_t nh = n_seen[h];
  const int64_t i = (int64_t)h * D * D + e;
  M[i] = nh > 0 ? __fdiv_rn(S[i], (float)nh) : (e / D == e % D ? 1.0f : 0.0f);
}

// Full-form ranking operand: b_j = M mu_j for every centroid j of every head (M symmetric, so thread c
// reads column c of M, coalesced across the block); mu_j staged in shared memory.
__global__ void __launch_bounds__(128) mfull_b_kernel(const float *__restrict__ M, const uint16_t *__restrict__ cent,
                                                      int C, float *__restrict__ Bq) {
  __shared__ float mu[D];
  const int j = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  mu[c] = bf16_to_f32(cent[((int64_t)h * C + j) * D + c]);
  __syncthreads();
  const float *Mh = M + (int64_t)h * D * D;
  float acc = 0.f;
  for (int c2 = 0; c2 < D; c2++) acc = fmaf(Mh[(int64_t)c2 * D + c], mu[c2], acc);
  Bq[((int64_t)h * C + j) * D + c] = acc;
}

template <bool KEY, int RMAX, int MP1, bool WIDE>
cudaError_t launch_one(const TensorMap128 &tmap, const QParams &p, int H, int smem, cudaStream_t st) {
  cudaError_t e =
      cudaFuncSetAttribute(quant_kernel<KEY, RMAX, MP1, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  quant_kernel<KEY, RMAX, MP1, WIDE><<<dim3(p.G, H), kThreads, smem, st>>>(tmap, p);
  return cudaGetLastError();
}

template <bool WIDE>
cudaError_t launch_pass(const TensorMap128 &tmap, const QParams &p, bool key, int H, int smem, cudaStream_t st) {
  // MP1 bounds the candidate count (top_m <= MP1 - 1): the small variant serves top_m 1..4
  if (!key) return launch_one<false, 8, 2, WIDE>(tmap, p, H, smem, st);
  if (p.rank <= 8 && p.top_m <= 4) return launch_one<true, 8, 5, WIDE>(tmap, p, H, smem, st);
  if (p.rank <= 8) return launch_one<true, 8, QWM_MAX_TOPM + 1, WIDE>(tmap, p, H, smem, st);
  if (p.top_m <= 4) return launch_one<true, 16, 5, WIDE>(tmap, p, H, smem, st);
  return launch_one<true, 16, QWM_MAX_TOPM + 1, WIDE>(tmap, p, H, smem, st);
}

}  // namespace

// Workspace of the WIDE operand images: [H][C / kSlice] slices (Keys' size; each a multiple of
// 1024 bytes), then img_max [H][2].
size_t quantize_image_bytes(int H, int C) {
  if (C <= QWM_MAX_RESIDENT_CENTROIDS) return 0;
  return (size_t)H * (C / kSlice) * QSmem(C, true, true).an + (size_t)H * 2 * sizeof(float);
}

cudaError_t launch_quantize(const qwm_config &cfg, const uint16_t *k, const uint16_t *v, int64_t n, const float *w,
                            const float *S, const int64_t *n_seen, float *Mq_ws, float *Bq, const uint16_t *u_r,
                            const qwm_chunk &out, const qwm_debug *dbg, int32_t *status, int num_sms,
                            unsigned char *img, cudaStream_t st, cudaStream_t side, cudaEvent_t fork,
                            cudaEvent_t join) {
  const float *Mq = S ? Mq_ws : nullptr;
  const int H = cfg.heads, C = cfg.n_centroids;
  const bool wide = C > QWM_MAX_RESIDENT_CENTROIDS;
  float *img_max = wide ? (float *)(img + (size_t)H * (C / kSlice) * QSmem(C, true, true).an) : nullptr;
  const int64_t tiles = (n + TILE - 1) / TILE;
  // one CTA per SM at most (each holds ~220 KB of shared memory): a single wave
  int G = num_sms / H;
  if (G > tiles) G = (int)tiles;
  if (G < 1) G = 1;
  {
    const int64_t n8 = (int64_t)H * C * QWM_D / 8;
    codebook_f16_kernel<<<num_sms, 256, 0, st>>>(out.cent_k, out.cent_v, out.cent_k16, out.cent_v16, n8, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (Mq) {  // full-form ranking: M = S / n, then the Key distance operand b_j = M mu_j
    mfull_kernel<<<dim3(D * D / 256, H), 256, 0, st>>>(S, n_seen, Mq_ws);
    mfull_b_kernel<<<dim3(C, H), D, 0, st>>>(Mq, out.cent_k, C, Bq);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // The Value pass runs on the context's second stream beside the Key pass (the two read and write
  // disjoint data), and the caller's stream waits for it at the end.  With streamed 1024-centroid
  // codebooks both passes share one operand image, so they run one after the other.
  const bool concurrent = !wide;
  if (concurrent) {
    cudaError_t e = cudaEventRecord(fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, fork, 0);
    if (e != cudaSuccess) return e;
  }
  for (int pass = 0; pass < 2; pass++) {
    const bool key = pass == 0;
    cudaStream_t ps = (concurrent && !key) ? side : st;
    TensorMap128 tmap;
    if (!make_tmap_rows128_bf16(&tmap, key ? k : v, (uint64_t)H * n, TILE)) return cudaErrorInvalidValue;
    QParams p;
    p.n = n; p.w = key ? w : nullptr; p.u_r = key ? u_r : nullptr;
    p.cent = key ? out.cent_k : out.cent_v;
    p.C = C; p.top_m = cfg.top_m; p.rank = (key && u_r) ? cfg.rank : 0; p.G = G;
    p.img = img; p.img_max = img_max;
    p.codes = key ? out.k_codes : out.v_codes; p.idx = key ? out.k_idx : out.v_idx;
    p.scale = key ? out.k_scale : out.v_scale; p.minv = key ? out.k_min : out.v_min;
    p.compact = cfg.storage == QWM_STORAGE_COMPACT;
    p.gate = (key && cfg.psac_gate) ? 1 : 0;
    p.s8 = key ? out.k_s8 : out.v_s8; p.zp = key ? out.k_zp : out.v_zp;
    p.sigma = key ? out.k_sigma : out.v_sigma;
    p.wk = key ? w : nullptr;
    p.Mq = key ? Mq : nullptr;
    p.Bq = (key && Mq) ? Bq : nullptr;
    p.dbg_gate = (key && dbg) ? dbg->gate_err : nullptr;
    p.c = out.c; p.c_scale = out.c_scale;
    p.dbg_c = (key && dbg) ? dbg->c_f32 : nullptr;
    p.dbg_cand = (key && dbg) ? dbg->cand : nullptr;
    p.dbg_score = (key && dbg) ? dbg->score : nullptr;
    p.status = status;
    const int smem = QSmem(C, key, wide).total + 1024;
    cudaError_t e;
    if (wide) {  // this pass's operand image (the two passes reuse one buffer, in stream order)
      e = cudaMemsetAsync(img_max, 0, (size_t)H * 2 * sizeof(float), st);
      if (e != cudaSuccess) return e;
      quant_image_kernel<<<dim3(C / kSlice, H), 256, 0, st>>>(p.cent, p.w, p.Bq, C, key ? 1 : 0, img, img_max);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      e = launch_pass<true>(tmap, p, key, H, smem, st);
    } else {
      e = launch_pass<false>(tmap, p, key, H, smem, ps);
    }
    if (e != cudaSuccess) return e;
  }
  if (concurrent) {
    cudaError_t e = cudaEventRecord(join, side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, join, 0);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
