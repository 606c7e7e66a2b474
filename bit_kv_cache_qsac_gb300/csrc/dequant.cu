// Step 5': BF16 reconstruction of packed chunks (QuantWM English v2 summary §D.1: the fused decoder
// unpacks the INT2 residuals, rebuilds the affine parameters, gathers the centroids and adds the
// PSAC term; Chinese summary step (5)).
//   K_hat = (mu^K_idx + (m + s q)) + sum_k (sC c_k) U_r[:, k],   V_hat = mu^V_idx + (m + s q),
// evaluated in fp32 (m + s q is exact: s q is exact and both are fp16 values) and rounded to bf16.
//
// A bandwidth kernel: per token-head it reads 92 bytes of packed data (plus a codebook row that
// stays in L2) and writes 512 bytes of bf16, so it is bound by the HBM write stream.  One CTA takes
// 256 tokens of one chunk for one head, 16 threads per token (8 channels each, one 16-byte store per
// tensor), in passes of 16 tokens; the token metadata is staged in shared memory first, and the
// centroid rows of four passes are gathered before they are used.  A thread keeps the same 8 channels for the whole
// CTA, so it holds their rows of U_r (fp32) in registers, loaded once (16-byte loads).  All chunks of a call go in one launch, each chunk's
// rows written at its offset in the [H][sum N][d] output.  The centroids come from the chunk's stored
// fp16 codebook; the PSAC coefficients from the dense [H][N][r] arrays or, in the per-head layout,
// through the head's entry (its rank, and for a sparse head the tile bitmap).
#include "qwm_internal.cuh"
#include "tc.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int kTok = 256;                // tokens per CTA
constexpr int kThreads = 256;            // 16 threads per token, 16 tokens per pass
constexpr int kPasses = kTok / (kThreads / 16);
constexpr int kMaxChunks = 128;

struct DqChunk {
  int64_t n;        // tokens of the chunk
  int64_t out0;     // output row of its token 0
  int tile0;        // first CTA column of the chunk
  int rank;         // PSAC rank (0: none)
  const uint8_t *k_codes, *v_codes, *k_idx, *v_idx, *k_s8, *v_s8, *k_zp, *v_zp;
  const uint16_t *k_scale, *k_min, *v_scale, *v_min, *k_sigma, *v_sigma, *cent_k16, *cent_v16, *c_scale, *u_r;
  const int8_t *c;
  int per_head;     // QWM_C_PER_HEAD coefficients
  const qwm_psac_head *c_heads;
  const uint32_t *c_mask;
  const int32_t *c_tile_rank;
};

struct DqParams {
  int H, C, n_chunks;
  int64_t n_out;    // output rows per head (sum of the chunks' tokens)
  uint16_t *k_hat, *v_hat;
  DqChunk ch[kMaxChunks];
};

__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}

__device__ __forceinline__ uint4 to_bf16x8(const float (&x)[8]) {
  uint32_t o[4];
#pragma unroll
  for (int u = 0; u < 4; u++) o[u] = (uint32_t)f32_to_bf16_rn(x[2 * u]) | ((uint32_t)f32_to_bf16_rn(x[2 * u + 1]) << 16);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// A CTA's token metadata, staged in shared memory by one coalesced pass (thread = token) so that the
// decode loop reads it from there: codes, centroid indices, the INT2 step and offset of both groups
// (fp16 pairs; the compact form's s = sigma s8 and m = -z s are exact fp16 values), and, for Keys,
// the PSAC row resolved from either coefficient layout (dense [H][N][r], or per head through its
// entry).
struct DqStage {
  uint4 codes[kTok][2];  // [token][32 bytes]
  uint32_t s2[kTok];     // fp16 step of group 0 | group 1 << 16
  uint32_t m2[kTok];     // fp16 offset, likewise
  uint16_t idx[kTok];
  uint4 c[kTok];         // Keys: up to 16 PSAC coefficient bytes (zero past the row's rank)
  float sc[kTok];        // Keys: PSAC scale sC (0: no correction)
};

template <bool VAL, bool IDX16, bool COMPACT>
__device__ __forceinline__ void stage_tensor(const DqChunk &c, int h, int64_t tok, int C, DqStage &st, int t) {
  const int64_t row = (int64_t)h * c.n + tok;
  const uint4 *cp = (const uint4 *)((VAL ? c.v_codes : c.k_codes) + row * (D / 4));
  st.codes[t][0] = cp[0];
  st.codes[t][1] = cp[1];
  const uint8_t *ip = VAL ? c.v_idx : c.k_idx;
  const int j = IDX16 ? (int)((const uint16_t *)ip)[row] : (int)ip[row];
  st.idx[t] = (uint16_t)(j < C ? j : C - 1);  // never read past the codebook
  if (COMPACT) {
    const int64_t tiles = (c.n + 127) / 128;
    const uint32_t sg2 = *(const uint32_t *)((VAL ? c.v_sigma : c.k_sigma) + ((int64_t)h * tiles + tok / 128) * 2);
    const uint32_t s8 = *(const uint16_t *)((VAL ? c.v_s8 : c.k_s8) + row * 2);
    const uint32_t z = (VAL ? c.v_zp : c.k_zp)[row];
    uint32_t s2 = 0, m2 = 0;
#pragma unroll
    for (int g = 0; g < 2; g++) {
      const float sv = f16_to_f32((uint16_t)(sg2 >> (16 * g))) * (float)((s8 >> (8 * g)) & 0xFFu);
      const float mv = -(float)((z >> (2 * g)) & 3u) * sv;
      s2 |= (uint32_t)__half_as_ushort(__float2half_rn(sv)) << (16 * g);
      m2 |= (uint32_t)__half_as_ushort(__float2half_rn(mv)) << (16 * g);
    }
    st.s2[t] = s2;
    st.m2[t] = m2;
  } else {
    st.s2[t] = *(const uint32_t *)((VAL ? c.v_scale : c.k_scale) + row * 2);
    st.m2[t] = *(const uint32_t *)((VAL ? c.v_min : c.k_min) + row * 2);
  }
}

// One tensor per launch (VAL: Values, else Keys), so that the Value decoder, which holds no basis,
// runs at the occupancy its smaller register footprint allows.  RU: bound on the PSAC rank of the
// call's chunks (0, 8 or 16; 0 for Values).
template <bool VAL, int RU, bool IDX16, bool COMPACT>
__global__ void __launch_bounds__(kThreads, RU > 8 ? 1 : (RU > 0 ? 2 : 3))
    dequant_kernel(const __grid_constant__ DqParams p) {
  __shared__ DqStage st;
  const int h = blockIdx.y, tid = threadIdx.x;
  int t = 0;  // the chunk of this CTA column (chunks are in column order)
  while (t + 1 < p.n_chunks && p.ch[t + 1].tile0 <= (int)blockIdx.x) t++;
  const DqChunk &c = p.ch[t];
  const int64_t tok0 = (int64_t)((int)blockIdx.x - c.tile0) * kTok;
  const int R = c.rank;
  const bool psac = !VAL && RU > 0 && R > 0;
  uint16_t *out = VAL ? p.v_hat : p.k_hat;
  // ---- staging: thread = token ----
  {
    const int64_t tok = tok0 + tid;
    if (tok < c.n) {
      stage_tensor<VAL, IDX16, COMPACT>(c, h, tok, p.C, st, tid);
      if (!VAL && RU > 0) {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        float sc = 0.f;
        if (psac) {
          int64_t crow = (int64_t)h * c.n + tok;
          int rr = R;
          const int8_t *cbase = c.c;
          const uint16_t *sbase = c.c_scale;
          bool has = true;
          if (c.per_head) {  // the head's rank and layout
            const qwm_psac_head hd = c.c_heads[h];
            has = psac_row(hd, c.c_mask, c.c_tile_rank, (c.n + 127) / 128, h, tok, crow);
            rr = hd.rank;
            cbase += hd.c_off;
            sbase += hd.s_off;
          }
          if (has) {
            sc = f16_to_f32(sbase[crow]);
            const int8_t *cc = cbase + crow * rr;
            if (!c.per_head && rr == 8) {
              const uint2 v = *(const uint2 *)cc;
              w[0] = v.x; w[1] = v.y;
            } else {
#pragma unroll
              for (int k = 0; k < 16; k++)
                if (k < rr) w[k >> 2] |= ((uint32_t)(uint8_t)cc[k]) << (8 * (k & 3));
            }
          }
        }
        st.c[tid] = make_uint4(w[0], w[1], w[2], w[3]);
        st.sc[tid] = sc;
      }
    }
  }
  // ---- Keys: this thread's 8 rows of U_r (zero past the rank), packed in pairs of channels ----
  const int cb = tid & 15, c0 = 8 * cb, g = c0 / QWM_GROUP;
  constexpr int kRU = RU > 0 ? RU : 1;
  uint64_t U2[4][kRU];
#pragma unroll
  for (int u = 0; u < 4; u++)
#pragma unroll
    for (int k = 0; k < kRU; k++) U2[u][k] = 0ull;
  if (RU > 0 && psac) {
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const uint16_t *ur = c.u_r + ((int64_t)h * D + c0 + u) * R;
      float uf[kRU];
      if (R == RU) {  // a full row: 16-byte loads
#pragma unroll
        for (int k8 = 0; k8 < (kRU + 7) / 8; k8++) {
          const uint4 v = ((const uint4 *)ur)[k8];
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; q++) {
            if (8 * k8 + 2 * q + 1 < kRU) {
              uf[8 * k8 + 2 * q] = __uint_as_float(w[q] << 16);
              uf[8 * k8 + 2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
            }
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < kRU; k++) uf[k] = k < R ? bf16_to_f32(ur[k]) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < kRU; k++) U2[u >> 1][k] |= (uint64_t)__float_as_uint(uf[k]) << (32 * (u & 1));
    }
  }
  __syncthreads();
  // ---- decode: 16 threads per token (8 channels each), 16 tokens per pass.  The centroid rows of
  // four passes are gathered first (the loads cannot move past the output stores on their own: the
  // compiler has to assume the output may alias the codebook) ----
  constexpr int kU = VAL ? 8 : 4;  // passes whose centroid rows are gathered together
  const uint16_t *cent = (VAL ? c.cent_v16 : c.cent_k16) + (int64_t)h * p.C * D + c0;
  const int nt = (int)((c.n - tok0) < kTok ? (c.n - tok0) : kTok);  // tokens of this CTA
#pragma unroll 1
  for (int p0 = 0; p0 < kPasses; p0 += kU) {
    uint4 mu[kU];
#pragma unroll
    for (int a = 0; a < kU; a++) {
      const int tt = (p0 + a) * (kThreads / 16) + (tid >> 4);
      mu[a] = tt < nt ? *(const uint4 *)(cent + (int64_t)st.idx[tt] * D) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int a = 0; a < kU; a++) {
      const int tt = (p0 + a) * (kThreads / 16) + (tid >> 4);
      if (tt >= nt) continue;
      const uint4 cw = st.codes[tt][cb >> 3];
      const uint32_t cword = (cb & 4) ? ((cb & 2) ? cw.w : cw.z) : ((cb & 2) ? cw.y : cw.x);
      const uint32_t b2 = (cb & 1) ? (cword >> 16) : (cword & 0xFFFFu);  // the 8 codes of channels c0..c0+7
      const float s = f16_to_f32((uint16_t)(st.s2[tt] >> (16 * g)));
      const float m = f16_to_f32((uint16_t)(st.m2[tt] >> (16 * g)));
      const uint32_t muw[4] = {mu[a].x, mu[a].y, mu[a].z, mu[a].w};
      float x[8];
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const float q = (float)((b2 >> (2 * u)) & 3u);
        const float muf = f16_to_f32((uint16_t)(muw[u / 2] >> (16 * (u & 1))));
        x[u] = __fadd_rn(muf, __fmaf_rn(s, q, m));
      }
      if (RU > 0 && psac) {
        const float sC = st.sc[tt];
        const uint4 cw2 = st.c[tt];
        const uint32_t w[4] = {cw2.x, cw2.y, cw2.z, cw2.w};
        uint64_t x2[4];
#pragma unroll
        for (int u = 0; u < 4; u++) x2[u] = pk2(x[2 * u], x[2 * u + 1]);
#pragma unroll
        for (int k = 0; k < kRU; k++) {
          const float chat = sC * (float)(int8_t)((w[k >> 2] >> (8 * (k & 3))) & 0xFFu);  // exact
          const uint64_t c2 = pk2(chat, chat);
#pragma unroll
          for (int u = 0; u < 4; u++) x2[u] = tc::fma2(c2, U2[u][k], x2[u]);  // one rounding each, as fmaf
        }
#pragma unroll
        for (int u = 0; u < 4; u++) { x[2 * u] = tc::f2lo(x2[u]); x[2 * u + 1] = tc::f2hi(x2[u]); }
      }
      const int64_t orow = (int64_t)h * p.n_out + c.out0 + tok0 + tt;
      *(uint4 *)(out + orow * D + c0) = to_bf16x8(x);
    }
  }
}

template <bool VAL, int RU, bool IDX16>
cudaError_t launch_one(const DqParams &p, dim3 grid, bool compact, cudaStream_t st) {
  if (compact) dequant_kernel<VAL, RU, IDX16, true><<<grid, kThreads, 0, st>>>(p);
  else dequant_kernel<VAL, RU, IDX16, false><<<grid, kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

template <bool IDX16>
cudaError_t launch_idx(const DqParams &p, dim3 grid, bool compact, int rmax, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  if (p.k_hat) {
    if (rmax == 0) e = launch_one<false, 0, IDX16>(p, grid, compact, st);
    else if (rmax <= 8) e = launch_one<false, 8, IDX16>(p, grid, compact, st);
    else e = launch_one<false, 16, IDX16>(p, grid, compact, st);
  }
  if (e == cudaSuccess && p.v_hat) e = launch_one<true, 0, IDX16>(p, grid, compact, st);
  return e;
}

}  // namespace

cudaError_t launch_dequantize(const qwm_config &cfg, const qwm_chunk *chunks, int n_chunks, uint16_t *k_hat,
                              uint16_t *v_hat, cudaStream_t st) {
  DqParams p;  // passed by value (about 23 KB of kernel parameters)
  p.H = cfg.heads;
  p.C = cfg.n_centroids;
  p.k_hat = k_hat;
  p.v_hat = v_hat;
  int used = 0, tiles = 0, rmax = 0;
  int64_t rows = 0;
  for (int i = 0; i < n_chunks; i++) {
    const qwm_chunk &c = chunks[i];
    if (c.n_tokens == 0) continue;
    if (used == kMaxChunks) return cudaErrorInvalidValue;
    DqChunk &a = p.ch[used++];
    a.n = c.n_tokens; a.out0 = rows; a.tile0 = tiles; a.rank = c.rank_eff;
    a.k_codes = c.k_codes; a.v_codes = c.v_codes;
    a.k_idx = (const uint8_t *)c.k_idx; a.v_idx = (const uint8_t *)c.v_idx;
    a.k_s8 = c.k_s8; a.v_s8 = c.v_s8; a.k_zp = c.k_zp; a.v_zp = c.v_zp;
    a.k_scale = c.k_scale; a.k_min = c.k_min; a.v_scale = c.v_scale; a.v_min = c.v_min;
    a.k_sigma = c.k_sigma; a.v_sigma = c.v_sigma;
    a.cent_k16 = c.cent_k16; a.cent_v16 = c.cent_v16; a.c_scale = c.c_scale; a.u_r = c.u_r; a.c = c.c;
    a.per_head = c.rank_eff > 0 && c.c_layout == QWM_C_PER_HEAD;
    a.c_heads = c.c_heads; a.c_mask = c.c_mask; a.c_tile_rank = c.c_tile_rank;
    rows += c.n_tokens;
    tiles += (int)((c.n_tokens + kTok - 1) / kTok);
    if (c.rank_eff > rmax) rmax = c.rank_eff;
  }
  p.n_chunks = used;
  p.n_out = rows;
  if (used == 0 || (!k_hat && !v_hat)) return cudaSuccess;
  const dim3 grid((unsigned)tiles, (unsigned)cfg.heads);
  const bool idx16 = cfg.n_centroids > 256, compact = cfg.storage == QWM_STORAGE_COMPACT;
  return idx16 ? launch_idx<true>(p, grid, compact, rmax, st) : launch_idx<false>(p, grid, compact, rmax, st);
}
