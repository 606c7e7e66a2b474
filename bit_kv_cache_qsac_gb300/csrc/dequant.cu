// Step 5': BF16 reconstruction of packed chunks (QuantWM English v2 summary §D.1: the fused decoder
// unpacks the INT2 residuals, rebuilds the affine parameters, gathers the centroids and adds the
// PSAC term; Chinese summary step (5)).
//   K_hat = (mu^K_idx + (m + s q)) + sC * sum_k c_k U_r[:, k],   V_hat = mu^V_idx + (m + s q),
// evaluated in fp32 and rounded to bf16.
//
// A bandwidth kernel: per token-head it reads about 50 bytes of packed data (plus a codebook row that
// stays in L2) and writes 256 bytes of bf16, so it is bound by the HBM write stream.  One CTA takes
// 256 tokens of one chunk for one head; the token metadata is staged in shared memory first (one
// coalesced pass, thread = token), and each centroid gather is issued ahead of the stores that come
// before its use (the compiler has to assume the output may alias the codebook, so it cannot move
// the loads past the stores by itself).
// Values (and Keys without PSAC): 16 threads per token, 8 channels each, one 16-byte store per
// token.  Keys with PSAC: the correction sum_k c_k U_r[:, k] of 16 tokens x 128 channels is one
// warp's set of mma.sync m16n8k8 (rank <= 8) or m16n8k16 products: bf16 operands (the int8
// coefficients and the bf16 basis are exact bf16 values, so every product is exact) with fp32
// accumulation.  The n-tiles' columns are permuted so that each thread's accumulators are 4 runs of
// 8 consecutive channels (32 i + 8 t .. + 7 for the thread's t = lane % 4) of its two tokens (rows
// lane / 4 and lane / 4 + 8), decoded in place and stored 16 bytes at a time.  All chunks of a call
// go in one launch, each chunk's rows written at its offset in the [H][sum N][d] output.  The
// centroids come from the chunk's stored fp16 codebook; the PSAC coefficients from the dense
// [H][N][r] arrays or, in the per-head layout, through the head's entry (its rank, and for a
// sparse head the tile bitmap).
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

// Eight channels of one token: x_u = mu_u + (m + s q_u) (+ sC corr_u), rounded to bf16.  `bits` holds
// the 8 two-bit codes (channel u in bits 2u..2u+1), `mu` the 8 fp16 centroid elements.
template <bool CORR>
__device__ __forceinline__ uint4 decode8(const uint4 mu, uint32_t bits, float s, float m, float sc,
                                         const float (&corr)[8]) {
  const uint32_t muw[4] = {mu.x, mu.y, mu.z, mu.w};
  uint32_t o[4];
#pragma unroll
  for (int v = 0; v < 4; v++) {
    float x[2];
#pragma unroll
    for (int e = 0; e < 2; e++) {
      const int u = 2 * v + e;
      const float q = (float)((bits >> (2 * u)) & 3u);
      const float muf = f16_to_f32((uint16_t)(muw[v] >> (16 * e)));
      x[e] = __fadd_rn(muf, __fmaf_rn(s, q, m));
      if (CORR) x[e] = __fmaf_rn(sc, corr[u], x[e]);
    }
    o[v] = tc::pack_bf16x2(x[0], x[1]);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Staging of one CTA's token metadata (thread = token; tokens past the chunk staged as zeros, so
// that every later read of the stage is in bounds and decodes to finite values).
template <bool VAL, bool PSAC, bool IDX16, bool COMPACT>
__device__ __forceinline__ void stage_cta(const DqChunk &c, int h, int64_t tok0, int C, DqStage &st, int tid) {
  const int64_t tok = tok0 + tid;
  if (tok >= c.n) {
    st.codes[tid][0] = st.codes[tid][1] = make_uint4(0, 0, 0, 0);
    st.s2[tid] = st.m2[tid] = 0u;
    st.idx[tid] = 0;
    if (PSAC) {
      st.c[tid] = make_uint4(0, 0, 0, 0);
      st.sc[tid] = 0.f;
    }
    return;
  }
  stage_tensor<VAL, IDX16, COMPACT>(c, h, tok, C, st, tid);
  if (PSAC) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    float sc = 0.f;
    if (c.rank > 0) {
      int64_t crow = (int64_t)h * c.n + tok;
      int rr = c.rank;
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

__device__ __forceinline__ int chunk_of_cta(const DqParams &p) {
  int t = 0;  // chunks are in CTA-column order
  while (t + 1 < p.n_chunks && p.ch[t + 1].tile0 <= (int)blockIdx.x) t++;
  return t;
}

// Values, or Keys without any PSAC term in the call: 16 threads per token (8 channels each), 16
// tokens per pass; the centroid rows of 8 passes are gathered before they are used.  Four CTAs per
// SM (64 registers), as the Key kernel below.
template <bool VAL, bool IDX16, bool COMPACT>
__global__ void __launch_bounds__(kThreads, 4) dequant_kernel(const __grid_constant__ DqParams p) {
  __shared__ DqStage st;
  const int h = blockIdx.y, tid = threadIdx.x;
  const DqChunk &c = p.ch[chunk_of_cta(p)];
  const int64_t tok0 = (int64_t)((int)blockIdx.x - c.tile0) * kTok;
  stage_cta<VAL, false, IDX16, COMPACT>(c, h, tok0, p.C, st, tid);
  __syncthreads();
  constexpr int kU = 8;
  const int cb = tid & 15, c0 = 8 * cb, g = c0 / QWM_GROUP;
  const uint16_t *cent = (VAL ? c.cent_v16 : c.cent_k16) + (int64_t)h * p.C * D + c0;
  uint16_t *out = (VAL ? p.v_hat : p.k_hat) + ((int64_t)h * p.n_out + c.out0 + tok0) * D + c0;
  const int nt = (int)((c.n - tok0) < kTok ? (c.n - tok0) : kTok);  // tokens of this CTA
  const float none[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int p0 = 0; p0 < kPasses; p0 += kU) {
    if (p0 * (kThreads / 16) >= nt) break;
    uint4 mu[kU];
#pragma unroll
    for (int a = 0; a < kU; a++) {
      const int tt = (p0 + a) * (kThreads / 16) + (tid >> 4);
      mu[a] = *(const uint4 *)(cent + (int64_t)st.idx[tt] * D);  // staged index 0 past the chunk
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
      *(uint4 *)(out + (int64_t)tt * D) = decode8<false>(mu[a], b2, s, m, 0.f, none);
    }
  }
}

// One warp-level product D[16][8] += A[16][K] B[K][8] (bf16 A, B; fp32 D), K = 8 or 16.
template <int KS>
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[KS / 4], const uint32_t (&b)[KS / 8]) {
  if constexpr (KS == 8) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(b[0]));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
}

// Coefficients k = 2 t, 2 t + 1 (+ 8 kb) of a staged row as a bf16 pair (int8 values: exact).
__device__ __forceinline__ uint32_t coef_pair(const uint4 cw, int t, int kb) {
  const uint32_t w = kb == 0 ? ((t >> 1) ? cw.y : cw.x) : ((t >> 1) ? cw.w : cw.z);
  const uint32_t hw = (t & 1) ? (w >> 16) : (w & 0xFFFFu);
  return tc::pack_bf16x2((float)(int8_t)(hw & 0xFFu), (float)(int8_t)(hw >> 8));
}

// Keys with PSAC (RU: bound on the call's ranks, 8 or 16).  Warp w decodes the 16-token tiles w and
// w + 8 of the CTA; thread (g, t) = (lane / 4, lane % 4) owns tokens g and g + 8 of a tile and
// channels 32 i + 8 t .. 32 i + 8 t + 7, i = 0..3.  Column j of n-tile n = 4 i + a is channel
// 32 i + 8 (j / 2) + 2 a + j % 2, so the accumulator pair (a, 2 t + e) of the fragment layout is the
// thread's channel 32 i + 8 t + 2 a + e.
template <int RU, bool IDX16, bool COMPACT>
__global__ void __launch_bounds__(kThreads, 4) dequant_key_kernel(const __grid_constant__ DqParams p) {
  constexpr int KS = RU > 8 ? 16 : 8, KB = KS / 8;
  __shared__ DqStage st;
  const int h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const DqChunk &c = p.ch[chunk_of_cta(p)];
  const int64_t tok0 = (int64_t)((int)blockIdx.x - c.tile0) * kTok;
  const int R = c.rank;
  // B fragments in shared memory, in fragment order: word (n * KB + kb) * 32 + lane holds, for lane
  // (g, t), the basis entries k = 2 t + 8 kb, k + 1 of column g of n-tile n (zero past the rank)
  __shared__ uint32_t ufrag[16 * KB * 32];
  for (int e = tid; e < 16 * KB * 32; e += kThreads) {
    const int ln = e & 31, n = (e >> 5) / KB, kb = (e >> 5) % KB, gg = ln >> 2, tt = ln & 3;
    const int ch = 32 * (n >> 2) + 8 * (gg >> 1) + 2 * (n & 3) + (gg & 1);
    const uint16_t *ur = c.u_r + ((int64_t)h * D + ch) * R;
    const int k = 2 * tt + 8 * kb;
    uint32_t v = 0u;
    if ((R & 1) == 0) {
      if (k < R) v = *(const uint32_t *)(ur + k);  // 4-byte aligned: R and k even
    } else {
      if (k < R) v = ur[k];
      if (k + 1 < R) v |= (uint32_t)ur[k + 1] << 16;
    }
    ufrag[e] = v;
  }
  stage_cta<false, true, IDX16, COMPACT>(c, h, tok0, p.C, st, tid);
  __syncthreads();
  const int nt = (int)((c.n - tok0) < kTok ? (c.n - tok0) : kTok);
  const uint16_t *cent = c.cent_k16 + (int64_t)h * p.C * D + 8 * t4;
  uint16_t *out = p.k_hat + ((int64_t)h * p.n_out + c.out0 + tok0) * D + 8 * t4;
  const uint32_t *codes32 = (const uint32_t *)&st.codes[0][0];
#pragma unroll 1
  for (int wt = warp; 16 * wt < nt; wt += kThreads / 32) {
    const int r0 = 16 * wt + g, r1 = r0 + 8;
    // the two tokens' centroid chunks, gathered one run of 8 channels ahead of the stores
    const uint16_t *row0 = cent + (int)st.idx[r0] * D, *row1 = cent + (int)st.idx[r1] * D;
    uint4 mu0c = *(const uint4 *)row0, mu1c = *(const uint4 *)row1;
    const uint4 cA = st.c[r0], cB = st.c[r1];
    uint32_t af[KS / 4];
    af[0] = coef_pair(cA, t4, 0);
    af[1] = coef_pair(cB, t4, 0);
    if constexpr (KS == 16) {
      af[2] = coef_pair(cA, t4, 1);
      af[3] = coef_pair(cB, t4, 1);
    }
    const uint32_t sA = st.s2[r0], mA = st.m2[r0], sB = st.s2[r1], mB = st.m2[r1];
    const float scA = st.sc[r0], scB = st.sc[r1];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      uint4 mu0n = mu0c, mu1n = mu1c;
      if (i < 3) {  // the next run's chunks, loaded before this run's stores
        mu0n = *(const uint4 *)(row0 + 32 * (i + 1));
        mu1n = *(const uint4 *)(row1 + 32 * (i + 1));
      }
      float acc[4][4];
#pragma unroll
      for (int a = 0; a < 4; a++) {
        acc[a][0] = acc[a][1] = acc[a][2] = acc[a][3] = 0.f;
        uint32_t bfr[KB];
#pragma unroll
        for (int kb = 0; kb < KB; kb++) bfr[kb] = ufrag[((4 * i + a) * KB + kb) * 32 + lane];
        mma_bf16<KS>(acc[a], af, bfr);
      }
      const int gi = i >> 1, sh = 16 * (t4 & 1);
      // the 8 codes of channels 32 i + 8 t .. + 7: halfword (t % 2) of word 2 i + t / 2 of the row
      const uint32_t bA = (codes32[8 * r0 + 2 * i + (t4 >> 1)] >> sh) & 0xFFFFu;
      const uint32_t bB = (codes32[8 * r1 + 2 * i + (t4 >> 1)] >> sh) & 0xFFFFu;
      float cr0[8], cr1[8];
#pragma unroll
      for (int u = 0; u < 8; u++) {
        cr0[u] = acc[u >> 1][u & 1];
        cr1[u] = acc[u >> 1][2 + (u & 1)];
      }
      if (r0 < nt)
        *(uint4 *)(out + (int64_t)r0 * D + 32 * i) =
            decode8<true>(mu0c, bA, f16_to_f32((uint16_t)(sA >> (16 * gi))), f16_to_f32((uint16_t)(mA >> (16 * gi))),
                          scA, cr0);
      if (r1 < nt)
        *(uint4 *)(out + (int64_t)r1 * D + 32 * i) =
            decode8<true>(mu1c, bB, f16_to_f32((uint16_t)(sB >> (16 * gi))), f16_to_f32((uint16_t)(mB >> (16 * gi))),
                          scB, cr1);
      mu0c = mu0n;
      mu1c = mu1n;
    }
  }
}

template <bool VAL, bool IDX16>
cudaError_t launch_plain(const DqParams &p, dim3 grid, bool compact, cudaStream_t st) {
  if (compact) dequant_kernel<VAL, IDX16, true><<<grid, kThreads, 0, st>>>(p);
  else dequant_kernel<VAL, IDX16, false><<<grid, kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

template <int RU, bool IDX16>
cudaError_t launch_keys(const DqParams &p, dim3 grid, bool compact, cudaStream_t st) {
  if (compact) dequant_key_kernel<RU, IDX16, true><<<grid, kThreads, 0, st>>>(p);
  else dequant_key_kernel<RU, IDX16, false><<<grid, kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

template <bool IDX16>
cudaError_t launch_idx(const DqParams &p, dim3 grid, bool compact, int rmax, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  if (p.k_hat) {
    if (rmax == 0) e = launch_plain<false, IDX16>(p, grid, compact, st);
    else if (rmax <= 8) e = launch_keys<8, IDX16>(p, grid, compact, st);
    else e = launch_keys<16, IDX16>(p, grid, compact, st);
  }
  if (e == cudaSuccess && p.v_hat) e = launch_plain<true, IDX16>(p, grid, compact, st);
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
