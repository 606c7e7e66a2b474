// Step 5: attention over the packed cache (QuantWM Chinese summary: logits L = Q K^T / sqrt(d)
// in "注意力logits与时空token选择"; PSAC logits Q K_hat_0^T + (Q U_r) C^T in "核心方法").
//   l_ij = scale * (q_i . k_hat_0_j + (q_i U_r^(chunk j)) . c_hat_j),  o_i = softmax(l_i) V_hat.
// Each CTA owns 64 Queries of one head and streams every chunk in 64-token tiles: the
// tile's Keys and Values are decoded (centroid gather + INT2 + PSAC coefficients) into
// shared memory, then logits, online softmax and the P V product run on the CUDA cores.
#include "qwm_internal.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int BQ = 64, BK = 64, LDS = D + 1, LDP = BK + 1;
constexpr int kThreads = 256;
constexpr int kMaxChunks = 128;

struct AttnChunk {
  int64_t n;
  int rank;
  const uint8_t *k_codes, *v_codes, *k_idx, *v_idx;
  const uint16_t *k_scale, *k_min, *v_scale, *v_min, *cent_k, *cent_v, *c_scale, *u_r;
  const int8_t *c;
};

struct AttnParams {
  const uint16_t *q;
  uint16_t *out;
  int64_t nq;
  int H, C, n_chunks;
  float scale;
  AttnChunk ch[kMaxChunks];
};

__global__ void __launch_bounds__(kThreads) attend_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(16) float asmem[];
  float *Qs = asmem;              // [BQ][LDS]
  float *Ks = Qs + BQ * LDS;      // [BK][LDS]
  float *Vs = Ks + BK * LDS;      // [BK][LDS]
  float *Ps = Vs + BK * LDS;      // [BQ][LDP]
  float *QU = Ps + BQ * LDP;      // [BQ][16]
  float *Cs = QU + BQ * 16;       // [BK][16]
  float *rowm = Cs + BK * 16;     // [BQ]
  float *rowl = rowm + BQ;        // [BQ]
  float *rowa = rowl + BQ;        // [BQ]
  const int h = blockIdx.y, tid = threadIdx.x;
  const int64_t q0 = (int64_t)blockIdx.x * BQ;
  const int ty = tid / 16, tx = tid % 16;
  const int G = D / QWM_GROUP;
  for (int e = tid; e < BQ * D; e += kThreads) {
    const int r = e / D, c = e % D;
    const int64_t qi = q0 + r;
    Qs[r * LDS + c] = qi < p.nq ? bf16_to_f32(p.q[((int64_t)h * p.nq + qi) * D + c]) : 0.f;
  }
  if (tid < BQ) { rowm[tid] = -INFINITY; rowl[tid] = 0.f; }
  float o[4][8];
#pragma unroll
  for (int i = 0; i < 4; i++)
#pragma unroll
    for (int j = 0; j < 8; j++) o[i][j] = 0.f;
  __syncthreads();
  for (int t = 0; t < p.n_chunks; t++) {
    const AttnChunk &ch = p.ch[t];
    const int R = ch.rank;
    // Q U_r of this chunk
    for (int e = tid; e < BQ * R; e += kThreads) {
      const int r = e / R, kk = e % R;
      float acc = 0.f;
      for (int c = 0; c < D; c++) acc = fmaf(Qs[r * LDS + c], bf16_to_f32(ch.u_r[((int64_t)h * D + c) * R + kk]), acc);
      QU[r * 16 + kk] = acc;
    }
    for (int64_t k0 = 0; k0 < ch.n; k0 += BK) {
      const int nk = (ch.n - k0 < BK) ? (int)(ch.n - k0) : BK;
      __syncthreads();
      // decode the tile: thread handles (token, 8-channel block) pairs
      for (int e = tid; e < BK * (D / 8); e += kThreads) {
        const int tok = e / (D / 8), cb = e % (D / 8), c0 = 8 * cb, g = c0 / QWM_GROUP;
        if (tok >= nk) {
#pragma unroll
          for (int u = 0; u < 8; u++) { Ks[tok * LDS + c0 + u] = 0.f; Vs[tok * LDS + c0 + u] = 0.f; }
          continue;
        }
        const int64_t row = (int64_t)h * ch.n + k0 + tok;
        for (int pass = 0; pass < 2; pass++) {
          const uint8_t *codes = pass ? ch.v_codes : ch.k_codes;
          const uint8_t *idx = pass ? ch.v_idx : ch.k_idx;
          const float s = f16_to_f32((pass ? ch.v_scale : ch.k_scale)[row * G + g]);
          const float m = f16_to_f32((pass ? ch.v_min : ch.k_min)[row * G + g]);
          const uint16_t *mu = (pass ? ch.cent_v : ch.cent_k) + ((int64_t)h * p.C + idx[row]) * D + c0;
          const uint32_t b2 = *(const uint16_t *)(codes + row * (D / 4) + 2 * cb);
          float *dst = (pass ? Vs : Ks) + tok * LDS + c0;
#pragma unroll
          for (int u = 0; u < 8; u++)
            dst[u] = __fadd_rn(bf16_to_f32(mu[u]), __fmaf_rn(s, (float)((b2 >> (2 * u)) & 3u), m));
        }
      }
      for (int e = tid; e < BK * R; e += kThreads) {
        const int tok = e / R, kk = e % R;
        float v = 0.f;
        if (tok < nk) {
          const int64_t row = (int64_t)h * ch.n + k0 + tok;
          v = f16_to_f32(ch.c_scale[row]) * (float)ch.c[row * R + kk];
        }
        Cs[tok * 16 + kk] = v;
      }
      __syncthreads();
      // logits: thread (ty, tx) -> rows 4ty..4ty+3, key columns tx + 16 j
      float s[4][4];
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) s[i][j] = 0.f;
      for (int c = 0; c < D; c++) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; i++) a[i] = Qs[(4 * ty + i) * LDS + c];
#pragma unroll
        for (int j = 0; j < 4; j++) b[j] = Ks[(tx + 16 * j) * LDS + c];
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
          for (int j = 0; j < 4; j++) s[i][j] = fmaf(a[i], b[j], s[i][j]);
      }
      for (int kk = 0; kk < R; kk++) {
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
          for (int j = 0; j < 4; j++) s[i][j] = fmaf(QU[(4 * ty + i) * 16 + kk], Cs[(tx + 16 * j) * 16 + kk], s[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const int col = tx + 16 * j;
          Ps[(4 * ty + i) * LDP + col] = col < nk ? s[i][j] * p.scale : -INFINITY;
        }
      __syncthreads();
      if (tid < BQ) {
        const float mo = rowm[tid];
        float mx = mo;
        for (int j = 0; j < BK; j++) mx = fmaxf(mx, Ps[tid * LDP + j]);
        const float alpha = (mo == -INFINITY) ? 0.f : expf(mo - mx);
        float l = rowl[tid] * alpha;
        for (int j = 0; j < BK; j++) {
          const float pj = expf(Ps[tid * LDP + j] - mx);
          Ps[tid * LDP + j] = pj;
          l += pj;
        }
        rowm[tid] = mx; rowl[tid] = l; rowa[tid] = alpha;
      }
      __syncthreads();
      // O = alpha O + P V: thread owns rows 4ty..4ty+3, columns tx + 16 j
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const float al = rowa[4 * ty + i];
#pragma unroll
        for (int j = 0; j < 8; j++) o[i][j] *= al;
      }
      for (int kt = 0; kt < nk; kt++) {
        float pv[4], vv[8];
#pragma unroll
        for (int i = 0; i < 4; i++) pv[i] = Ps[(4 * ty + i) * LDP + kt];
#pragma unroll
        for (int j = 0; j < 8; j++) vv[j] = Vs[kt * LDS + tx + 16 * j];
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
          for (int j = 0; j < 8; j++) o[i][j] = fmaf(pv[i], vv[j], o[i][j]);
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const int r = 4 * ty + i;
    const int64_t qi = q0 + r;
    if (qi >= p.nq) continue;
    const float inv = 1.f / rowl[r];
#pragma unroll
    for (int j = 0; j < 8; j++) p.out[((int64_t)h * p.nq + qi) * D + tx + 16 * j] = f32_to_bf16_rn(o[i][j] * inv);
  }
}

}  // namespace

cudaError_t launch_attend(const qwm_config &cfg, const uint16_t *q, int64_t nq, const qwm_chunk *chunks,
                          int n_chunks, float scale, uint16_t *out, int num_sms, cudaStream_t st) {
  (void)num_sms;
  if (n_chunks > kMaxChunks) return cudaErrorInvalidValue;
  AttnParams p;  // passed by value (about 15 KB of kernel parameters)
  p.q = q; p.out = out; p.nq = nq; p.H = cfg.heads; p.C = cfg.n_centroids; p.n_chunks = n_chunks; p.scale = scale;
  for (int i = 0; i < n_chunks; i++) {
    const qwm_chunk &c = chunks[i];
    AttnChunk &a = p.ch[i];
    a.n = c.n_tokens; a.rank = c.rank_eff;
    a.k_codes = c.k_codes; a.v_codes = c.v_codes; a.k_idx = c.k_idx; a.v_idx = c.v_idx;
    a.k_scale = c.k_scale; a.k_min = c.k_min; a.v_scale = c.v_scale; a.v_min = c.v_min;
    a.cent_k = c.cent_k; a.cent_v = c.cent_v; a.c_scale = c.c_scale; a.u_r = c.u_r; a.c = c.c;
  }
  const size_t smem = (size_t)(BQ * LDS + 2 * BK * LDS + BQ * LDP + BQ * 16 + BK * 16 + 3 * BQ) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  attend_kernel<<<dim3((unsigned)((nq + BQ - 1) / BQ), cfg.heads), kThreads, smem, st>>>(p);
  return cudaGetLastError();
}
