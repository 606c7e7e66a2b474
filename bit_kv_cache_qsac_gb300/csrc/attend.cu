// Step 5: attention over the packed cache on the tensor cores (tcgen05 + TMEM).
//
// QuantWM (Chinese summary, "注意力logits与时空token选择": L = Q K^T / sqrt(d); "核心方法":
// PSAC logits Q K_hat_0^T + (Q U_r) C^T; English v2 summary §D.1):
//   l_ij = scale * ([q_i | q_i U_r^(t)] . [k_hat_0_j | c_hat_j]),  o_i = softmax(l_i) V_hat,
// with k_hat_0 = mu^K_idx + m + s q, c_hat = sC c and v_hat = mu^V_idx + m + s q decoded from the
// packed chunk inside the kernel.  Nothing decoded is written back to memory.
// Operands of both MMAs are fp16 (fp32 accumulate): the decode is exact in fp32 and rounded once
// to fp16, whose 11-bit mantissa keeps the logits of the outlier channels (|k| up to ~40)
// accurate; Q (bf16 in memory) converts to fp16 exactly for every normal value.
//
// One CTA = one head x 256 Queries (two 128-row tiles that share every decoded K/V tile).
// Warp roles (512 threads):
//   warps 0-3, 4-7  softmax for Query tile 0 / 1: thread = Query row = TMEM lane; reads the
//                   logits from TMEM, keeps the running max and sum, writes P (bf16) back over
//                   the logits, rescales O in TMEM when the max grows by more than 2^8;
//   warp 8          allocates TMEM and issues every tcgen05.mma (one thread);
//   warps 9-15      producers: decode each 128-token tile of the packed cache into shared memory
//                   (K_hat_0 rows and V_hat^T rows as 128-byte-swizzled fp16, c_hat in the
//                   no-swizzle layout) and, at each chunk start, Q U_r for both Query tiles.
// Tensor memory (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each; P_x overlays S_x.
// MMA order per tile j: S0(j), PV1(j-1), S1(j), PV0(j).  tcgen05 operations complete in issue
// order, so the commit after S_x(j) also certifies PV_x(j-1): when softmax x sees S_x(j), O_x
// is stable and may be rescaled.
// O is written in fp32: the output is an average over thousands of keys, its largest entries are
// ~16x its RMS, and rounding those to bf16 alone would cost ~0.03 x RMS(O).
// Every wait is bounded (about one second of wall time); on expiry the CTA records
// QWM_ERR_DEVICE_TIMEOUT, every role stops, outstanding MMAs are drained and TMEM is freed.
#include <cuda_bf16.h>

#include "qwm_internal.cuh"
#include "tc.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int BM = 128, BN = 128, NQT = 2;
constexpr int kSoftmaxWarps = 8, kMmaWarp = 8, kProdWarp0 = 9, kProdWarps = 7;
constexpr int kThreads = 32 * (kSoftmaxWarps + 1 + kProdWarps);  // 512
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kMaxChunks = 128;
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8

// shared-memory map (bytes from a 1024-aligned base)
constexpr int kBlk = BM * 128;                    // one [128 rows][64 bf16] swizzled block: 16 KB
constexpr int OFF_Q = 0;                          // 2 tiles x 2 blocks
constexpr int OFF_K = OFF_Q + NQT * 2 * kBlk;     // 2 stages x 2 blocks (K_hat_0 rows)
constexpr int OFF_V = OFF_K + 2 * 2 * kBlk;       // 2 stages x 2 blocks (V_hat^T rows)
constexpr int OFF_C = OFF_V + 2 * 2 * kBlk;       // 2 stages x [128][16] c_hat (no swizzle)
constexpr int OFF_QU = OFF_C + 2 * 4096;          // 2 slots x 2 tiles x [128][16] Q U_r
constexpr int SMEM_BYTES = OFF_QU + 2 * NQT * 4096;
constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;

struct AttnChunk {
  int64_t n;
  int rank;
  int tiles;
  const uint8_t *k_codes, *v_codes, *k_idx, *v_idx;
  const uint16_t *k_scale, *k_min, *v_scale, *v_min, *cent_k, *cent_v, *c_scale, *u_r;
  const int8_t *c;
};

struct AttnParams {
  const uint16_t *q;
  float *out;
  int64_t nq;
  int H, C, n_chunks, total_tiles;
  float scale_log2;  // softmax_scale * log2(e)
  int32_t *status;
  AttnChunk ch[kMaxChunks];
};

struct Bars {
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_ready[2], o_done, drain;
};

__device__ __forceinline__ float half_bits_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// 2^23 + q as a float for a 2-bit code q in the low bits of c (exact), and its removal.
__device__ __forceinline__ float magic_code(uint32_t c) { return __uint_as_float((c & 3u) | 0x4B000000u); }
constexpr float kMagic = 8388608.0f;

// Decode 32 channels (quarter of a token) of a Key exactly in fp32 -- r_hat = fl(m + s q) and
// k_hat_0 = fl(mu + r_hat), as in the packing -- then round to fp16: 16 words, channel pairs.
__device__ __forceinline__ void decode_key_quarter(const uint2 codes, const uint4 (&mu)[4], float s, float m,
                                                   uint32_t (&out)[16]) {
  const uint64_t s2 = tc::f2(s, s), m2 = tc::f2(m, m), neg = tc::f2(-kMagic, -kMagic);
  const uint32_t cw[2] = {codes.x, codes.y};
#pragma unroll
  for (int hw = 0; hw < 4; hw++) {  // 8 channels per 16-bit halfword of codes
    const uint32_t h16 = cw[hw >> 1] >> (16 * (hw & 1));
    const uint32_t muw[4] = {mu[hw].x, mu[hw].y, mu[hw].z, mu[hw].w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const uint64_t q2 = tc::add2(tc::f2(magic_code(h16 >> (4 * i)), magic_code(h16 >> (4 * i + 2))), neg);
      const uint64_t r2 = tc::fma2(s2, q2, m2);
      const uint64_t k2 = tc::add2(tc::f2(__uint_as_float(muw[i] << 16), __uint_as_float(muw[i] & 0xFFFF0000u)), r2);
      out[4 * hw + i] = tc::pack_f16x2(tc::f2lo(k2), tc::f2hi(k2));
    }
  }
}

__device__ __forceinline__ void fail(int *abort_flag, int32_t *status) {
  *(volatile int *)abort_flag = 1;
  qwm_dev_error(status, QWM_ERR_DEVICE_TIMEOUT);
}

__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char *sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  const int64_t q0 = (int64_t)blockIdx.x * (BM * NQT);
  volatile int *abort_v = &abort_flag;

  // ---- Query tiles -> shared memory (zero rows past nq) ----
  for (int e = tid; e < NQT * BM * (D / 8); e += kThreads) {
    const int row = e / (D / 8), ci = e % (D / 8);  // row in [0, 256), 16-byte chunk in [0, 16)
    const int x = row / BM, rr = row % BM, b = ci / 8;
    const int64_t qi = q0 + row;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (qi < p.nq) v = *(const uint4 *)(p.q + ((int64_t)h * p.nq + qi) * D + 8 * ci);
    const uint32_t bw[4] = {v.x, v.y, v.z, v.w};
    uint32_t hw[4];
#pragma unroll
    for (int u = 0; u < 4; u++) hw[u] = tc::pack_f16x2(__uint_as_float(bw[u] << 16), __uint_as_float(bw[u] & 0xFFFF0000u));
    *(uint4 *)(sm + OFF_Q + (x * 2 + b) * kBlk + tc::sw128_offset(rr, 8 * (ci % 8))) =
        make_uint4(hw[0], hw[1], hw[2], hw[3]);
  }
  if (tid == 0) {
    for (int i = 0; i < 2; i++) {
      tc::mbar_init(&bars.k_full[i], kProdWarps);
      tc::mbar_init(&bars.v_full[i], kProdWarps);
      tc::mbar_init(&bars.k_empty[i], 1);
      tc::mbar_init(&bars.v_empty[i], 1);
      tc::mbar_init(&bars.s_full[i], 1);
      tc::mbar_init(&bars.p_ready[i], 4);
    }
    tc::mbar_init(&bars.o_done, 1);
    tc::mbar_init(&bars.drain, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&tmem_base_sh, 512);
    tc::tmem_relinquish();
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const int J = p.total_tiles;

  if (warp < kSoftmaxWarps) {
    // ======================= softmax (Query tile x, row = TMEM lane) =======================
    const int x = warp / 4, sub = warp % 4, row = 32 * sub + lane;
    const uint32_t lane_addr = (uint32_t)(32 * sub) << 16;
    const uint32_t tS = tmem + lane_addr + 128u * x, tO = tmem + lane_addr + 256u + 128u * x;
    float m_used = -INFINITY, l = 0.f;
    int t = 0, tile_in_chunk = 0;
    bool ok = true;
    for (int j = 0; j < J; j++) {
      const AttnChunk &ch = p.ch[t];
      const int64_t left = ch.n - (int64_t)tile_in_chunk * BN;
      const int nk = left < BN ? (int)left : BN;
      if (!tc::mbar_wait(&bars.s_full[x], j & 1, kWaitNs)) fail(&abort_flag, p.status);
      if (*abort_v) { ok = false; break; }
      tc::fence_after_sync();
      uint32_t r[32];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN; c += 32) {
        tc::tmem_ld32(tS + c, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; i++)
          if (c + i < nk) mx = fmaxf(mx, __uint_as_float(r[i]));
      }
      const float m_new = fmaxf(m_used, mx * p.scale_log2);
      const bool need = (j == 0) || (m_new > m_used + kRescaleThreshold);
      if (__any_sync(0xffffffffu, need)) {
        if (j > 0) {
          const float alpha = tc::ex2_approx(m_used - m_new);
          l *= alpha;
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            tc::tmem_ld32(tO + c, r);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; i++) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tc::tmem_st32(tO + c, r);
          }
        }
        m_used = m_new;
      }
#pragma unroll
      for (int c = 0; c < BN; c += 32) {
        tc::tmem_ld32(tS + c, r);
        tc::tmem_ld_wait();
        uint32_t pw[16];
#pragma unroll
        for (int i = 0; i < 16; i++) {
          const float x0 = (c + 2 * i < nk) ? tc::ex2_approx(__uint_as_float(r[2 * i]) * p.scale_log2 - m_used) : 0.f;
          const float x1 =
              (c + 2 * i + 1 < nk) ? tc::ex2_approx(__uint_as_float(r[2 * i + 1]) * p.scale_log2 - m_used) : 0.f;
          l += x0 + x1;
          pw[i] = tc::pack_f16x2(x0, x1);
        }
        tc::tmem_st16(tS + c / 2, pw);  // P overlays the first 64 columns of S
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars.p_ready[x]);
      if (++tile_in_chunk == ch.tiles) { tile_in_chunk = 0; t++; }
    }
    // ---- epilogue: O / l -> bf16 ----
    if (ok && !tc::mbar_wait(&bars.o_done, 0, kWaitNs)) fail(&abort_flag, p.status);
    if (ok && !*abort_v) {
      tc::fence_after_sync();
      const int64_t qi = q0 + (int64_t)x * BM + row;
      const float inv = 1.f / l;
      uint32_t r[32];
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        tc::tmem_ld32(tO + c, r);
        tc::tmem_ld_wait();
        if (qi < p.nq) {
          float4 *dst = (float4 *)(p.out + ((int64_t)h * p.nq + qi) * D + c);
#pragma unroll
          for (int v = 0; v < 8; v++)
            dst[v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                 __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ======================= MMA issue (one thread) =======================
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16_f32(BM, BN);
      const uint32_t tS[2] = {tmem, tmem + 128u}, tO[2] = {tmem + 256u, tmem + 384u};
      const uint32_t sQ = tc::smem_u32(sm + OFF_Q), sK = tc::smem_u32(sm + OFF_K), sV = tc::smem_u32(sm + OFF_V);
      const uint32_t sC = tc::smem_u32(sm + OFF_C), sQU = tc::smem_u32(sm + OFF_QU);
      int t = 0, tile_in_chunk = 0, prev_stage = 0;
      bool ok = true;
      auto qk = [&](int x, int s, int slot, int rank) {
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
          const uint32_t off = (uint32_t)((kk / 4) * kBlk + 32 * (kk % 4));
          tc::mma_ss(tS[x], tc::desc_sw128(sQ + (x * 2) * kBlk + off), tc::desc_sw128(sK + (s * 2) * kBlk + off),
                     idesc, kk > 0);
        }
        if (rank > 0)
          tc::mma_ss(tS[x], tc::desc_noswz(sQU + (slot * NQT + x) * 4096, 128, 256),
                     tc::desc_noswz(sC + s * 4096, 128, 256), idesc, 1);
      };
      auto pv = [&](int x, int s, bool first) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; kk++) {
          const uint32_t off = (uint32_t)((kk / 4) * kBlk + 32 * (kk % 4));
          tc::mma_ts(tO[x], tS[x] + 8u * kk, tc::desc_sw128(sV + (s * 2) * kBlk + off), idesc, (!first || kk > 0));
        }
      };
      for (int j = 0; j < J; j++) {
        const int s = j & 1;
        const AttnChunk &ch = p.ch[t];
        ok = tc::mbar_wait(&bars.k_full[s], (j >> 1) & 1, kWaitNs) && !*abort_v;
        if (!ok) break;
        tc::fence_after_sync();
        qk(0, s, t & 1, ch.rank);
        tc::mma_commit(&bars.s_full[0]);
        if (j > 0) {
          ok = tc::mbar_wait(&bars.p_ready[1], (j - 1) & 1, kWaitNs) && !*abort_v;
          if (!ok) break;
          tc::fence_after_sync();
          pv(1, prev_stage, j - 1 == 0);
          tc::mma_commit(&bars.v_empty[prev_stage]);
        }
        qk(1, s, t & 1, ch.rank);
        tc::mma_commit(&bars.s_full[1]);
        tc::mma_commit(&bars.k_empty[s]);
        ok = tc::mbar_wait(&bars.v_full[s], (j >> 1) & 1, kWaitNs) && tc::mbar_wait(&bars.p_ready[0], j & 1, kWaitNs) &&
             !*abort_v;
        if (!ok) break;
        tc::fence_after_sync();
        pv(0, s, j == 0);
        prev_stage = s;
        if (++tile_in_chunk == ch.tiles) { tile_in_chunk = 0; t++; }
      }
      if (ok && J > 0) {
        ok = tc::mbar_wait(&bars.p_ready[1], (J - 1) & 1, kWaitNs) && !*abort_v;
        if (ok) {
          tc::fence_after_sync();
          pv(1, prev_stage, J - 1 == 0);
          tc::mma_commit(&bars.o_done);
        }
      }
      if (!ok) fail(&abort_flag, p.status);
      // drain: every MMA issued above completes before TMEM is released
      tc::mma_commit(&bars.drain);
      if (!tc::mbar_wait(&bars.drain, 0, kWaitNs)) qwm_dev_error(p.status, QWM_ERR_DEVICE_TIMEOUT);
    }
  } else {
    // ======================= producers: decode tiles of the packed cache =======================
    const int pt = tid - 32 * kProdWarp0;  // 0..223
    int t = 0, tile_in_chunk = 0;
    for (int j = 0; j < J; j++) {
      const int s = j & 1;
      const AttnChunk &ch = p.ch[t];
      const int64_t k0 = (int64_t)tile_in_chunk * BN;
      const int64_t left = ch.n - k0;
      const int nk = left < BN ? (int)left : BN;
      const int R = ch.rank;
      if (j >= 2 && !tc::mbar_wait(&bars.k_empty[s], ((j >> 1) - 1) & 1, kWaitNs)) fail(&abort_flag, p.status);
      if (*abort_v) break;
      // --- Q U_r of this chunk, for both Query tiles (first tile of the chunk only) ---
      if (tile_in_chunk == 0 && R > 0) {
        const uint16_t *U = ch.u_r + (int64_t)h * D * R;
        for (int row = pt; row < NQT * BM; row += kProdThreads) {
          const int x = row / BM, rr = row % BM;
          float acc[16];
#pragma unroll
          for (int kq = 0; kq < 16; kq++) acc[kq] = 0.f;
          const int64_t qi = q0 + row;
          for (int ci = 0; ci < D / 8; ci++) {
            uint4 qv = make_uint4(0, 0, 0, 0);
            if (qi < p.nq) qv = *(const uint4 *)(p.q + ((int64_t)h * p.nq + qi) * D + 8 * ci);
            const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
            for (int u = 0; u < 8; u++) {
              const float qc = __uint_as_float((u & 1) ? (qw[u / 2] & 0xFFFF0000u) : (qw[u / 2] << 16));
              const uint16_t *Uc = U + (8 * ci + u) * R;
#pragma unroll
              for (int kq = 0; kq < 16; kq++)
                if (kq < R) acc[kq] = fmaf(qc, bf16_to_f32(Uc[kq]), acc[kq]);
            }
          }
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; i++) w[i] = tc::pack_f16x2(acc[2 * i], acc[2 * i + 1]);
          unsigned char *dst = sm + OFF_QU + ((t & 1) * NQT + x) * 4096;
          *(uint4 *)(dst + tc::noswz16_offset(rr, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
          *(uint4 *)(dst + tc::noswz16_offset(rr, 8)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
      // --- K_hat_0 rows: item = (token row, quarter of 32 channels), up to 3 per thread.  All
      // index loads are issued first, then all centroid gathers, then the decode, so that each
      // thread has its loads in flight together instead of one dependent chain per item. ---
      {
        constexpr int kItems = (BN * 4 + kProdThreads - 1) / kProdThreads;  // 3
        int idx[kItems];
        float sc[kItems], mn[kItems];
        uint2 cd[kItems];
        bool ok[kItems];
#pragma unroll
        for (int i = 0; i < kItems; i++) {
          const int it = pt + i * kProdThreads, row = it >> 2, qd = it & 3;
          ok[i] = it < BN * 4 && row < nk;
          idx[i] = 0; sc[i] = 0.f; mn[i] = 0.f; cd[i] = make_uint2(0, 0);
          if (ok[i]) {
            const int64_t gi = (int64_t)h * ch.n + k0 + row;
            idx[i] = min((int)ch.k_idx[gi], p.C - 1);  // never read past the codebook
            sc[i] = half_bits_to_f32(ch.k_scale[gi * 2 + (qd >> 1)]);
            mn[i] = half_bits_to_f32(ch.k_min[gi * 2 + (qd >> 1)]);
            cd[i] = *(const uint2 *)(ch.k_codes + gi * (D / 4) + 8 * qd);
          }
        }
        uint4 muv[kItems][4];
#pragma unroll
        for (int i = 0; i < kItems; i++) {
          const int qd = (pt + i * kProdThreads) & 3;
          const uint4 *mu = (const uint4 *)(ch.cent_k + ((int64_t)h * p.C + idx[i]) * D + 32 * qd);
#pragma unroll
          for (int v = 0; v < 4; v++) muv[i][v] = ok[i] ? mu[v] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kItems; i++) {
          const int it = pt + i * kProdThreads, row = it >> 2, qd = it & 3;
          if (it >= BN * 4) continue;
          uint32_t w[16];
          if (ok[i]) {
            decode_key_quarter(cd[i], muv[i], sc[i], mn[i], w);
          } else {
#pragma unroll
            for (int u = 0; u < 16; u++) w[u] = 0u;
          }
          unsigned char *blk = sm + OFF_K + (s * 2 + (qd >> 1)) * kBlk;
#pragma unroll
          for (int v = 0; v < 4; v++)
            *(uint4 *)(blk + tc::sw128_offset(row, 32 * (qd & 1) + 8 * v)) =
                make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
      }
      // --- c_hat rows (PSAC coefficients, fp16, zero past the rank) ---
      if (R > 0) {
        for (int row = pt; row < BN; row += kProdThreads) {
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; i++) w[i] = 0u;
          if (row < nk) {
            const int64_t gi = (int64_t)h * ch.n + k0 + row;
            const float sc = half_bits_to_f32(ch.c_scale[gi]);
            const int8_t *cc = ch.c + gi * R;
#pragma unroll
            for (int i = 0; i < 8; i++) {
              const float a = (2 * i < R) ? sc * (float)cc[2 * i] : 0.f;
              const float bq = (2 * i + 1 < R) ? sc * (float)cc[2 * i + 1] : 0.f;
              w[i] = tc::pack_f16x2(a, bq);
            }
          }
          unsigned char *dst = sm + OFF_C + s * 4096;
          *(uint4 *)(dst + tc::noswz16_offset(row, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
          *(uint4 *)(dst + tc::noswz16_offset(row, 8)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars.k_full[s]);
      // --- V_hat^T rows: item = (token pair, quarter of 32 channels) ---
      if (j >= 2 && !tc::mbar_wait(&bars.v_empty[s], ((j >> 1) - 1) & 1, kWaitNs)) fail(&abort_flag, p.status);
      if (*abort_v) break;
      for (int it = pt; it < (BN / 2) * 4; it += kProdThreads) {
        const int pair = it >> 2, qd = it & 3, g = qd >> 1;
        uint2 codes[2] = {make_uint2(0, 0), make_uint2(0, 0)};
        uint4 muv[2][4];
        float sv[2] = {0.f, 0.f}, mv[2] = {0.f, 0.f};
#pragma unroll
        for (int u = 0; u < 2; u++) {
          const int row = 2 * pair + u;
          if (row < nk) {
            const int64_t gi = (int64_t)h * ch.n + k0 + row;
            const int idx = min((int)ch.v_idx[gi], p.C - 1);
            sv[u] = half_bits_to_f32(ch.v_scale[gi * 2 + g]);
            mv[u] = half_bits_to_f32(ch.v_min[gi * 2 + g]);
            codes[u] = *(const uint2 *)(ch.v_codes + gi * (D / 4) + 8 * qd);
            const uint4 *mu = (const uint4 *)(ch.cent_v + ((int64_t)h * p.C + idx) * D + 32 * qd);
#pragma unroll
            for (int v = 0; v < 4; v++) muv[u][v] = mu[v];
          } else {
#pragma unroll
            for (int v = 0; v < 4; v++) muv[u][v] = make_uint4(0, 0, 0, 0);
          }
        }
        const bool valid0 = (2 * pair) < nk, valid1 = (2 * pair + 1) < nk;
        const uint64_t s2 = tc::f2(sv[0], sv[1]), m2 = tc::f2(mv[0], mv[1]), neg = tc::f2(-kMagic, -kMagic);
        const uint32_t cw0[2] = {codes[0].x, codes[0].y}, cw1[2] = {codes[1].x, codes[1].y};
        const int key = 2 * pair, vb = key / 64, kin = key % 64;
        unsigned char *blk = sm + OFF_V + (s * 2 + vb) * kBlk;
#pragma unroll
        for (int hw = 0; hw < 4; hw++) {  // 8 channels each
          const uint32_t a16 = cw0[hw >> 1] >> (16 * (hw & 1));
          const uint32_t b16 = cw1[hw >> 1] >> (16 * (hw & 1));
          const uint32_t mu0[4] = {muv[0][hw].x, muv[0][hw].y, muv[0][hw].z, muv[0][hw].w};
          const uint32_t mu1[4] = {muv[1][hw].x, muv[1][hw].y, muv[1][hw].z, muv[1][hw].w};
#pragma unroll
          for (int u = 0; u < 8; u++) {
            const int c = 32 * qd + 8 * hw + u;  // channel = V_hat^T row
            const uint64_t q2 = tc::add2(tc::f2(magic_code(a16 >> (2 * u)), magic_code(b16 >> (2 * u))), neg);
            const uint64_t r2 = tc::fma2(s2, q2, m2);
            const float mua = __uint_as_float((u & 1) ? (mu0[u >> 1] & 0xFFFF0000u) : (mu0[u >> 1] << 16));
            const float mub = __uint_as_float((u & 1) ? (mu1[u >> 1] & 0xFFFF0000u) : (mu1[u >> 1] << 16));
            const uint64_t v2 = tc::add2(tc::f2(mua, mub), r2);
            uint32_t vw = tc::pack_f16x2(tc::f2lo(v2), tc::f2hi(v2));
            if (!valid1) vw &= 0x0000FFFFu;
            if (!valid0) vw = 0u;
            *(uint32_t *)(blk + tc::sw128_offset(c, kin)) = vw;
          }
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars.v_full[s]);
      if (++tile_in_chunk == ch.tiles) { tile_in_chunk = 0; t++; }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_attend(const qwm_config &cfg, const uint16_t *q, int64_t nq, const qwm_chunk *chunks,
                          int n_chunks, float scale, float *out, int num_sms, int32_t *status, cudaStream_t st) {
  (void)num_sms;
  AttnParams p;  // passed by value (about 17 KB of kernel parameters)
  p.q = q; p.out = out; p.nq = nq; p.H = cfg.heads; p.C = cfg.n_centroids;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  int used = 0, tiles = 0;
  for (int i = 0; i < n_chunks; i++) {
    const qwm_chunk &c = chunks[i];
    if (c.n_tokens == 0) continue;  // empty chunks contribute nothing
    if (used == kMaxChunks) return cudaErrorInvalidValue;
    AttnChunk &a = p.ch[used++];
    a.n = c.n_tokens; a.rank = c.rank_eff; a.tiles = (int)((c.n_tokens + BN - 1) / BN);
    a.k_codes = c.k_codes; a.v_codes = c.v_codes; a.k_idx = c.k_idx; a.v_idx = c.v_idx;
    a.k_scale = c.k_scale; a.k_min = c.k_min; a.v_scale = c.v_scale; a.v_min = c.v_min;
    a.cent_k = c.cent_k; a.cent_v = c.cent_v; a.c_scale = c.c_scale; a.u_r = c.u_r; a.c = c.c;
    tiles += a.tiles;
  }
  p.n_chunks = used;
  p.total_tiles = tiles;
  cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  attend_tc_kernel<<<dim3((unsigned)((nq + BM * NQT - 1) / (BM * NQT)), cfg.heads), kThreads, SMEM_ALLOC, st>>>(p);
  return cudaGetLastError();
}
