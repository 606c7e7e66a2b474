// Step 5: attention over the packed cache on the tensor cores (tcgen05 + TMEM).
//
// QuantWM (Chinese summary, "注意力logits与时空token选择": L = Q K^T / sqrt(d); "核心方法":
// PSAC logits Q K_hat_0^T + (Q U_r) C^T; English v2 summary §D.1):
//   l_ij = scale * (q_i . k_hat_0_j + (q_i U_r) . c_hat_j),  o_i = softmax(l_i) V_hat,
// with k_hat_0 = mu^K_idx + m + s q, c_hat = sC c and v_hat = mu^V_idx + m + s q decoded from the
// packed chunk inside the kernel.  Nothing decoded is written to global memory.
//
// Arithmetic.  Both MMAs take fp16 operands (fp32 accumulate): fp16's 11-bit significand keeps the
// logits of the outlier channels (|k| up to ~40) accurate where bf16 would not.  Q (bf16 in memory)
// converts to fp16 exactly for magnitudes in [2^-24, 65504] (an element beyond 65504 records
// QWM_ERR_RANGE; smaller ones round to fp16's subnormal grid, far below any logit's rounding).  A Key
// or Value row is decoded in packed fp16 pairs from the chunk's fp16 codebook row as
// fp16(mu + fp16(m + s q_code)): the small residual first, as in the packing, then the centroid (two
// roundings, both at the scale of their results).  The PSAC term rides on a
// small second MMA whose K columns are [q U_r | 0 | 1] against [c_hat | 0 | mask], where mask = -inf
// (fp16) on the zero rows that pad the last tile of a chunk and 0 elsewhere: their logits are -inf
// whatever the softmax scale and their weights exactly 0.
// O is written in fp32: the output is an average over thousands of keys, its largest entries are
// ~16x its RMS, and rounding those to bf16 alone would cost ~0.03 x RMS(O).
// The chunk still being generated (English v2 summary §5.1, §D.1: a chunk is quantised once it is
// complete) may join the call as a bf16 chunk: its producers copy the rows themselves and convert
// them to fp16 in place instead of decoding (an element beyond the fp16 range records
// QWM_ERR_RANGE), its second-MMA operands carry only the padding mask, and an optional block-causal
// mask (frames of tpf tokens; Query row i = token i of that chunk) is applied by the softmax, which
// sets the logits of later frames to -inf.  Chunks with the compact INT2 metadata (8-bit step s8, 2-bit zero-point z,
// power-of-two second-level scale sigma per 128-token tile) decode with s = sigma s8 and m = -z s,
// exact in fp16, through the same fp16(mu + fp16(m + s q)).  Chunks whose PSAC coefficients are in
// the per-head layout (each head its own rank, rows for every token or only for the kept ones) have
// each Key row's coefficients looked up through the head's entry and, for a sparse head, the tile
// bitmap.  Calls with none of these run a variant compiled without any of it.
//
// Work split: a pair of CTAs (a cluster of two, cta_group::2 MMAs) takes one head x 512 Queries;
// CTA c of the pair holds Query rows 256 x + 128 c .. 256 x + 128 c + 127 of its two tiles x = 0, 1.
// One M = 256 MMA covers both CTAs' rows of a tile.  Its B operand is split by N, so CTA c decodes
// only Key rows 64 c .. 64 c + 63 of each 128-key tile (all channels) for Q K_hat^T, and only
// channels 64 c .. 64 c + 63 (INT2 group c) of all 128 Value rows for P V_hat: each CTA decodes half
// of every tile for its 256 Queries.
// Warp roles of each CTA (17 warps):
//   warps 0-3, 4-7  softmax for Query tile 0 / 1: thread = Query row = TMEM lane; reads the
//                   logits from TMEM, keeps the running max and sum, writes P (fp16) over the
//                   logits, rescales O in TMEM when the max grows by more than 2^8;
//   warp 8          allocates the pair's TMEM; in the even CTA, one thread issues every MMA of the
//                   pair;
//   warps 9-12      Key producers: thread = (channel group, key row); copies that half row of the
//                   row's centroid (cp.async, 16 bytes at a time) into the 128-byte-swizzled K-major
//                   stage, decodes it in place; group-0 threads write the row of the second MMA's B
//                   operand; at each chunk start every thread builds one row of its A operand for
//                   both Query tiles;
//   warps 13-16     Value producers: thread = key row, channel group c ([key][d], read as an
//                   MN-major B).
// Each producer thread keeps its row's index data two tiles ahead in registers and its centroid
// copies one tile ahead in the next of three shared-memory stages.
// The odd CTA's producers and softmax warps arrive on the even CTA's barriers through
// shared::cluster addresses; the MMA commits reach both CTAs' barriers by multicast.
// Tensor memory (512 columns in each CTA): S0 | S1 | O0 | O1, 128 fp32 columns each; P_x overlays
// S_x.  MMA order per tile j: S0(j), PV1(j-1), S1(j), PV0(j).  tcgen05 operations complete in
// issue order, so the commit after S_x(j) also certifies PV_x(j-1): when softmax x sees S_x(j),
// O_x is stable and may be rescaled.
// Every wait is bounded (about one second of wall time); on expiry the CTA records
// QWM_ERR_DEVICE_TIMEOUT, every role stops, outstanding MMAs are drained, the pair meets at a
// cluster barrier and TMEM is freed.
#include <cuda_fp16.h>

#include "qwm_internal.cuh"
#include "tc.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int BM = 128, BN = 128, NQT = 2;
constexpr int kSoftmaxWarps = 8, kMmaWarp = 8, kKWarp0 = 9, kVWarp0 = 13, kProdWarps = 4;
constexpr int kThreads = 32 * (kSoftmaxWarps + 1 + 2 * kProdWarps);  // 544
constexpr int kMaxChunks = 128;
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint64_t kTestWaitNs = 1000000ull;  // the test hook's wait limit
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8
constexpr uint32_t kMaskBits = 0xFC00u;    // fp16 -inf: the logit of a row that pads a chunk's last tile

constexpr int kStages = 3;                 // K / V / X stages in shared memory
constexpr int kPairQ = 2 * NQT * BM;       // Queries per CTA pair

// shared-memory map of one CTA (bytes from a 1024-aligned base)
constexpr int kBlk = BM * 128;             // a [128 rows][64 fp16] swizzled block: 16 KB
constexpr int kBlkH = 64 * 128;            // a [64 rows][64 fp16] swizzled block: 8 KB
constexpr int OFF_Q = 0;                   // 2 Query tiles x 2 blocks (channels 0-63, 64-127)
constexpr int OFF_K = OFF_Q + NQT * 2 * kBlk;          // stages x 2 blocks [64 keys][64 ch]
constexpr int OFF_V = OFF_K + kStages * 2 * kBlkH;     // stages x [128 keys][64 ch] (MN-major B)
constexpr int OFF_X = OFF_V + kStages * kBlk;          // stages of X [64][cols], then 2 QX [128][cols]

// Layout of the second MMA's operands, X = [c_hat | 0 | mask] rows of keys and QX = [q U_r | 0 | 1]
// rows of Queries: [rows][16 or 32 fp16 columns], K-major without swizzle (8x8 core matrices, 128
// bytes apart along K and 16 x columns bytes apart along the rows).  The narrow form (every chunk
// of the call has PSAC rank <= 8) leaves room for a byte-indexed code table; the wide form serves
// ranks up to 16.
template <bool WIDE>
struct XL {
  static constexpr int kCols = WIDE ? 32 : 16;
  static constexpr uint32_t kSbo = 16u * kCols;
  static constexpr int kXBytes = 64 * kCols * 2;    // one X stage: this CTA's 64 key rows
  static constexpr int kQXBytes = 128 * kCols * 2;  // one QX tile: this CTA's 128 Query rows
  static constexpr int kOffQX = OFF_X + kStages * kXBytes;  // 2 buffers (alternate chunks) x NQT tiles
  static constexpr int kUBytes = 128 * (WIDE ? 16 : 8) * 4;  // U_r of one chunk as fp32 [128][kRU]
  static constexpr int kOffU = kOffQX + 2 * NQT * kQXBytes;  // 2 buffers (alternate chunks)
  static constexpr int kSmemBytes = kOffU + 2 * kUBytes;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  __host__ __device__ static constexpr uint32_t off(uint32_t row, uint32_t k) {
    return (row >> 3) * kSbo + (k >> 3) * 128u + (row & 7u) * 16u + (k & 7u) * 2u;
  }
};

struct AttnChunk {
  int64_t n;
  int rank;
  int tiles;
  int raw;              // the chunk being generated: bf16 rows k_raw / v_raw instead of packed data
  int64_t tpf;          // raw only: > 0 = block-causal mask over frames of tpf tokens
  const uint16_t *k_raw, *v_raw;
  const uint8_t *k_s8, *v_s8, *k_zp, *v_zp;  // compact metadata (steps, zero-points)
  const uint16_t *k_sigma, *v_sigma;         // compact second-level scales [H][tiles][2]
  const uint8_t *k_codes, *v_codes, *k_idx, *v_idx;
  const uint16_t *k_scale, *k_min, *v_scale, *v_min, *cent_k16, *cent_v16, *c_scale, *u_r;
  const int8_t *c;
  int per_head;                       // QWM_C_PER_HEAD coefficients (c_heads, c_mask, c_tile_rank)
  const qwm_psac_head *c_heads;
  const uint32_t *c_mask;
  const int32_t *c_tile_rank;
};

struct AttnParams {
  const uint16_t *q;
  float *out;
  float *lse;        // [H][nq] log2-sum-exp of the scaled logits, or NULL
  int merge;         // 1: out and lse hold a result over other keys; merge this call's into them
  int64_t nq;
  int H, C, n_chunks, total_tiles;
  int compact;       // the chunks' INT2 metadata is the compact form (8-bit step, 2-bit zero-point)
  int any_causal;    // a bf16 chunk with a block-causal mask
  float scale_log2;  // softmax_scale * log2(e)
  int test_expire;   // QWM_TEST_EXPIRE_WAIT: the MMA thread's wait before its first tile runs out
  int32_t *status;
  AttnChunk ch[kMaxChunks];
};

struct Bars {
  uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], p_ready[2], qx_full[2], qx_free[2], u_ready[2], o_done, drain;
  uint64_t never;  // test hook: a barrier nothing completes
};

__device__ __forceinline__ void fail(int *abort_flag, int32_t *status) {
  *(volatile int *)abort_flag = 1;
  qwm_dev_error(status, QWM_ERR_DEVICE_TIMEOUT);
}
__device__ __forceinline__ uint32_t f16pair(float lo, float hi) { return tc::pack_f16x2(lo, hi); }
// two 32-bit registers as one 64-bit operand of the packed fp32 instructions
__device__ __forceinline__ uint64_t pk64(uint32_t lo, uint32_t hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}

// This thread's row of the second MMA's B operand: [c_hat (8 or 16) | 0 0 0 0 | mask | 0 ...].
template <bool WIDE, typename Row>
__device__ __forceinline__ void write_x_row(const Row &d, int R, uint32_t xs, int r) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; i++) w[i] = 0u;
  const float sc = __half2float(__ushort_as_half((uint16_t)d.csc));
  const uint32_t cwd[4] = {d.ca.x, d.ca.y, d.cb.x, d.cb.y};
  const uint32_t mask = d.idx >= 0 ? 0u : kMaskBits;
  if (R <= 8) {
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const uint32_t cv = cwd[i >> 1] >> (16 * (i & 1));
      w[i] = f16pair(sc * (float)(int8_t)(cv & 0xFFu), sc * (float)(int8_t)(cv >> 8));
    }
    w[6] = mask;
  } else {
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const uint32_t cv = cwd[i >> 1] >> (16 * (i & 1));
      w[i] = f16pair(sc * (float)(int8_t)(cv & 0xFFu), sc * (float)(int8_t)(cv >> 8));
    }
    w[10] = mask;
  }
#pragma unroll
  for (int kc = 0; kc < XL<WIDE>::kCols / 8; kc++)
    tc::sts128(xs + XL<WIDE>::off((uint32_t)r, 8u * kc),
               make_uint4(w[4 * kc], w[4 * kc + 1], w[4 * kc + 2], w[4 * kc + 3]));
}

// Query row rr of a Query tile: its row of the second MMA's A operand, [q U_r | 0 0 0 0 | 1 | 0 ...],
// with q read from the tile's fp16 copy in shared memory and U_r from its fp32 copy in shared memory ([128 channels][kRU], zero past the rank;
// every lane reads the same words, so the reads broadcast).
template <bool WIDE>
__device__ __forceinline__ void write_qx_row(int R, bool live, uint32_t qtile, uint32_t ubuf, uint32_t dst, int rr) {
  constexpr int kRU = WIDE ? 16 : 8;
  float acc[kRU];
#pragma unroll
  for (int k = 0; k < kRU; k++) acc[k] = 0.f;
  if (live && R > 0) {
#pragma unroll 2
    for (int ci = 0; ci < D / 8; ci++) {
      const uint4 qv = tc::lds128(qtile + (uint32_t)(ci / 8) * kBlk + tc::sw128_offset(rr, 8 * (ci % 8)));
      const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const float qc = __half2float(__ushort_as_half((uint16_t)(qw[u >> 1] >> (16 * (u & 1)))));
        const uint32_t ua = ubuf + (uint32_t)(8 * ci + u) * (kRU * 4);
#pragma unroll
        for (int k4 = 0; k4 < kRU / 4; k4++) {
          const uint4 uv = tc::lds128(ua + 16u * k4);
          acc[4 * k4] = fmaf(qc, __uint_as_float(uv.x), acc[4 * k4]);
          acc[4 * k4 + 1] = fmaf(qc, __uint_as_float(uv.y), acc[4 * k4 + 1]);
          acc[4 * k4 + 2] = fmaf(qc, __uint_as_float(uv.z), acc[4 * k4 + 2]);
          acc[4 * k4 + 3] = fmaf(qc, __uint_as_float(uv.w), acc[4 * k4 + 3]);
        }
      }
    }
  }
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; i++) w[i] = 0u;
  const uint32_t one = 0x3C00u;  // also on the zero rows past nq: their logits stay finite (0 or -inf)
  if (R <= 8) {
#pragma unroll
    for (int i = 0; i < 4; i++) w[i] = f16pair(acc[2 * i], acc[2 * i + 1]);
    w[6] = one;
  } else {
#pragma unroll
    for (int i = 0; i < kRU / 2; i++) w[i] = f16pair(acc[2 * i], acc[(2 * i + 1) % kRU]);
    w[10] = one;
  }
#pragma unroll
  for (int kc = 0; kc < XL<WIDE>::kCols / 8; kc++)
    tc::sts128(dst + XL<WIDE>::off((uint32_t)rr, 8u * kc),
               make_uint4(w[4 * kc], w[4 * kc + 1], w[4 * kc + 2], w[4 * kc + 3]));
}

// Index data of one half row: one INT2 group's fp16 step and offset (each duplicated into a pair),
// its 64 codes, and (Keys, group 0 only) the PSAC coefficients and their scale.
struct HalfRow {
  int idx;  // centroid, or -1 for a row past the end of the chunk
  uint32_t s2, m2;
  uint4 c;
  uint2 ca, cb;
  uint32_t csc;
};

template <bool VAL, bool IDX16, bool EXT>
__device__ __forceinline__ void load_half(const AttnChunk &c, int h, int64_t k0, int nk, int r, int g, bool coef,
                                          bool compact, HalfRow &d) {
  d.idx = -1;
  d.s2 = d.m2 = d.csc = 0u;
  d.c = make_uint4(0, 0, 0, 0);
  d.ca = d.cb = make_uint2(0, 0);
  if (r >= nk) return;
  if (EXT && c.raw) {  // the row of the chunk itself (a bf16 row: nothing to decode)
    d.idx = (int)(k0 + r);
    return;
  }
  const int64_t gi = (int64_t)h * c.n + k0 + r;
  const uint8_t *ip = VAL ? c.v_idx : c.k_idx;
  d.idx = IDX16 ? (int)((const uint16_t *)ip)[gi] : (int)ip[gi];  // clamped where used
  if (EXT && compact) {  // s = sigma s8 and m = -z s, both exact in fp16
    const float sg = f16_to_f32((VAL ? c.v_sigma : c.k_sigma)[((int64_t)h * c.tiles + k0 / BN) * 2 + g]);
    const float st = sg * (float)(VAL ? c.v_s8 : c.k_s8)[gi * 2 + g];
    const float z = (float)(((VAL ? c.v_zp : c.k_zp)[gi] >> (2 * g)) & 3u);
    const uint32_t sv = __half_as_ushort(__float2half_rn(st)), mv = __half_as_ushort(__float2half_rn(-z * st));
    d.s2 = sv | (sv << 16);
    d.m2 = mv | (mv << 16);
  } else {
    const uint32_t sv = (VAL ? c.v_scale : c.k_scale)[gi * 2 + g];
    const uint32_t mv = (VAL ? c.v_min : c.k_min)[gi * 2 + g];
    d.s2 = sv | (sv << 16);
    d.m2 = mv | (mv << 16);
  }
  d.c = ((const uint4 *)((VAL ? c.v_codes : c.k_codes) + gi * (D / 4)))[g];
  if (EXT && !VAL && coef && c.rank > 0 && c.per_head) {  // the head's own rank and layout
    const qwm_psac_head hd = c.c_heads[h];
    int64_t row;
    if (psac_row(hd, c.c_mask, c.c_tile_rank, c.tiles, h, k0 + r, row)) {
      const int8_t *src = c.c + hd.c_off + row * hd.rank;
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int k = 0; k < 16; k++)
        if (k < hd.rank) w[k >> 2] |= ((uint32_t)(uint8_t)src[k]) << (8 * (k & 3));
      d.ca = make_uint2(w[0], w[1]);
      d.cb = make_uint2(w[2], w[3]);
      d.csc = c.c_scale[hd.s_off + row];
    }
  } else if (!VAL && coef && c.rank > 0) {
    const int R = c.rank;
    const int8_t *src = c.c + gi * R;
    if (R == 8) {
      d.ca = *(const uint2 *)src;
    } else if (R == 16) {
      const uint4 v = *(const uint4 *)src;
      d.ca = make_uint2(v.x, v.y);
      d.cb = make_uint2(v.z, v.w);
    } else {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int k = 0; k < 16; k++)
        if (k < R) w[k >> 2] |= ((uint32_t)(uint8_t)src[k]) << (8 * (k & 3));
      d.ca = make_uint2(w[0], w[1]);
      d.cb = make_uint2(w[2], w[3]);
    }
    d.csc = c.c_scale[gi];
  }
}

// Half rows (64 channels from channel ch0) of this warp's 32 tile rows rbase .. rbase + 31 -> a
// [rows][64] swizzled block: row `idx` (the lane's; < 0: zeros) of `base`, a [rows][d] fp16 or bf16
// array of `nrows` rows (a codebook, or the bf16 chunk itself).  Each copy instruction moves four
// half rows (8 lanes each).
__device__ __forceinline__ void issue_half_copies(const uint16_t *base, int64_t nrows, int idx, uint32_t block,
                                                  int rbase, int ch0, int lane) {
  const uint32_t v = (uint32_t)lane & 7u;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const int rl = 4 * i + (lane >> 3);
    int ix = __shfl_sync(0xffffffffu, idx, rl);
    ix = ix < nrows ? ix : (int)nrows - 1;  // never past the array
    const uint32_t row = (uint32_t)(rbase + rl);
    const uint32_t dst = block + row * 128u + ((v ^ (row & 7u)) << 4);
    const uint16_t *src = base + (int64_t)(ix >= 0 ? ix : 0) * D + ch0 + 8 * v;
    tc::cp_async16_zfill(dst, src, ix >= 0 ? 16u : 0u);
  }
}

// Two bf16 values (one 32-bit word) -> two fp16 values, rounded to nearest (exact for magnitudes in
// [2^-17, 65504] and for 0).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return f16pair(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// In-place decode of this thread's half row (one 128-byte row of a swizzled block).
template <bool BYTE_LUT>
__device__ __forceinline__ void decode_half(const HalfRow &d, uint32_t block, int r, uint32_t lut) {
  if (d.idx < 0) return;  // zero-filled by the copies
  const uint32_t rowb = block + (uint32_t)r * 128u, rx = (uint32_t)r & 7u;
  const uint32_t words[4] = {d.c.x, d.c.y, d.c.z, d.c.w};
#pragma unroll
  for (int v = 0; v < 8; v++) {
    const uint32_t addr = rowb + ((((uint32_t)v) ^ rx) << 4);
    const uint4 mu = tc::lds128(addr);
    const uint32_t h16 = words[v >> 1] >> (16 * (v & 1));
    uint32_t q0, q1, q2, q3;
    if (BYTE_LUT) {
      const uint2 qa = tc::lds64(lut + ((h16 << 3) & 0x7F8u));
      const uint2 qb = tc::lds64(lut + ((h16 >> 5) & 0x7F8u));
      q0 = qa.x; q1 = qa.y; q2 = qb.x; q3 = qb.y;
    } else {
      q0 = tc::lds32(lut + ((h16 << 2) & 0x3Cu));
      q1 = tc::lds32(lut + ((h16 >> 2) & 0x3Cu));
      q2 = tc::lds32(lut + ((h16 >> 6) & 0x3Cu));
      q3 = tc::lds32(lut + ((h16 >> 10) & 0x3Cu));
    }
    uint4 o;
    o.x = tc::hadd2(mu.x, tc::hfma2(d.s2, q0, d.m2));
    o.y = tc::hadd2(mu.y, tc::hfma2(d.s2, q1, d.m2));
    o.z = tc::hadd2(mu.z, tc::hfma2(d.s2, q2, d.m2));
    o.w = tc::hadd2(mu.w, tc::hfma2(d.s2, q3, d.m2));
    tc::sts128(addr, o);
  }
}

// A pair of fp16 values one of which is infinite or NaN (exponent field all ones).
__device__ __forceinline__ bool f16pair_nonfinite(uint32_t h) {
  return (h & 0x7C00u) == 0x7C00u || (h & 0x7C000000u) == 0x7C000000u;
}

// In-place bf16 -> fp16 of this thread's half row (a row of the chunk being generated); an element
// beyond the fp16 range records QWM_ERR_RANGE.
__device__ __forceinline__ void convert_half(const HalfRow &d, uint32_t block, int r, int32_t *status) {
  if (d.idx < 0) return;  // zero-filled by the copies
  const uint32_t rowb = block + (uint32_t)r * 128u;
  bool bad = false;
#pragma unroll
  for (int v = 0; v < 8; v++) {
    const uint32_t addr = rowb + ((uint32_t)v << 4);  // the swizzle permutes whole 16-byte chunks
    const uint4 b = tc::lds128(addr);
    const uint32_t w[4] = {b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      o[u] = bf16x2_to_f16x2(w[u]);
      bad |= f16pair_nonfinite(o[u]);
    }
    tc::sts128(addr, make_uint4(o[0], o[1], o[2], o[3]));
  }
  if (bad) qwm_dev_error(status, QWM_ERR_RANGE);
}

// Producer loop of one thread of a pair CTA (rank `cr`).  Keys: thread pr = (group g = pr / 64,
// row pr % 64), decoding channel group g of key row 64 cr + pr % 64 of every tile.  Values: thread pr
// = key row pr, decoding channel group cr.  Same schedule as the single-CTA producer.
template <bool VAL, bool WIDE, bool IDX16, bool EXT>
__device__ __forceinline__ void producer_pair(const AttnParams &p, unsigned char *sm, Bars &bars, int *abort_flag,
                                              uint32_t lut, int h, int64_t qrow0, int cr, int pr, int lane) {
  volatile int *abort_v = abort_flag;
  const int J = p.total_tiles, C = p.C;
  const int g = VAL ? cr : pr >> 6;              // channel group
  const int rr = VAL ? pr : pr & 63;             // row in this CTA's block
  const int rbase = rr - lane;                   // first row of this warp's 32
  const int krow = VAL ? pr : 64 * cr + (pr & 63);  // key row in the tile
  const bool coef = !VAL && g == 0;              // writes the row of the second MMA's B operand
  uint64_t *empty = VAL ? bars.v_empty : bars.k_empty;
  // the even CTA's full barriers (consecutive 8-byte words), as shared::cluster addresses
  const uint32_t full_base = tc::mapa(tc::smem_u32(VAL ? &bars.v_full[0] : &bars.k_full[0]), 0);
  constexpr uint32_t kStage = VAL ? (uint32_t)kBlk : 2u * kBlkH;
  const uint32_t block0 = tc::smem_u32(sm + (VAL ? OFF_V : OFF_K)) + (VAL ? 0u : (uint32_t)g * kBlkH);
  const uint32_t xs0 = tc::smem_u32(sm + OFF_X), qx0 = tc::smem_u32(sm + XL<WIDE>::kOffQX);
  // Value producers: the second MMA's A operand [q U_r | 0 | 1] of chunk t for both Query tiles, into
  // buffer t % 2 once chunk t - 2 has released it (row pr of each tile per thread)
  auto build_qx = [&](int t) -> bool {
    const int b = t & 1, R = p.ch[t].rank;
    constexpr int kRU = WIDE ? 16 : 8;
    if (t >= 2 && !tc::mbar_wait(&bars.qx_free[b], ((t >> 1) - 1) & 1, kWaitNs)) fail(abort_flag, p.status);
    if (__any_sync(0xffffffffu, *abort_v != 0)) return false;  // warp-uniform exit
    // U_r of chunk t -> fp32 buffer b (thread pr = channel pr); the four Value warps meet on u_ready[b]
    // (buffer b was last read for chunk t - 2, before every warp's arrival for chunk t - 1)
    const uint32_t ub = tc::smem_u32(sm + XL<WIDE>::kOffU) + (uint32_t)b * XL<WIDE>::kUBytes;
    {
      float u[kRU];
#pragma unroll
      for (int k = 0; k < kRU; k++) u[k] = (k < R) ? bf16_to_f32(p.ch[t].u_r[((int64_t)h * D + pr) * R + k]) : 0.f;
#pragma unroll
      for (int k4 = 0; k4 < kRU / 4; k4++)
        tc::sts128(ub + (uint32_t)pr * (kRU * 4) + 16u * k4,
                   make_uint4(__float_as_uint(u[4 * k4]), __float_as_uint(u[4 * k4 + 1]),
                              __float_as_uint(u[4 * k4 + 2]), __float_as_uint(u[4 * k4 + 3])));
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&bars.u_ready[b]);
    if (!tc::mbar_wait(&bars.u_ready[b], (t >> 1) & 1, kWaitNs)) fail(abort_flag, p.status);
    if (__any_sync(0xffffffffu, *abort_v != 0)) return false;  // warp-uniform exit
    const uint32_t sq = tc::smem_u32(sm + OFF_Q), dst = qx0 + (uint32_t)(b * NQT) * XL<WIDE>::kQXBytes;
    write_qx_row<WIDE>(R, qrow0 + pr < p.nq, sq, ub, dst, pr);
    write_qx_row<WIDE>(R, qrow0 + 2 * BM + pr < p.nq, sq + 2u * kBlk, ub, dst + XL<WIDE>::kQXBytes, pr);
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive_remote(tc::mapa(tc::smem_u32(&bars.qx_full[b]), 0));
    return true;
  };
  int t0 = 0, ti0 = 0, t1 = 0, ti1 = 0, t2 = 0, ti2 = 0;
  auto advance = [&](int &tt, int &ti) {
    if (++ti == p.ch[tt].tiles) { ti = 0; tt++; }
  };
  auto load_at = [&](int tt, int ti, HalfRow &d) {
    const AttnChunk &c = p.ch[tt];
    const int64_t k0 = (int64_t)ti * BN;
    const int nk = (c.n - k0) < BN ? (int)(c.n - k0) : BN;
    load_half<VAL, IDX16, EXT>(c, h, k0, nk, krow, g, coef, p.compact != 0, d);
  };
  HalfRow A, B;
  B.idx = -1;
  load_at(0, 0, A);
  if (J > 1) {
    advance(t1, ti1);
    load_at(t1, ti1, B);
  }
  // rows that the copies read: the chunk's fp16 codebook, or the bf16 chunk itself
  auto copies = [&](int tt, int idx, uint32_t block) {
    const AttnChunk &c = p.ch[tt];
    if (EXT && c.raw)
      issue_half_copies((VAL ? c.v_raw : c.k_raw) + (int64_t)h * c.n * D, c.n, idx, block, rbase, 64 * g, lane);
    else
      issue_half_copies((VAL ? c.cent_v16 : c.cent_k16) + (int64_t)h * C * D, C, idx, block, rbase, 64 * g, lane);
  };
  copies(0, A.idx, block0);
  tc::cp_async_commit();
  bool live = !VAL || build_qx(0);  // chunk 0's QX while the first copies fly
  auto step = [&](int j, HalfRow &cur, const HalfRow &nxt) -> bool {
    const int s = j % kStages;
    const AttnChunk &ch = p.ch[t0];
    tc::cp_async_wait<0>();
    __syncwarp();  // the warp's copies of tile j, made visible to every lane
    if (EXT && ch.raw) convert_half(cur, block0 + (uint32_t)s * kStage, rr, p.status);
    else decode_half<!WIDE>(cur, block0 + (uint32_t)s * kStage, rr, lut);
    if (!VAL && coef) write_x_row<WIDE>(cur, ch.rank, xs0 + (uint32_t)s * XL<WIDE>::kXBytes, rr);
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive_remote(full_base + 8u * (uint32_t)s);
    if (VAL && ti0 == 0 && t0 + 1 < p.n_chunks) {  // chunk start: the next chunk's QX, ahead of time
      if (!build_qx(t0 + 1)) return false;
    }
    if (j + 1 < J) {  // copies of tile j+1 into its stage once tile j+1-kStages has released it
      const int sn = (j + 1) % kStages;
      if (j + 1 >= kStages && !tc::mbar_wait(&empty[sn], ((j + 1) / kStages - 1) & 1, kWaitNs))
        fail(abort_flag, p.status);
      if (__any_sync(0xffffffffu, *abort_v != 0)) return false;  // warp-uniform exit
      copies(t1, nxt.idx, block0 + (uint32_t)sn * kStage);
      tc::cp_async_commit();
    }
    t2 = t1; ti2 = ti1;
    if (j + 2 < J) {
      advance(t2, ti2);
      load_at(t2, ti2, cur);
    }
    t0 = t1; ti0 = ti1;
    t1 = t2; ti1 = ti2;
    return true;
  };
  for (int j = 0; live && j < J; j += 2) {
    if (!step(j, A, B)) break;
    if (j + 1 < J && !step(j + 1, B, A)) break;
  }
  tc::cp_async_wait<0>();
}

// WIDE: PSAC ranks above 8 (32-column second-MMA operands).  IDX16: uint16 centroid indices.
// EXT: the call includes a bf16 chunk (the chunk being generated), compact INT2 metadata or per-head
// PSAC coefficient layouts.  LSE: the rows' log-sum-exp is written (and, merging, read with O).
template <bool WIDE, bool IDX16, bool EXT, bool LSE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attend_pair_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char *sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ __align__(64) uint32_t code_lut[WIDE ? 16 : 512];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // one head's items run next to each other (launch order): its packed cache stays in L2
  const int h = (int)blockIdx.y, item = (int)(blockIdx.x >> 1);
  const int cr = (int)tc::cluster_ctarank();
  const int64_t qb = (int64_t)item * kPairQ + (int64_t)cr * BM;  // this CTA's row 0 of tile 0
  // a short last item whose second 256-row Query tile is empty runs the first tile only
  const bool skip1 = (int64_t)item * kPairQ + 2 * BM >= p.nq;
  volatile int *abort_v = &abort_flag;

  // ---- this CTA's two Query tiles (rows qb + 256 x + rr) -> shared memory as fp16 ----
  for (int e = tid; e < NQT * BM * (D / 8); e += kThreads) {
    const int row = e / (D / 8), ci = e % (D / 8);
    const int x = row / BM, rr = row % BM, b = ci / 8;
    const int64_t qi = qb + (int64_t)x * 2 * BM + rr;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (qi < p.nq) v = *(const uint4 *)(p.q + ((int64_t)h * p.nq + qi) * D + 8 * ci);
    const uint32_t bw[4] = {v.x, v.y, v.z, v.w};
    uint32_t hw[4];
    bool bad = false;
#pragma unroll
    for (int u = 0; u < 4; u++) {
      hw[u] = bf16x2_to_f16x2(bw[u]);
      bad |= f16pair_nonfinite(hw[u]);
    }
    if (bad) qwm_dev_error(p.status, QWM_ERR_RANGE);  // a Query element beyond the fp16 range
    *(uint4 *)(sm + OFF_Q + (x * 2 + b) * kBlk + tc::sw128_offset(rr, 8 * (ci % 8))) =
        make_uint4(hw[0], hw[1], hw[2], hw[3]);
  }
  if (!WIDE && tid < 256) {
    uint32_t f[4];
#pragma unroll
    for (int t = 0; t < 4; t++) f[t] = ((0x42403C00u >> (8 * ((tid >> (2 * t)) & 3))) & 0xFFu) << 8;
    code_lut[2 * tid] = f[0] | (f[1] << 16);
    code_lut[2 * tid + 1] = f[2] | (f[3] << 16);
  }
  if (WIDE && tid < 16) {
    const uint32_t lo = ((0x42403C00u >> (8 * (tid & 3))) & 0xFFu) << 8;
    const uint32_t hi = ((0x42403C00u >> (8 * (tid >> 2))) & 0xFFu) << 8;
    code_lut[tid] = lo | (hi << 16);
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; i++) {
      tc::mbar_init(&bars.k_full[i], 2 * kProdWarps);  // both CTAs' producer warps (even CTA's copy used)
      tc::mbar_init(&bars.v_full[i], 2 * kProdWarps);
      tc::mbar_init(&bars.k_empty[i], 1);
      tc::mbar_init(&bars.v_empty[i], 1);
    }
    for (int i = 0; i < 2; i++) {
      tc::mbar_init(&bars.s_full[i], 1);
      tc::mbar_init(&bars.p_ready[i], 8);              // both CTAs' 4 softmax warps of tile i
    }
    for (int i = 0; i < 2; i++) {
      tc::mbar_init(&bars.qx_full[i], 2 * kProdWarps);  // both CTAs' Value producer warps
      tc::mbar_init(&bars.qx_free[i], 1);
      tc::mbar_init(&bars.u_ready[i], kProdWarps);      // this CTA's Value producer warps
    }
    tc::mbar_init(&bars.o_done, 1);
    tc::mbar_init(&bars.drain, 1);
    tc::mbar_init(&bars.never, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc2(&tmem_base_sh, 512);
    tc::tmem_relinquish2();
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // both CTAs' barriers exist before the first arrival from the peer
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const int J = p.total_tiles;

  if (warp < kSoftmaxWarps) {
    // ======================= softmax (Query tile x, row = TMEM lane) =======================
    const int x = warp / 4, sub = warp % 4, row = 32 * sub + lane;
    const int Jx = (x == 1 && skip1) ? 0 : J;  // tiles this softmax group sees
    const uint32_t lane_addr = (uint32_t)(32 * sub) << 16;
    const uint32_t tS = tmem + lane_addr + 128u * x, tO = tmem + lane_addr + 256u + 128u * x;
    const uint32_t p_ready0 = tc::mapa(tc::smem_u32(&bars.p_ready[x]), 0);
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY;
    uint64_t acc0 = 0ull, acc1 = 0ull;
    const uint64_t sc2 = pk64(__float_as_uint(sl2), __float_as_uint(sl2));
    const int64_t qrow = qb + (int64_t)x * 2 * BM + row;  // this thread's Query row
    int tc_ = 0, ti_ = 0;                                  // chunk and tile in chunk of tile j
    bool ok = true;
    for (int j = 0; j < Jx; j++) {
      if (!tc::mbar_wait(&bars.s_full[x], j & 1, kWaitNs)) fail(&abort_flag, p.status);
      if (*abort_v) { ok = false; break; }
      tc::fence_after_sync();
      // block-causal mask of the chunk being generated: columns from `lim` on belong to a later frame
      int lim = BN;
      if (EXT && p.any_causal) {
        const AttnChunk &c = p.ch[tc_];
        if (c.tpf > 0) {
          const int64_t l = (qrow / c.tpf + 1) * c.tpf - (int64_t)ti_ * BN;
          lim = l < 0 ? 0 : (l < BN ? (int)l : BN);
        }
        if (++ti_ == c.tiles) { ti_ = 0; tc_++; }
      }
      // one pass over the tile, 32 columns at a time: the chunk's max, then its exponentials with the
      // running max m_used; when a chunk raises the max by more than 2^8 (rare after the first
      // chunk) the sum, O and the P chunks already stored for this tile are first rescaled
      uint32_t r[32];
#pragma unroll 1
      for (int cq = 0; cq < 4; cq++) {
        tc::tmem_ld16(tS + 32u * cq, r);
        tc::tmem_ld16(tS + 32u * cq + 16u, r + 16);
        tc::tmem_ld_wait();
        if (lim < 32 * cq + 32) {
#pragma unroll
          for (int i = 0; i < 32; i++)
            if (32 * cq + i >= lim) r[i] = 0xFF800000u;  // -inf: weight exactly 0
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          mx0 = tc::max3(mx0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
          mx1 = tc::max3(mx1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
        }
        const float m_new = fmaxf(m_used, fmaxf(mx0, mx1) * sl2);
        if (__any_sync(0xffffffffu, m_new > m_used + kRescaleThreshold)) {
          const float alpha = tc::ex2_approx(m_used - m_new);  // 0 while m_used is -inf
          const uint64_t a2 = pk64(__float_as_uint(alpha), __float_as_uint(alpha));
          acc0 = tc::fma2(acc0, a2, 0ull);
          acc1 = tc::fma2(acc1, a2, 0ull);
          if (j > 0) {  // O of the earlier tiles (complete: S_x(j) finished after PV_x(j-1))
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t o[32];
              tc::tmem_ld32(tO + c, o);
              tc::tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tc::tmem_st32(tO + c, o);
            }
          }
          tc::tmem_st_wait();
#pragma unroll 1
          for (int pc = 0; pc < cq; pc++) {  // P chunks of this tile already written
            uint32_t pw[16];
            tc::tmem_ld16(tS + 16u * pc, pw);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; i++) {
              const float2 v = __half22float2(*(const __half2 *)&pw[i]);
              pw[i] = f16pair(v.x * alpha, v.y * alpha);
            }
            tc::tmem_st16(tS + 16u * pc, pw);
          }
          m_used = m_new;
        }
        const float mneg = (EXT && m_used == -INFINITY) ? 0.f : -m_used;  // a row with no unmasked key yet
        const uint64_t nm2 = pk64(__float_as_uint(mneg), __float_as_uint(mneg));
        uint32_t pw[16];
#pragma unroll
        for (int i = 0; i < 16; i++) {  // packed fp32 pairs: x = S * scale - m, then 2^x
          const uint64_t x2 = tc::fma2(pk64(r[2 * i], r[2 * i + 1]), sc2, nm2);
          const float e0 = tc::ex2_approx(tc::f2lo(x2)), e1 = tc::ex2_approx(tc::f2hi(x2));
          const uint64_t e2 = pk64(__float_as_uint(e0), __float_as_uint(e1));
          if (i & 1) acc1 = tc::add2(acc1, e2);
          else acc0 = tc::add2(acc0, e2);
          pw[i] = f16pair(e0, e1);
        }
        tc::tmem_st16(tS + 16u * cq, pw);  // P (fp16 pairs) overlays logits already read
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_remote(p_ready0);
    }
    if (ok && Jx > 0 && !tc::mbar_wait(&bars.o_done, 0, kWaitNs)) fail(&abort_flag, p.status);
    if (ok && Jx > 0 && !*abort_v) {
      tc::fence_after_sync();
      const uint64_t lsum = tc::add2(acc0, acc1);
      const float l = tc::f2lo(lsum) + tc::f2hi(lsum);
      const int64_t qi = qb + (int64_t)x * 2 * BM + row;
      float inv = 1.f / l;
      float keep = 0.f;  // merge: the weight of the result already in out
      if (LSE && qi < p.nq) {
        // log2 of this call's exponential sum: sum_j 2^(S_j * scale * log2 e) = 2^m_used * l
        float *lp = p.lse + (int64_t)h * p.nq + qi;
        const float L = m_used + log2f(l);
        float Lout = L;
        if (p.merge) {  // out = w_prev out + w_this O / l, the weights the parts' shares of the union's sum
          const float Lp = *lp, Lm = fmaxf(Lp, L);
          const float wp = exp2f(Lp - Lm), wt = exp2f(L - Lm), den = wp + wt;
          keep = wp / den;
          inv = wt > 0.f ? wt / (den * l) : 0.f;
          Lout = Lm + log2f(den);
        }
        *lp = Lout;
      }
      uint32_t o[32];
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        tc::tmem_ld32(tO + c, o);
        tc::tmem_ld_wait();
        if (qi < p.nq) {
          float4 *dst = (float4 *)(p.out + ((int64_t)h * p.nq + qi) * D + c);
          if (LSE && keep > 0.f) {
#pragma unroll
            for (int v = 0; v < 8; v++) {
              const float4 a = dst[v];
              dst[v] = make_float4(fmaf(keep, a.x, __uint_as_float(o[4 * v]) * inv),
                                   fmaf(keep, a.y, __uint_as_float(o[4 * v + 1]) * inv),
                                   fmaf(keep, a.z, __uint_as_float(o[4 * v + 2]) * inv),
                                   fmaf(keep, a.w, __uint_as_float(o[4 * v + 3]) * inv));
            }
          } else {
#pragma unroll
            for (int v = 0; v < 8; v++)
              dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                   __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
          }
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ======================= MMA issue: one thread of the even CTA, for the pair =======================
    if (cr == 0 && lane == 0) {
      const uint32_t idesc = tc::idesc_f16_f32(2 * BM, BN);
      const uint32_t idesc_pv = tc::idesc_f16_f32_bmn(2 * BM, D);
      const uint32_t tS[2] = {tmem, tmem + 128u}, tO[2] = {tmem + 256u, tmem + 384u};
      const uint32_t sQ = tc::smem_u32(sm + OFF_Q), sK = tc::smem_u32(sm + OFF_K), sV = tc::smem_u32(sm + OFF_V);
      const uint32_t sX = tc::smem_u32(sm + OFF_X), sQX = tc::smem_u32(sm + XL<WIDE>::kOffQX);
      constexpr uint16_t kBoth = 3;
      int t = 0, tile_in_chunk = 0, prev_stage = 0;
      bool ok = true;
      auto qk = [&](int x, int s, int nx, int qb) {
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
          const uint32_t qo = (uint32_t)((kk / 4) * kBlk + 32 * (kk % 4));
          const uint32_t ko = (uint32_t)((kk / 4) * kBlkH + 32 * (kk % 4));
          tc::mma2_ss(tS[x], tc::desc_sw128(sQ + (x * 2) * kBlk + qo), tc::desc_sw128(sK + s * 2 * kBlkH + ko), idesc,
                      kk > 0);
        }
        for (int ks = 0; ks < nx; ks++)
          tc::mma2_ss(tS[x], tc::desc_noswz(sQX + (qb * NQT + x) * XL<WIDE>::kQXBytes + 256u * ks, 128, XL<WIDE>::kSbo),
                      tc::desc_noswz(sX + s * XL<WIDE>::kXBytes + 256u * ks, 128, XL<WIDE>::kSbo), idesc, 1);
      };
      auto pv = [&](int x, int s, bool first) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; kk++)
          tc::mma2_ts(tO[x], tS[x] + 8u * kk, tc::desc_sw128_mn(sV + s * kBlk + 2048u * kk, kBlk, 1024), idesc_pv,
                      (!first || kk > 0));
      };
      if (p.test_expire) ok = tc::mbar_wait(&bars.never, 0, kTestWaitNs);  // test hook: a wait nothing ends
      for (int j = 0; ok && j < J; j++) {
        const int s = j % kStages;
        const uint32_t ph = (uint32_t)(j / kStages) & 1u;
        const AttnChunk &ch = p.ch[t];
        const int nx = (WIDE && ch.rank > 8) ? 2 : 1;
        ok = tc::mbar_wait_cluster(&bars.k_full[s], ph, kWaitNs) && !*abort_v;
        if (ok && tile_in_chunk == 0) ok = tc::mbar_wait_cluster(&bars.qx_full[t & 1], (t >> 1) & 1, kWaitNs);
        if (!ok) break;
        tc::fence_after_sync();
        qk(0, s, nx, t & 1);
        tc::mma2_commit(&bars.s_full[0], kBoth);
        if (j > 0 && !skip1) {
          ok = tc::mbar_wait_cluster(&bars.p_ready[1], (j - 1) & 1, kWaitNs) && !*abort_v;
          if (!ok) break;
          tc::fence_after_sync();
          pv(1, prev_stage, j - 1 == 0);
          tc::mma2_commit(&bars.v_empty[prev_stage], kBoth);
        }
        if (!skip1) {
          qk(1, s, nx, t & 1);
          tc::mma2_commit(&bars.s_full[1], kBoth);
        }
        tc::mma2_commit(&bars.k_empty[s], kBoth);
        const bool last_of_chunk = tile_in_chunk + 1 == ch.tiles;
        if (last_of_chunk) tc::mma2_commit(&bars.qx_free[t & 1], kBoth);
        ok = tc::mbar_wait_cluster(&bars.v_full[s], ph, kWaitNs) &&
             tc::mbar_wait_cluster(&bars.p_ready[0], j & 1, kWaitNs) && !*abort_v;
        if (!ok) break;
        tc::fence_after_sync();
        pv(0, s, j == 0);
        if (skip1) tc::mma2_commit(&bars.v_empty[s], kBoth);  // no second tile reads this stage
        prev_stage = s;
        if (last_of_chunk) { tile_in_chunk = 0; t++; }
        else tile_in_chunk++;
      }
      if (ok && J > 0) {
        if (!skip1) {
          ok = tc::mbar_wait_cluster(&bars.p_ready[1], (J - 1) & 1, kWaitNs) && !*abort_v;
          if (ok) {
            tc::fence_after_sync();
            pv(1, prev_stage, J - 1 == 0);
          }
        }
        if (ok) tc::mma2_commit(&bars.o_done, kBoth);
      }
      if (!ok) fail(&abort_flag, p.status);
      tc::mma2_commit(&bars.drain, 1);  // every MMA issued above completes before TMEM is released
      if (!tc::mbar_wait(&bars.drain, 0, kWaitNs)) qwm_dev_error(p.status, QWM_ERR_DEVICE_TIMEOUT);
    }
  } else if (warp < kVWarp0) {
    producer_pair<false, WIDE, IDX16, EXT>(p, sm, bars, &abort_flag, tc::smem_u32(code_lut), h, qb, cr,
                                      tid - 32 * kKWarp0, lane);
  } else {
    producer_pair<true, WIDE, IDX16, EXT>(p, sm, bars, &abort_flag, tc::smem_u32(code_lut), h, qb, cr,
                                     tid - 32 * kVWarp0, lane);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // the peer has finished with this CTA's barriers, shared and tensor memory
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc2(tmem, 512);
  }
}

template <bool WIDE, bool IDX16, bool EXT, bool LSE>
cudaError_t launch_pair(const AttnParams &p, dim3 grid, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(attend_pair_kernel<WIDE, IDX16, EXT, LSE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, XL<WIDE>::kSmemAlloc);
  if (e != cudaSuccess) return e;
  attend_pair_kernel<WIDE, IDX16, EXT, LSE><<<grid, kThreads, XL<WIDE>::kSmemAlloc, st>>>(p);
  return cudaGetLastError();
}

template <bool EXT, bool LSE>
cudaError_t launch_pair_ext(const AttnParams &p, dim3 grid, bool wide, bool idx16, cudaStream_t st) {
  if (wide && idx16) return launch_pair<true, true, EXT, LSE>(p, grid, st);
  if (wide) return launch_pair<true, false, EXT, LSE>(p, grid, st);
  if (idx16) return launch_pair<false, true, EXT, LSE>(p, grid, st);
  return launch_pair<false, false, EXT, LSE>(p, grid, st);
}

}  // namespace

cudaError_t launch_attend(const qwm_config &cfg, const uint16_t *q, int64_t nq, const qwm_chunk *chunks,
                          int n_chunks, float scale, float *out, float *lse, int merge, int num_sms, int32_t *status,
                          cudaStream_t st) {
  (void)num_sms;
  AttnParams p;  // passed by value (about 17 KB of kernel parameters)
  p.q = q; p.out = out; p.lse = lse; p.merge = lse ? merge : 0; p.nq = nq; p.H = cfg.heads; p.C = cfg.n_centroids;
  p.compact = cfg.storage == QWM_STORAGE_COMPACT;
  p.any_causal = 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.test_expire = (cfg.test_flags & QWM_TEST_EXPIRE_WAIT) != 0;
  p.status = status;
  int used = 0, tiles = 0;
  bool wide = false;  // a chunk with PSAC rank above 8: the 32-column second-MMA operands
  bool raw = false;   // a bf16 chunk (the chunk being generated)
  bool per_head = false;  // a chunk with per-head PSAC ranks and layouts
  for (int i = 0; i < n_chunks; i++) {
    const qwm_chunk &c = chunks[i];
    if (c.n_tokens == 0) continue;  // empty chunks contribute nothing
    if (used == kMaxChunks) return cudaErrorInvalidValue;
    AttnChunk &a = p.ch[used++];
    a.n = c.n_tokens; a.rank = c.rank_eff; a.tiles = (int)((c.n_tokens + BN - 1) / BN);
    a.k_codes = c.k_codes; a.v_codes = c.v_codes;
    a.k_idx = (const uint8_t *)c.k_idx; a.v_idx = (const uint8_t *)c.v_idx;
    a.k_scale = c.k_scale; a.k_min = c.k_min; a.v_scale = c.v_scale; a.v_min = c.v_min;
    a.cent_k16 = c.cent_k16; a.cent_v16 = c.cent_v16; a.c_scale = c.c_scale; a.u_r = c.u_r; a.c = c.c;
    a.raw = c.kind == QWM_CHUNK_BF16;
    raw |= a.raw != 0;
    a.tpf = a.raw ? c.causal_tpf : 0;
    if (a.tpf > 0) p.any_causal = 1;
    a.k_raw = c.k_raw; a.v_raw = c.v_raw;
    a.k_s8 = c.k_s8; a.v_s8 = c.v_s8; a.k_zp = c.k_zp; a.v_zp = c.v_zp;
    a.k_sigma = c.k_sigma; a.v_sigma = c.v_sigma;
    a.per_head = c.kind == QWM_CHUNK_PACKED && c.rank_eff > 0 && c.c_layout == QWM_C_PER_HEAD;
    a.c_heads = c.c_heads; a.c_mask = c.c_mask; a.c_tile_rank = c.c_tile_rank;
    per_head |= a.per_head != 0;
    tiles += a.tiles;
    wide |= a.rank > 8;
  }
  p.n_chunks = used;
  p.total_tiles = tiles;
  const bool idx16 = cfg.n_centroids > 256;
  cudaError_t e;
  const dim3 grid((unsigned)(2 * ((nq + kPairQ - 1) / kPairQ)), cfg.heads);  // CTA pairs
  const bool ext = raw || p.compact || per_head;
  if (lse)
    e = ext ? launch_pair_ext<true, true>(p, grid, wide, idx16, st) : launch_pair_ext<false, true>(p, grid, wide, idx16, st);
  else
    e = ext ? launch_pair_ext<true, false>(p, grid, wide, idx16, st)
            : launch_pair_ext<false, false>(p, grid, wide, idx16, st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}
