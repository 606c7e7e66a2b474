// Step 2a: per-head Lloyd k-means codebook of one chunk, on the tensor cores.
//
// QVG summary §2A: tokens are grouped by k-means along the sequence axis and each token is
// represented by its centroid plus a residual; §2C: the k-means of a new chunk starts from
// the previous chunk's centroids (warm start).  Each Lloyd iteration assigns every token to
// its nearest centroid (Euclidean, lower index on ties) and moves each centroid to the mean of
// its members; a centroid left without members keeps its position.  Centroids stay fp32
// between iterations and are rounded to bf16 at the end.
//
// Assignment = distance GEMM: ||x - mu_j||^2 = ||x||^2 + ||mu_j||^2 - 2 x.mu_j, and only
// ||mu_j||^2 - 2 x.mu_j matters for the argmin.  x is bf16 (exact); the fp32 centroid is split
// as mu = hi + lo with hi, lo bf16, so two bf16 MMAs give x.mu to about 2^-17 relative.
//
// km_assign_kernel (one CTA = one head x a contiguous range of 128-token tiles; 320 threads):
//   warp 0    TMA producer: token tiles (2 x [128][64] bf16, 128-byte swizzle) into 2 stages
//   warp 1    TMEM owner and MMA issuer: D[128 x C] = X hi^T + X lo^T into 2 TMEM buffers
//   warps 2-9 epilogue, two warpgroups taking alternate tiles: thread = token = TMEM lane;
//             argmin over the C columns (two interleaved chains, lower index on ties)
// The assignments of up to 4096 tokens stay in shared memory.  Then the cluster sums: the token
// tiles stream through up to four token stages again (TMA), pairs of epilogue warps write the one-hot
// assignment matrix of each 64-token half-tile into one of three buffers over the codebook area, and
// the MMA warp accumulates sums = onehot^T X in TMEM; the CTA adds them to its own slice of the
// workspace and km_update_kernel reduces the slices in a fixed order.
// Resident codebooks also keep every token's assignment in a workspace array between iterations:
// from the second iteration on, phase 1 flags the 64-token half-tiles in which a token changed
// cluster, phase 2 re-reads only the tiles holding one, its one-hot matrix carries +1 at a moved
// token's new cluster and -1 at its old one, and the CTA adds the result (and the count changes) to
// its slice, which therefore holds the sums of the current assignment; only the centroids a moved
// token left or joined are written back.  After a warm start about 1% of the tokens move in the
// second iteration and fewer than 0.1% from the sixth on.
// The kernels that produce centroids (kmeans_init_kernel, km_update_kernel) also write the next
// assignment's operands: each head's hi/lo bf16 blocks, 128-byte swizzled exactly as the MMA reads
// them, and the squared norms ||mu_j||^2, so that the assignment kernel starts with one bulk copy
// instead of converting the fp32 codebook itself.  Codebooks of up to 256 centroids are one slice
// held in shared memory for the whole launch.  Codebooks of 1024 centroids (WIDE) do not fit: their
// operands are 128-centroid slices that the producer streams through one shared-memory buffer for
// every tile, and the argmin runs slice by slice over two 128-column TMEM halves per epilogue
// group.  Their cluster sums come from a stable counting sort of the super-chunk's assignments and
// one warp per centroid adding its members' rows in token order (a one-hot matrix would not fit).
// All waits are bounded; on expiry the kernel records QWM_ERR_DEVICE_TIMEOUT and stops.
#include "qwm_internal.cuh"
#include "tc.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int TILE = 128;
constexpr int kMaxTok = 4096;  // tokens per super-chunk (assignments kept in shared memory)
constexpr int kThreads = 320;
constexpr uint64_t kWaitNs = 1000000000ull;

constexpr int kSlice = 128;      // centroids per streamed slice (WIDE)
constexpr int kSliceBytes = 4 * kSlice * 128;  // hi and lo blocks of one slice

struct KmSmem {  // offsets from a 1024-aligned base, for a codebook of C centroids
  int bh, bl, x, norm, asg, cnt, cur, mem, old, flg, lst, total;
  __host__ __device__ KmSmem(int C, bool wide) {
    const int CB = wide ? kSlice : C;  // centroids held in shared memory at once
    bh = 0;                        // 2 blocks of [CB][64] bf16 (hi)
    bl = bh + 2 * CB * 128;        // 2 blocks of [CB][64] bf16 (lo)
    // resident: the codebook area doubles as the one-hot buffers and extra token stages of the cluster sums
    const int onehot = wide ? 0 : 2 * ((C + 127) / 128) * 2 * TILE * 128;
    x = 4 * CB * 128 > onehot ? 4 * CB * 128 : onehot;  // 2 stages x 2 blocks of [128][64]
    norm = x + 2 * 2 * TILE * 128; // C floats
    asg = norm + 4 * C;            // kMaxTok indices (uint8, or uint16 when WIDE)
    cnt = asg + (wide ? 2 : 1) * kMaxTok;  // WIDE cluster sums: counts [C], cursors [C], members
    cur = cnt + (wide ? 4 * C : 0);
    mem = cur + (wide ? 4 * C : 0);
    old = mem + (wide ? 2 * kMaxTok : 0);  // resident: previous assignments of the super-chunk
    flg = old + (wide ? 0 : kMaxTok);      // resident: per tile, bit h = half-tile h has a changed token
    lst = flg + (wide ? 0 : 4 * (kMaxTok / TILE));  // resident: tiles whose sums phase 2 reads
    total = lst + (wide ? 0 : 4 * (kMaxTok / TILE));
  }
};


// Centroids per operand slice: the whole codebook when it stays in shared memory, else kSlice.
__host__ __device__ __forceinline__ int slice_cents(int C) { return C > QWM_MAX_RESIDENT_CENTROIDS ? kSlice : C; }

// Operand image of one head's fp32 codebook: [C / CB] slices, each the (hi, lo) pair of
// 128-byte-swizzled [CB][64]-channel block pairs (CB = slice_cents(C)), mu = hi + lo with hi, lo bf16;
// then norms[j] = ||mu_j||^2.  Called by all D threads of a block, thread c holding channel c of
// centroid j.
__device__ __forceinline__ void write_operand(unsigned char *__restrict__ img, float *__restrict__ norms, int C, int j,
                                              int c, float mu) {
  __shared__ float part[D / 32];
  const int CB = slice_cents(C);
  const float hi = __bfloat162float(__float2bfloat16_rn(mu));
  unsigned char *sl = img + (int64_t)(j / CB) * 4 * CB * 128;
  const uint32_t off = (uint32_t)(c / 64) * CB * 128u + tc::sw128_offset(j % CB, c % 64);
  *(uint16_t *)(sl + off) = f32_to_bf16_rn(hi);
  *(uint16_t *)(sl + 2 * CB * 128 + off) = f32_to_bf16_rn(mu - hi);
  float s = mu * mu;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((c & 31) == 0) part[c >> 5] = s;
  __syncthreads();
  if (c == 0) norms[j] = (part[0] + part[1]) + (part[2] + part[3]);
}

// Initial centroids: the warm-start codebook, or tokens floor(j n / C) of the chunk.
__global__ void __launch_bounds__(D) kmeans_init_kernel(const uint16_t *__restrict__ x, int64_t n, int C,
                                                        const uint16_t *__restrict__ init, float *__restrict__ cent,
                                                        unsigned char *__restrict__ img, float *__restrict__ norms) {
  const int h = blockIdx.y, j = blockIdx.x, c = threadIdx.x;
  const uint16_t *src = init ? init + ((int64_t)h * C + j) * D : x + ((int64_t)h * n + (int64_t)j * n / C) * D;
  const float mu = bf16_to_f32(src[c]);
  cent[((int64_t)h * C + j) * D + c] = mu;
  write_operand(img + (int64_t)h * C * 512, norms + (int64_t)h * C, C, j, c, mu);
}

struct AssignParams {
  const uint16_t *x;     // [H][n][D] bf16
  const unsigned char *img;  // operand image [H][C / CB][slice]
  const float *norms;        // [H][C]
  float *part_sum;       // [H][G][C][D]
  int32_t *part_cnt;     // [H][G][C]
  uint8_t *prev;         // resident codebooks: [H][n] assignments of the previous iteration, or NULL
  int64_t n;
  int C, G;
  int delta;             // 1: update the CTA's sums with the tokens whose assignment changed
  int32_t *status;
};

template <bool WIDE>
__global__ void __launch_bounds__(kThreads, 1) km_assign_kernel(const __grid_constant__ TensorMap128 tmap,
                                                                 const AssignParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char *sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t x_full[2], x_empty[2], t_full[2], t_empty[2], drain;
  __shared__ uint64_t p2_full[4], p2_empty[4], a_full[3], a_empty[3], p2_done;
  __shared__ uint64_t tw_full[4], tw_empty[4], sl_full, sl_empty;  // WIDE: TMEM halves, slice buffer
  __shared__ uint64_t cb_full;  // operands and norms of the codebook
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int nl_sh;
  __shared__ uint32_t touched[QWM_MAX_RESIDENT_CENTROIDS / 32];  // delta: centroids a moved token left or joined
  const int C = p.C;
  const int NSL = WIDE ? C / kSlice : 1;
  const KmSmem L(C, WIDE);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, cta = blockIdx.x;
  const int64_t tiles = (p.n + TILE - 1) / TILE;
  const int64_t per = (tiles + p.G - 1) / p.G;
  const int64_t tile0 = (int64_t)cta * per;
  const int64_t tile1 = tile0 + per < tiles ? tile0 + per : tiles;
  int32_t *cnts = (int32_t *)(sm + L.norm);     // phase 2: [C], over the norms
  float *norm = (float *)(sm + L.norm);
  uint8_t *asg = sm + L.asg;
  uint16_t *asg16 = (uint16_t *)(sm + L.asg);  // WIDE
  uint8_t *asg_old = sm + L.old;               // delta: the previous assignments
  uint32_t *tflag = (uint32_t *)(sm + L.flg);
  int32_t *tlist = (int32_t *)(sm + L.lst);
  const bool delta = !WIDE && p.delta != 0;
  volatile int *abort_v = &abort_flag;

  if (tid == 0) {
    for (int i = 0; i < 2; i++) {
      tc::mbar_init(&x_full[i], 1);
      tc::mbar_init(&x_empty[i], 1);
      tc::mbar_init(&t_full[i], 1);
      tc::mbar_init(&t_empty[i], 4);
    }
    for (int i = 0; i < 3; i++) {
      tc::mbar_init(&a_full[i], 2);  // the two warps that build one-hot buffer i
      tc::mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 4; i++) {
      tc::mbar_init(&p2_full[i], 1);
      tc::mbar_init(&p2_empty[i], 1);
    }
    for (int i = 0; i < 4; i++) {
      tc::mbar_init(&tw_full[i], 1);
      tc::mbar_init(&tw_empty[i], 4);
    }
    tc::mbar_init(&sl_full, 1);
    tc::mbar_init(&sl_empty, 1);
    tc::mbar_init(&p2_done, 1);
    tc::mbar_init(&cb_full, 1);
    tc::mbar_init(&drain, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&tmem_base_sh, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  float *psum = p.part_sum + ((int64_t)h * p.G + cta) * C * D;
  int32_t *pcnt = p.part_cnt + ((int64_t)h * p.G + cta) * C;
  int64_t g_tile = 0;  // tiles this CTA has processed (barrier phases)
  int64_t g2 = 0;      // tiles re-read by phase 2 (barrier phases)
  int n_sc = 0;        // super-chunks done (phase of p2_done)
  int n_cb = 0;        // operand loads done (phase of cb_full)
  for (int64_t sc0 = tile0, first = 1; (first && !delta) || sc0 < tile1; sc0 += kMaxTok / TILE, first = 0) {
    const int64_t left = tile1 - sc0;
    const int nt = left <= 0 ? 0 : (left < kMaxTok / TILE ? (int)left : kMaxTok / TILE);
    // ---- operands of the codebook (resident: hi/lo blocks; WIDE: streamed per tile) and norms ----
    // (the previous super-chunk wrote the one-hot buffers and counts over these areas)
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      const uint32_t img_bytes = WIDE ? 0u : (uint32_t)C * 512u;
      tc::mbar_arrive_expect_tx(&cb_full, img_bytes + 4u * (uint32_t)C);
      if (!WIDE) tc::bulk_load(tc::smem_u32(sm + L.bh), p.img + (int64_t)h * C * 512, img_bytes, &cb_full);
      tc::bulk_load(tc::smem_u32(norm), p.norms + (int64_t)h * C, 4u * (uint32_t)C, &cb_full);
    }
    if (!tc::mbar_wait(&cb_full, (uint32_t)(n_cb & 1), kWaitNs)) *abort_v = 1;
    n_cb++;
    if (delta)
      for (int i = tid; i < kMaxTok / TILE; i += kThreads) tflag[i] = 0u;
    __syncthreads();
    if (*abort_v) break;
    // ---- phase 1: assignments of nt tiles ----
    if (warp == 0) {
      if (lane == 0) {
        for (int i = 0; i < nt && !*abort_v; i++) {
          const int64_t g = g_tile + i;
          const int s = (int)(g & 1);
          if (g >= 2 && !tc::mbar_wait(&x_empty[s], (uint32_t)(((g >> 1) - 1) & 1), kWaitNs)) {
            *abort_v = 1;
            break;
          }
          tc::mbar_arrive_expect_tx(&x_full[s], 2 * TILE * 128);
          const int row = (int)((int64_t)h * p.n + (sc0 + i) * TILE);
          unsigned char *dst = sm + L.x + s * 2 * TILE * 128;
          tc::tma_load_2d(dst, &tmap, 0, row, &x_full[s]);
          tc::tma_load_2d(dst + TILE * 128, &tmap, 64, row, &x_full[s]);
          if (WIDE) {  // this tile's pass over the codebook, one slice at a time
            const unsigned char *img = p.img + (int64_t)h * NSL * kSliceBytes;
            for (int sl = 0; sl < NSL; sl++) {
              const int64_t u = g * NSL + sl;
              if (u >= 1 && !tc::mbar_wait(&sl_empty, (uint32_t)((u - 1) & 1), kWaitNs)) { *abort_v = 1; break; }
              tc::mbar_arrive_expect_tx(&sl_full, kSliceBytes);
              tc::bulk_load(tc::smem_u32(sm), img + (int64_t)sl * kSliceBytes, kSliceBytes, &sl_full);
            }
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        const int CB = WIDE ? kSlice : C;  // centroids per MMA
        const uint32_t idesc = tc::idesc_bf16_f32(TILE, CB);
        const uint32_t sx = tc::smem_u32(sm + L.x), sbh = tc::smem_u32(sm + L.bh), sbl = tc::smem_u32(sm + L.bl);
        auto issue = [&](uint32_t d, int s) {
#pragma unroll
          for (int kk = 0; kk < D / 16; kk++) {
            const uint32_t xo = sx + s * 2 * TILE * 128 + (kk / 4) * TILE * 128 + 32 * (kk % 4);
            const uint32_t bo = (kk / 4) * CB * 128 + 32 * (kk % 4);
            tc::mma_ss(d, tc::desc_sw128(xo), tc::desc_sw128(sbh + bo), idesc, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; kk++) {
            const uint32_t xo = sx + s * 2 * TILE * 128 + (kk / 4) * TILE * 128 + 32 * (kk % 4);
            const uint32_t bo = (kk / 4) * CB * 128 + 32 * (kk % 4);
            tc::mma_ss(d, tc::desc_sw128(xo), tc::desc_sw128(sbl + bo), idesc, 1);
          }
        };
        for (int i = 0; i < nt && !*abort_v; i++) {
          const int64_t g = g_tile + i;
          const int s = (int)(g & 1);
          if (WIDE) {
            if (!tc::mbar_wait(&x_full[s], (uint32_t)((g >> 1) & 1), kWaitNs)) { *abort_v = 1; break; }
            for (int sl = 0; sl < NSL; sl++) {
              // slice sl of tile g -> TMEM half (sl & 1) of buffer s; that half's k-th use
              const int64_t u = g * NSL + sl, k = (g >> 1) * (NSL / 2) + (sl >> 1);
              const int hb = 2 * s + (sl & 1);
              if (!tc::mbar_wait(&sl_full, (uint32_t)(u & 1), kWaitNs) ||
                  (k >= 1 && !tc::mbar_wait(&tw_empty[hb], (uint32_t)((k - 1) & 1), kWaitNs))) {
                *abort_v = 1;
                break;
              }
              tc::fence_after_sync();
              issue(tmem + 256u * s + 128u * (sl & 1), s);
              tc::mma_commit(&tw_full[hb]);
              tc::mma_commit(&sl_empty);
            }
            tc::mma_commit(&x_empty[s]);
            continue;
          }
          if (!tc::mbar_wait(&x_full[s], (uint32_t)((g >> 1) & 1), kWaitNs) ||
              (g >= 2 && !tc::mbar_wait(&t_empty[s], (uint32_t)(((g >> 1) - 1) & 1), kWaitNs))) {
            *abort_v = 1;
            break;
          }
          tc::fence_after_sync();
          issue(tmem + 256u * s, s);
          tc::mma_commit(&x_empty[s]);
          tc::mma_commit(&t_full[s]);
        }
      }
    } else if (WIDE) {
      const int e = (warp - 2) >> 2, sub = warp & 3, row = 32 * sub + lane;
      const uint32_t lane_addr = (uint32_t)(32 * sub) << 16;
      for (int i = e; i < nt; i += 2) {
        const int64_t g = g_tile + i;
        const int s = (int)(g & 1);
        float b0 = INFINITY, b1 = INFINITY;  // even / odd columns
        int a0 = 0, a1 = 1;
        uint32_t r[32];
        bool bad = false;
#pragma unroll 1
        for (int sl = 0; sl < NSL; sl++) {
          const int64_t k = (g >> 1) * (NSL / 2) + (sl >> 1);
          const int hb = 2 * s + (sl & 1);
          const bool ok = tc::mbar_wait(&tw_full[hb], (uint32_t)(k & 1), kWaitNs);
          if (__any_sync(0xffffffffu, !ok || *abort_v != 0)) { bad = true; break; }  // warp-uniform
          tc::fence_after_sync();
#pragma unroll 1
          for (int c0 = 0; c0 < kSlice; c0 += 32) {
            tc::tmem_ld16(tmem + lane_addr + 256u * s + 128u * (sl & 1) + c0, r);
            tc::tmem_ld16(tmem + lane_addr + 256u * s + 128u * (sl & 1) + c0 + 16, r + 16);
            tc::tmem_ld_wait();
            const int j0 = sl * kSlice + c0;
#pragma unroll
            for (int kk = 0; kk < 32; kk += 2) {
              const float d0 = fmaf(-2.f, __uint_as_float(r[kk]), norm[j0 + kk]);
              const float d1 = fmaf(-2.f, __uint_as_float(r[kk + 1]), norm[j0 + kk + 1]);
              if (d0 < b0) { b0 = d0; a0 = j0 + kk; }
              if (d1 < b1) { b1 = d1; a1 = j0 + kk + 1; }
            }
          }
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&tw_empty[hb]);
        }
        if (bad) { *abort_v = 1; break; }
        asg16[i * TILE + row] = (uint16_t)((b1 < b0 || (b1 == b0 && a1 < a0)) ? a1 : a0);
      }
    } else {
      const int e = (warp - 2) >> 2, sub = warp & 3, row = 32 * sub + lane;
      const uint32_t lane_addr = (uint32_t)(32 * sub) << 16;
      for (int i = e; i < nt; i += 2) {
        const int64_t g = g_tile + i;
        const int s = (int)(g & 1);
        if (!tc::mbar_wait(&t_full[s], (uint32_t)((g >> 1) & 1), kWaitNs)) *abort_v = 1;
        if (*abort_v) break;
        tc::fence_after_sync();
        float b0 = INFINITY, b1 = INFINITY;  // even / odd columns
        int a0 = 0, a1 = 1;
        uint32_t r[32];
#pragma unroll 1
        for (int c0 = 0; c0 < C; c0 += 32) {
          tc::tmem_ld16(tmem + lane_addr + 256u * s + c0, r);
          tc::tmem_ld16(tmem + lane_addr + 256u * s + c0 + 16, r + 16);
          tc::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float d0 = fmaf(-2.f, __uint_as_float(r[k]), norm[c0 + k]);
            const float d1 = fmaf(-2.f, __uint_as_float(r[k + 1]), norm[c0 + k + 1]);
            if (d0 < b0) { b0 = d0; a0 = c0 + k; }
            if (d1 < b1) { b1 = d1; a1 = c0 + k + 1; }
          }
        }
        const int arg = (b1 < b0 || (b1 == b0 && a1 < a0)) ? a1 : a0;
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&t_empty[s]);
        asg[i * TILE + row] = (uint8_t)arg;
        const int64_t tok = (sc0 + i) * TILE + row;
        const bool tvalid = tok < p.n;
        if (delta) {  // the token's previous assignment; a half-tile with a change is re-read in phase 2
          const int old = tvalid ? (int)p.prev[(int64_t)h * p.n + tok] : arg;
          asg_old[i * TILE + row] = (uint8_t)old;
          const uint32_t moved = __ballot_sync(__activemask(), old != arg);
          if (lane == 0 && moved) atomicOr(tflag + i, 1u << (sub >> 1));
        }
        if (p.prev && tvalid) p.prev[(int64_t)h * p.n + tok] = (uint8_t)arg;
      }
    }
    __syncwarp();  // idle lanes of the TMA and MMA warps wait for lane 0 here
    __syncthreads();
    if (*abort_v) break;
    g_tile += nt;
    int nl = nt;  // tiles phase 2 re-reads: every tile, or (delta) those with a changed token
    if (delta) {
      if (tid == 0) {
        int c = 0;
        for (int i = 0; i < nt; i++)
          if (tflag[i]) tlist[c++] = i;
        nl_sh = c;
      }
      __syncthreads();
      nl = nl_sh;
      if (nl == 0) continue;  // no token of this super-chunk moved: its sums stand
    }
    if (WIDE) {
      // ---- phase 2 (WIDE): stable counting sort of the assignments, then per-centroid sums ----
      int32_t *cnt = (int32_t *)(sm + L.cnt), *cur = (int32_t *)(sm + L.cur);
      uint16_t *mem = (uint16_t *)(sm + L.mem);
      const int64_t tok0 = sc0 * TILE;
      const int64_t span = (int64_t)nt * TILE;
      const int ntok = nt == 0 ? 0 : (int)((p.n - tok0) < span ? (p.n - tok0) : span);
      for (int j = tid; j < C; j += kThreads) cnt[j] = 0;
      __syncthreads();
      for (int t = tid; t < ntok; t += kThreads) atomicAdd(cnt + asg16[t], 1);
      __syncthreads();
      if (warp == 0) {
        const int per = C / 32;  // lane l owns counts l * per .. l * per + per - 1
        int tot = 0;
        for (int q = 0; q < per; q++) tot += cnt[lane * per + q];
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        int run = incl - tot;  // exclusive prefix = where cluster j's members start
        for (int q = 0; q < per; q++) {
          cur[lane * per + q] = run;
          run += cnt[lane * per + q];
        }
        __syncwarp();
        const uint32_t below = (1u << lane) - 1u;
        for (int base = 0; base < ntok; base += 32) {  // tokens in order: a stable sort
          const int t = base + lane;
          const int j = t < ntok ? (int)asg16[t] : -1 - lane;  // past the end: a group of its own
          const uint32_t peers = __match_any_sync(0xffffffffu, j);
          const int pos = t < ntok ? cur[j] + __popc(peers & below) : 0;
          __syncwarp();
          if (t < ntok) {
            mem[pos] = (uint16_t)t;
            if ((peers & below) == 0) cur[j] += __popc(peers);  // the group's first lane moves the cursor
          }
          __syncwarp();
        }
      }
      __syncthreads();
      for (int j = warp; j < C; j += kThreads / 32) {  // one warp per centroid, lane = 4 channels
        const int nj = cnt[j], m0 = cur[j] - nj;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int m = 0; m < nj; m++) {
          const int t = mem[m0 + m];
          const uint2 v = *(const uint2 *)(p.x + ((int64_t)h * p.n + tok0 + t) * D + 4 * lane);
          a.x += __uint_as_float(v.x << 16);
          a.y += __uint_as_float(v.x & 0xFFFF0000u);
          a.z += __uint_as_float(v.y << 16);
          a.w += __uint_as_float(v.y & 0xFFFF0000u);
        }
        float4 *dst = (float4 *)(psum + (int64_t)j * D + 4 * lane);
        if (!first) {
          const float4 o = *dst;
          a.x += o.x; a.y += o.y; a.z += o.z; a.w += o.w;
        }
        *dst = a;
        if (lane == 0) pcnt[j] = first ? nj : pcnt[j] + nj;
      }
      __syncthreads();
      continue;
    }
    // ---- phase 2: cluster sums of this super-chunk on the tensor cores ----
    // sums[C][D] = A^T X accumulated over half-tiles of 64 tokens, A = the half-tile's one-hot
    // assignment matrix ([C][64 tokens] bf16, 1 where token t belongs to cluster j), X = the token
    // rows ([tokens][D], read as an N-major B operand); M = 128 centroids per MMA (two MMAs for
    // C = 256) into TMEM columns 0 .. C-1 (lane = centroid mod 128).  The one-hot matrices live in
    // kOneHot buffers at the start of the codebook area, each written by its own pair of warps, so
    // that building one half-tile's matrix overlaps the MMAs of the other; the token tiles stream
    // through the two token stages again (TMA) plus the stages that fit in the rest of the codebook
    // area (nxs in all: the re-read comes mostly from HBM, and a deeper ring hides its latency).
    constexpr int kOneHot = 3;
    const int Mb = (C + 127) / 128;                         // 128-centroid blocks
    const uint32_t aBytes = (uint32_t)Mb * TILE * 128u;     // one one-hot buffer: Mb x [128][64 tokens]
    constexpr uint32_t kStage = 2u * TILE * 128u;           // one token tile
    const int nxs_extra = L.x > (int)(kOneHot * aBytes) ? (int)(((uint32_t)L.x - kOneHot * aBytes) / kStage) : 0;
    const int nxs = 2 + (nxs_extra < 2 ? nxs_extra : 2);    // 2 to 4 token stages
    auto xstage = [&](int s) -> uint32_t {                   // byte offset of token stage s
      return s < 2 ? (uint32_t)L.x + (uint32_t)s * kStage : kOneHot * aBytes + (uint32_t)(s - 2) * kStage;
    };
    for (int e = tid; e < (int)(kOneHot * aBytes / 16u); e += kThreads) *(uint4 *)(sm + 16 * e) = make_uint4(0, 0, 0, 0);
    for (int j = tid; j < C; j += kThreads) cnts[j] = 0;
    if (tid < QWM_MAX_RESIDENT_CENTROIDS / 32) touched[tid] = 0u;
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    auto onehot_off = [&](int j, int t) -> uint32_t {  // byte offset of A[j][t] inside a buffer (t < 64)
      return (uint32_t)(j >> 7) * TILE * 128u + tc::sw128_offset(j & 127, t);
    };
    const int64_t u0 = 2 * g2;  // half-tiles before this super-chunk (barrier phases)
    if (warp == 0) {
      if (lane == 0) {  // TMA: token tiles
        for (int li = 0; li < nl && !*abort_v; li++) {
          const int i = delta ? tlist[li] : li;
          const int64_t g = g2 + li;
          const int s = (int)(g % nxs);
          if (g >= nxs && !tc::mbar_wait(&p2_empty[s], (uint32_t)(((g / nxs) - 1) & 1), kWaitNs)) {
            *abort_v = 1;
            break;
          }
          tc::mbar_arrive_expect_tx(&p2_full[s], 2 * TILE * 128);
          const int row = (int)((int64_t)h * p.n + (sc0 + i) * TILE);
          unsigned char *dst = sm + xstage(s);
          tc::tma_load_2d(dst, &tmap, 0, row, &p2_full[s]);
          tc::tma_load_2d(dst + TILE * 128, &tmap, 64, row, &p2_full[s]);
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {  // MMA: sums += A^T X
        const uint32_t idesc = tc::idesc_bf16_f32(TILE, D) | (1u << 16);  // B (token rows) N-major
        const uint32_t sa = tc::smem_u32(sm);
        for (int li = 0; li < nl && !*abort_v; li++) {
          const int64_t g = g2 + li;
          const int s = (int)(g % nxs);
          if (!tc::mbar_wait(&p2_full[s], (uint32_t)((g / nxs) & 1), kWaitNs)) { *abort_v = 1; break; }
          const uint32_t sx = sa + xstage(s);
          for (int hh = 0; hh < 2; hh++) {
            const int64_t U = u0 + 2 * li + hh;
            const int b = (int)(U % kOneHot);
            if (!tc::mbar_wait(&a_full[b], (uint32_t)((U / kOneHot) & 1), kWaitNs)) { *abort_v = 1; break; }
            tc::fence_after_sync();
            for (int mb = 0; mb < Mb; mb++) {
#pragma unroll
              for (int kk = 0; kk < 4; kk++) {  // 16 tokens per K step
                const uint32_t ao = sa + (uint32_t)b * aBytes + (uint32_t)mb * TILE * 128u + 32u * kk;
                const uint32_t bo = sx + 2048u * (4 * hh + kk);
                tc::mma_ss(tmem + 128u * mb, tc::desc_sw128(ao), tc::desc_sw128_mn(bo, TILE * 128, 1024), idesc,
                           (li > 0 || hh > 0 || kk > 0) ? 1u : 0u);
              }
            }
            tc::mma_commit(&a_empty[b]);
          }
          if (*abort_v) break;
          tc::mma_commit(&p2_empty[s]);
        }
        tc::mma_commit(&p2_done);
      }
    } else if (warp < 2 + 2 * kOneHot) {  // warp pair b builds the one-hot matrices of buffer b; thread = token
      const int b = (warp - 2) >> 1, lt = ((warp - 2) & 1) * 32 + lane;
      int u = (int)(((b - u0) % kOneHot + kOneHot) % kOneHot);  // this super-chunk's first half-tile in buffer b
      for (; u < 2 * nl; u += kOneHot) {
        const int64_t U = u0 + u;
        const bool ok = U < kOneHot || tc::mbar_wait(&a_empty[b], (uint32_t)(((U / kOneHot) - 1) & 1), kWaitNs);
        if (__any_sync(0xffffffffu, !ok || *abort_v != 0)) {  // warp-uniform exit
          *abort_v = 1;
          break;
        }
        unsigned char *abuf = sm + (uint32_t)b * aBytes;
        const int bt = 64 * (u & 1) + lt;                 // token within its tile
        if (u >= kOneHot) {  // clear this buffer's entries of its previous half-tile (same super-chunk)
          const int up = u - kOneHot;
          const int tp = delta ? tlist[up >> 1] : (up >> 1);
          const int64_t tokp = (sc0 + tp) * TILE;
          const int rowsp = (int)((p.n - tokp) < TILE ? (p.n - tokp) : TILE);
          const int btp = 64 * (up & 1) + lt;
          if (btp < rowsp) {
            const int jn = asg[tp * TILE + btp];
            if (!delta) {
              *(uint16_t *)(abuf + onehot_off(jn, lt)) = 0;
            } else if (asg_old[tp * TILE + btp] != jn) {
              *(uint16_t *)(abuf + onehot_off(jn, lt)) = 0;
              *(uint16_t *)(abuf + onehot_off(asg_old[tp * TILE + btp], lt)) = 0;
            }
          }
        }
        const int ti = delta ? tlist[u >> 1] : (u >> 1);
        const int64_t tok0 = (sc0 + ti) * TILE;
        const int rows = (int)((p.n - tok0) < TILE ? (p.n - tok0) : TILE);
        const bool valid = bt < rows;
        if (!delta) {  // +1 at the token's cluster
          const int j = valid ? asg[ti * TILE + bt] : -1 - lane;
          if (valid) *(uint16_t *)(abuf + onehot_off(j, lt)) = 0x3F80u;  // bf16 1.0
          const uint32_t peers = __match_any_sync(0xffffffffu, j);  // one count update per cluster
          if (valid && (peers & ((1u << lane) - 1u)) == 0) atomicAdd(cnts + j, __popc(peers));
        } else if (valid) {  // a moved token: +1 at its new cluster, -1 at its old one
          const int jn = asg[ti * TILE + bt], jo = asg_old[ti * TILE + bt];
          if (jn != jo) {
            *(uint16_t *)(abuf + onehot_off(jn, lt)) = 0x3F80u;  // bf16 1.0
            *(uint16_t *)(abuf + onehot_off(jo, lt)) = 0xBF80u;  // bf16 -1.0
            atomicAdd(cnts + jn, 1);
            atomicAdd(cnts + jo, -1);
            atomicOr(touched + (jn >> 5), 1u << (jn & 31));
            atomicOr(touched + (jo >> 5), 1u << (jo & 31));
          }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&a_full[b]);
      }
    }
    // the idle lanes of the TMA and MMA warps wait here for lane 0, not in the spin below: a lane
    // polling an mbarrier holds up the diverged lane 0 of its own warp
    __syncwarp();
    g2 += nl;
    if (!*abort_v && !tc::mbar_wait(&p2_done, (uint32_t)(n_sc & 1), kWaitNs)) *abort_v = 1;
    n_sc++;
    tc::fence_after_sync();
    __syncthreads();
    if (*abort_v) break;
    // sums from TMEM (warps 2-9: lane quarter warp % 4, centroid block (warp - 2) / 4) -> the workspace
    // (delta: only the centroids a moved token left or joined change)
    if (warp >= 2) {
      const int mb = (warp - 2) >> 2, sub = warp & 3;
      const int j = 128 * mb + 32 * sub + lane;
      const bool mine = !delta || ((touched[j >> 5] >> (j & 31)) & 1u);
      if (mb < Mb && __any_sync(0xffffffffu, mine)) {
        uint32_t r[32];
        for (int c0 = 0; c0 < D; c0 += 32) {
          tc::tmem_ld32(tmem + ((uint32_t)(32 * sub) << 16) + 128u * mb + c0, r);
          tc::tmem_ld_wait();
          if (j < C && mine) {
            float4 *dst = (float4 *)(psum + (int64_t)j * D + c0);
#pragma unroll
            for (int v = 0; v < 8; v++) {
              float4 a = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                     __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
              if (nt == 0) a = make_float4(0.f, 0.f, 0.f, 0.f);  // no tiles: no MMA wrote TMEM
              if (!first || delta) {
                const float4 o = dst[v];
                a.x += o.x; a.y += o.y; a.z += o.z; a.w += o.w;
              }
              dst[v] = a;
            }
          }
        }
      }
    }
    for (int j = tid; j < C; j += kThreads) pcnt[j] = (first && !delta) ? cnts[j] : pcnt[j] + cnts[j];
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  }
  // drain outstanding MMAs, then release TMEM
  if (warp == 1 && lane == 0) {
    tc::mma_commit(&drain);
    if (!tc::mbar_wait(&drain, 0, kWaitNs)) *abort_v = 1;
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

// New centroid = (sum of the G partial sums, in order) / count; empty clusters keep theirs.  Also
// writes the next assignment's operands (write_operand).  One block takes kUpd centroids of a head
// (thread = channel), with all their partial sums and counts loaded before the first is used.
constexpr int kUpd = 4;
__global__ void __launch_bounds__(D) km_update_kernel(int C, int G, float *__restrict__ cent,
                                                      const float *__restrict__ part_sum,
                                                      const int32_t *__restrict__ part_cnt,
                                                      uint16_t *__restrict__ out_bf16, unsigned char *__restrict__ img,
                                                      float *__restrict__ norms) {
  const int h = blockIdx.y, j0 = blockIdx.x * kUpd, c = threadIdx.x;
  float s[kUpd], old[kUpd];
  int cnt[kUpd];
#pragma unroll
  for (int u = 0; u < kUpd; u++) {
    s[u] = 0.f;
    cnt[u] = 0;
    old[u] = j0 + u < C ? cent[((int64_t)h * C + j0 + u) * D + c] : 0.f;
  }
  for (int g = 0; g < G; g++) {
#pragma unroll
    for (int u = 0; u < kUpd; u++) {
      if (j0 + u < C) {
        s[u] += part_sum[(((int64_t)h * G + g) * C + j0 + u) * D + c];
        cnt[u] += part_cnt[((int64_t)h * G + g) * C + j0 + u];
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kUpd; u++) {
    const int j = j0 + u;
    if (j >= C) break;  // block-uniform
    const int64_t e = ((int64_t)h * C + j) * D + c;
    float mu = old[u];
    if (cnt[u] > 0) mu = __fdiv_rn(s[u], (float)cnt[u]);  // counts are exact in fp32 (< 2^24)
    cent[e] = mu;
    if (out_bf16) {
      out_bf16[e] = f32_to_bf16_rn(mu);
    } else {
      write_operand(img + (int64_t)h * C * 512, norms + (int64_t)h * C, C, j, c, mu);
      __syncthreads();  // write_operand's norm buffer is read by thread 0 before the next centroid reuses it
    }
  }
}

}  // namespace

// CTAs per head: one wave at most (each CTA holds ~200 KB of shared memory).
int kmeans_ctas_per_head(int H, int num_sms) { return num_sms / H > 1 ? num_sms / H : 1; }

// Workspace of the operand images: [H] heads of C x 512 bytes, then the norms [H][C].
size_t kmeans_image_bytes(int H, int C) { return (size_t)H * C * 512 + (size_t)H * C * sizeof(float); }

cudaError_t launch_kmeans(const uint16_t *x, int64_t n, int H, int C, const uint16_t *init, int iters,
                          uint16_t *cent, float *km_cent, float *km_sum, int32_t *km_cnt, int num_sms,
                          int32_t *status, unsigned char *img, uint8_t *prev, int64_t prev_cap, cudaStream_t st) {
  TensorMap128 tmap;
  if (!make_tmap_rows128_bf16(&tmap, x, (uint64_t)H * n, TILE)) return cudaErrorInvalidValue;
  float *norms = (float *)(img + (size_t)H * C * 512);
  kmeans_init_kernel<<<dim3(C, H), D, 0, st>>>(x, n, C, init, km_cent, img, norms);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const bool wide = C > QWM_MAX_RESIDENT_CENTROIDS;
  const int G = kmeans_ctas_per_head(H, num_sms);
  const int smem = KmSmem(C, wide).total + 1024;
  e = wide ? cudaFuncSetAttribute(km_assign_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
           : cudaFuncSetAttribute(km_assign_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // Resident codebooks keep every token's assignment between iterations (when the chunk fits the
  // buffer): from the second iteration on, each CTA adds to its sums only the tokens that moved.
  uint8_t *keep = (!wide && prev && n <= prev_cap) ? prev : nullptr;
  AssignParams p{x, img, norms, km_sum, km_cnt, keep, n, C, G, 0, status};
  for (int it = 0; it < iters; it++) {
    p.delta = (keep && it > 0) ? 1 : 0;
    if (wide) km_assign_kernel<true><<<dim3(G, H), kThreads, smem, st>>>(tmap, p);
    else km_assign_kernel<false><<<dim3(G, H), kThreads, smem, st>>>(tmap, p);
    km_update_kernel<<<dim3((C + kUpd - 1) / kUpd, H), D, 0, st>>>(C, G, km_cent, km_sum, km_cnt,
                                                                    it == iters - 1 ? cent : nullptr, img, norms);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
