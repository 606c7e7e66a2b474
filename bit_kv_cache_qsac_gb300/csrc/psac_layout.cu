// PSAC rank per (chunk, head) and the per-head coefficient layouts.
//
// Rank: the Chinese summary's critique (独立分析的弱点, weakness three) notes that the share of the
// Query energy held by the top directions differs by model and layer; the English v2 summary (§C.2)
// reports that a larger r still helps.  select_rank_kernel takes, per head, the smallest r_h whose
// top-r_h eigenvalues hold a given share of tr M and zeroes the basis columns past it, so the packing
// writes zero coefficients there.
// Layouts (English v2 summary §D.1: the smaller of a dense and a sparse coefficient layout, with
// sparse-index storage; Chinese summary step (4): C kept only where it lowers the Query-weighted
// error): a head's rows are stored for every token (dense) or only for the tokens whose scale is not
// zero (sparse), each row r_h bytes.  A sparse head's row of token i is found from a bitmap per
// 128-token tile and the count of rows before the tile: row = tile_rank[t] + (set bits below i).
#include "qwm_internal.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int kTile = 128;  // tokens per bitmap tile (four 32-bit words)

// One block per head: the rank rule in double precision (thread 0, the same sequential sums as a
// plain implementation), then the basis columns past r_h zeroed by the block.
__global__ void select_rank_kernel(const float *__restrict__ eigvals, float energy, int R, uint16_t *__restrict__ u_r,
                                   int32_t *__restrict__ head_rank) {
  __shared__ int rh;
  const int h = blockIdx.x;
  if (threadIdx.x == 0) {
    const float *lam = eigvals + (int64_t)h * D;
    double tr = 0.0;
    for (int k = 0; k < D; k++) tr += (double)lam[k];
    int r = R;
    if (!(tr > 0.0)) {
      r = 0;
    } else {
      const double target = (double)energy * tr;
      double cum = 0.0;
      for (int k = 0; k <= R; k++) {
        if (cum >= target) { r = k; break; }
        if (k < D) cum += (double)lam[k];
      }
    }
    rh = r;
    head_rank[h] = r;
  }
  __syncthreads();
  const int r = rh;
  for (int e = threadIdx.x; e < D * R; e += blockDim.x)
    if (e % R >= r) u_r[(int64_t)h * D * R + e] = 0;
}

// Tokens of head h with a non-zero PSAC scale.
__global__ void psac_kept_kernel(const uint16_t *__restrict__ c_scale, int64_t n, int32_t *__restrict__ kept) {
  __shared__ int part[8];
  const int h = blockIdx.x, tid = threadIdx.x;
  int cnt = 0;
  for (int64_t i = tid; i < n; i += blockDim.x) cnt += c_scale[(int64_t)h * n + i] != 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((tid & 31) == 0) part[tid >> 5] = cnt;
  __syncthreads();
  if (tid == 0) {
    int t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) t += part[w];
    kept[h] = t;
  }
}

// One block of 128 threads per head: tile by tile, thread = token; the bitmap words by warp ballots,
// the row of each stored token from the running count, the tile's count before it, and the warp
// prefix.  A dense head stores a row for every token (its bitmap marks every token).
__global__ void __launch_bounds__(kTile) psac_pack_kernel(const int8_t *__restrict__ c_dense,
                                                          const uint16_t *__restrict__ s_dense, int64_t n, int R,
                                                          const qwm_psac_head *__restrict__ plan,
                                                          int8_t *__restrict__ c_out, uint16_t *__restrict__ s_out,
                                                          uint32_t *__restrict__ c_mask,
                                                          int32_t *__restrict__ c_tile_rank) {
  __shared__ int warp_cnt[kTile / 32];
  const int h = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const qwm_psac_head hd = plan[h];
  const int64_t tiles = (n + kTile - 1) / kTile;
  int64_t running = 0;
  for (int64_t t = 0; t < tiles; t++) {
    const int64_t tok = t * kTile + tid;
    const int64_t gi = (int64_t)h * n + tok;
    const uint16_t sc = tok < n ? s_dense[gi] : (uint16_t)0;
    const bool has = tok < n && (hd.sparse == 0 || sc != 0);
    const uint32_t bal = __ballot_sync(0xffffffffu, has);
    if (lane == 0) {
      c_mask[(h * tiles + t) * 4 + warp] = bal;
      warp_cnt[warp] = __popc(bal);
    }
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kTile / 32; w++) {
      before += w < warp ? warp_cnt[w] : 0;
      total += warp_cnt[w];
    }
    if (tid == 0) c_tile_rank[h * tiles + t] = (int32_t)running;
    if (has && hd.rank > 0) {
      const int64_t row = running + before + __popc(bal & ((1u << lane) - 1u));
      const int8_t *src = c_dense + gi * R;
      int8_t *dst = c_out + hd.c_off + row * hd.rank;
      for (int k = 0; k < hd.rank; k++) dst[k] = src[k];
      s_out[hd.s_off + row] = sc;
    }
    running += total;
    __syncthreads();  // warp_cnt is rewritten by the next tile
  }
}

}  // namespace

cudaError_t launch_select_rank(const float *eigvals, float energy, int H, int R, uint16_t *u_r, int32_t *head_rank,
                               cudaStream_t st) {
  select_rank_kernel<<<H, 128, 0, st>>>(eigvals, energy, R, u_r, head_rank);
  return cudaGetLastError();
}

cudaError_t launch_psac_kept(const uint16_t *c_scale, int64_t n, int H, int32_t *kept, cudaStream_t st) {
  psac_kept_kernel<<<H, 256, 0, st>>>(c_scale, n, kept);
  return cudaGetLastError();
}

cudaError_t launch_psac_pack(const int8_t *c_dense, const uint16_t *s_dense, int64_t n, int H, int R,
                             const qwm_psac_head *plan, int8_t *c_out, uint16_t *s_out, uint32_t *c_mask,
                             int32_t *c_tile_rank, cudaStream_t st) {
  psac_pack_kernel<<<H, kTile, 0, st>>>(c_dense, s_dense, n, R, plan, c_out, s_out, c_mask, c_tile_rank);
  return cudaGetLastError();
}

// Host: the layout choice per head (the smaller of the two; dense on a tie; nothing for r_h = 0).
void psac_plan_host(int H, int64_t n, const int32_t *head_rank, const int32_t *kept, qwm_psac_head *plan,
                    int64_t *c_bytes, int64_t *n_scales) {
  const int64_t tiles = (n + kTile - 1) / kTile;
  int64_t cb = 0, ns = 0;
  for (int h = 0; h < H; h++) {
    const int64_t r = head_rank[h], k = kept[h];
    qwm_psac_head &p = plan[h];
    p.c_off = cb;
    p.s_off = ns;
    p.rank = (int32_t)r;
    p.sparse = 0;
    if (r == 0) continue;
    const int64_t dense = n * (r + 2), sparse = k * (r + 2) + tiles * 20;
    p.sparse = sparse < dense ? 1 : 0;
    const int64_t rows = p.sparse ? k : n;
    cb += rows * r;
    ns += rows;
  }
  if (c_bytes) *c_bytes = cb;
  if (n_scales) *n_scales = ns;
}
