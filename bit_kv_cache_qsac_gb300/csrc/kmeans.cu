// Step 2a: per-head Lloyd k-means codebook of one chunk.
//
// QVG summary §2A: tokens are grouped by k-means along the sequence axis and each
// token is represented by its centroid plus a residual; §2C: the k-means of a new
// chunk starts from the previous chunk's centroids (warm start).  Every Lloyd
// iteration assigns each token to its nearest centroid (Euclidean, lower index on
// ties) and replaces each centroid by the mean of its members; a centroid left
// without members keeps its position.  Centroids stay fp32 between iterations and
// are rounded to bf16 at the end.
//
// Kernels: kmeans_init_kernel (starting centroids), kmeans_assign_kernel (one warp per
// token, exact fp32 distances against the fp32 codebook held transposed in shared
// memory; cluster sums by fp32 atomics), kmeans_update_kernel (means; clears sums).
#include "qwm_internal.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int kAssignThreads = 256;

__global__ void kmeans_init_kernel(const uint16_t *__restrict__ x, int64_t n, int C, const uint16_t *__restrict__ init,
                                   float *__restrict__ cent, float *__restrict__ sum, int32_t *__restrict__ cnt) {
  const int h = blockIdx.y, j = blockIdx.x, c = threadIdx.x;
  const uint16_t *src = init ? init + ((int64_t)h * C + j) * D : x + ((int64_t)h * n + (int64_t)j * n / C) * D;
  cent[((int64_t)h * C + j) * D + c] = bf16_to_f32(src[c]);
  sum[((int64_t)h * C + j) * D + c] = 0.f;
  if (c == 0) cnt[(int64_t)h * C + j] = 0;
}

// grid (ceil(n / tokens_per_cta), H); dynamic smem: centroids transposed [D][C] fp32
__global__ void __launch_bounds__(kAssignThreads) kmeans_assign_kernel(const uint16_t *__restrict__ x, int64_t n,
                                                                       int C, const float *__restrict__ cent,
                                                                       float *__restrict__ sum,
                                                                       int32_t *__restrict__ cnt, int tok_per_cta) {
  extern __shared__ __align__(16) float ksm[];
  float *cT = ksm;  // [D][C]
  __shared__ float tokbuf[kAssignThreads / 32][D];
  const int h = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float *ch = cent + (int64_t)h * C * D;
  for (int e = threadIdx.x; e < C * (D / 4); e += kAssignThreads) {  // lanes write consecutive centroids
    const int j = e % C, cb = e / C;
    const float4 a = *(const float4 *)(ch + (int64_t)j * D + 4 * cb);
    cT[(4 * cb + 0) * C + j] = a.x;
    cT[(4 * cb + 1) * C + j] = a.y;
    cT[(4 * cb + 2) * C + j] = a.z;
    cT[(4 * cb + 3) * C + j] = a.w;
  }
  __syncthreads();
  const int per_lane = C / 32;  // 2, 4 or 8
  const int64_t t_begin = (int64_t)blockIdx.x * tok_per_cta;
  const int64_t t_end = min(n, t_begin + tok_per_cta);
  for (int64_t i = t_begin + warp; i < t_end; i += kAssignThreads / 32) {
    const uint16_t *xi = x + ((int64_t)h * n + i) * D;
    const uint2 raw = *(const uint2 *)(xi + 4 * lane);
    float xv[4];
    xv[0] = __uint_as_float(raw.x << 16); xv[1] = __uint_as_float(raw.x & 0xFFFF0000u);
    xv[2] = __uint_as_float(raw.y << 16); xv[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 4; u++) tokbuf[warp][4 * lane + u] = xv[u];
    __syncwarp();
    float dist[8];
#pragma unroll
    for (int t = 0; t < 8; t++) dist[t] = 0.f;
    for (int c = 0; c < D; c++) {
      const float xc = tokbuf[warp][c];
#pragma unroll
      for (int t = 0; t < 8; t++) {
        if (t < per_lane) {
          const float df = __fsub_rn(xc, cT[c * C + lane + 32 * t]);
          dist[t] = __fmaf_rn(df, df, dist[t]);
        }
      }
    }
    // argmin over the warp (centroid j = lane + 32 t), lower index on ties
    float best = dist[0];
    int arg = lane;
#pragma unroll
    for (int t = 1; t < 8; t++)
      if (t < per_lane && dist[t] < best) { best = dist[t]; arg = lane + 32 * t; }
    for (int off = 16; off > 0; off >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int oa = __shfl_xor_sync(0xffffffffu, arg, off);
      if (ob < best || (ob == best && oa < arg)) { best = ob; arg = oa; }
    }
    float *sj = sum + ((int64_t)h * C + arg) * D + 4 * lane;
#pragma unroll
    for (int u = 0; u < 4; u++) atomicAdd(sj + u, xv[u]);
    if (lane == 0) atomicAdd(cnt + (int64_t)h * C + arg, 1);
  }
}

__global__ void kmeans_update_kernel(int C, float *__restrict__ cent, float *__restrict__ sum, int32_t *__restrict__ cnt,
                                     uint16_t *__restrict__ out_bf16) {
  const int h = blockIdx.y, j = blockIdx.x, c = threadIdx.x;
  const int64_t e = ((int64_t)h * C + j) * D + c;
  const int m = cnt[(int64_t)h * C + j];
  float mu = cent[e];
  if (m > 0) mu = (float)((double)sum[e] / (double)m);
  cent[e] = mu;
  sum[e] = 0.f;
  __syncthreads();
  if (c == 0) cnt[(int64_t)h * C + j] = 0;
  if (out_bf16) out_bf16[e] = f32_to_bf16_rn(mu);
}

}  // namespace

cudaError_t launch_kmeans(const uint16_t *x, int64_t n, int H, int C, const uint16_t *init, int iters,
                          uint16_t *cent, float *km_cent, float *km_sum, int32_t *km_cnt, int num_sms,
                          cudaStream_t st) {
  kmeans_init_kernel<<<dim3(C, H), D, 0, st>>>(x, n, C, init, km_cent, km_sum, km_cnt);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)C * D * sizeof(float);
  e = cudaFuncSetAttribute(kmeans_assign_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // enough CTAs to cover the SMs about twice
  int64_t blocks_per_head = (2LL * num_sms + H - 1) / H;
  int tok_per_cta = (int)((n + blocks_per_head - 1) / blocks_per_head);
  if (tok_per_cta < 64) tok_per_cta = 64;
  const int gx = (int)((n + tok_per_cta - 1) / tok_per_cta);
  for (int it = 0; it < iters; it++) {
    kmeans_assign_kernel<<<dim3(gx, H), kAssignThreads, smem, st>>>(x, n, C, km_cent, km_sum, km_cnt, tok_per_cta);
    kmeans_update_kernel<<<dim3(C, H), D, 0, st>>>(C, km_cent, km_sum, km_cnt, it == iters - 1 ? cent : nullptr);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
