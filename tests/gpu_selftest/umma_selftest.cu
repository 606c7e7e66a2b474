// Self-test of the tcgen05 building blocks used by the attention kernel (tests only):
//   S = [A | A16] [B | B16]^T   (M = N = 128, K = 128 via two 128-byte-swizzled blocks + 16 via
//                                the no-swizzle layout), fp32 in tensor memory;
//   O = P V^T                   with P (bf16) stored into tensor memory over S's columns and
//                                used as the A operand from tensor memory;
//   O = P V                     (second kernel) with V stored [key][d] -- N contiguous -- and read
//                                as an MN-major, 128-byte-swizzled B operand;
//   the same two products on a CTA pair (third kernel, cta_group::2): M = 256 rows split over the
//   two CTAs, B's N columns split likewise, commits multicast to both CTAs.
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../bit_kv_cache_qsac_gb300/csrc/tc.cuh"

namespace {
constexpr int M = 128, N = 128, K = 128;
constexpr uint64_t kLimitNs = 1000000000ull;

__device__ void put_sw128(unsigned char *base, const __nv_bfloat16 *src, int rows, int ld) {
  // block b covers columns [64 b, 64 b + 64)
  for (int r = threadIdx.x; r < rows; r += blockDim.x)
    for (int k = 0; k < K; k++) {
      const int b = k / 64;
      *(__nv_bfloat16 *)(base + b * rows * 128 + tc::sw128_offset(r, k % 64)) = src[r * ld + k];
    }
}
__device__ void put_noswz16(unsigned char *base, const __nv_bfloat16 *src, int rows, int ld, int col0) {
  for (int r = threadIdx.x; r < rows; r += blockDim.x)
    for (int k = 0; k < 16; k++) *(__nv_bfloat16 *)(base + tc::noswz16_offset(r, k)) = src[r * ld + col0 + k];
}

__global__ void __launch_bounds__(128) umma_selftest_kernel(const __nv_bfloat16 *A, const __nv_bfloat16 *B,
                                                            const __nv_bfloat16 *P, const __nv_bfloat16 *Vt,
                                                            float *S_out, float *O_out, int *err) {
  extern __shared__ __align__(16) unsigned char sm_raw[];
  // 128-byte-swizzled tiles must start on a 1024-byte boundary
  unsigned char *sm = sm_raw + ((1024 - (tc::smem_u32(sm_raw) & 1023)) & 1023);
  unsigned char *sA = sm;                    // 2 x [128][64] swizzled = 32 KB
  unsigned char *sB = sA + 32768;            // 32 KB
  unsigned char *sV = sB + 32768;            // 32 KB
  unsigned char *sA16 = sV + 32768;          // 4 KB
  unsigned char *sB16 = sA16 + 4096;         // 4 KB
  __shared__ uint64_t bar[2];
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid / 32;
  put_sw128(sA, A, M, K + 16);
  put_sw128(sB, B, N, K + 16);
  put_sw128(sV, Vt, N, K);
  put_noswz16(sA16, A, M, K + 16, K);
  put_noswz16(sB16, B, N, K + 16, K);
  tc::fence_proxy_async_smem();
  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 256);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tS = tmem_base, tO = tmem_base + 128;
  const uint32_t idesc = tc::idesc_bf16_f32(M, N);
  if (tid == 0) {
    for (int kk = 0; kk < K / 16; kk++) {
      const int b = kk / 4, w = kk % 4;
      const uint64_t da = tc::desc_sw128(tc::smem_u32(sA + b * M * 128) + 32 * w);
      const uint64_t db = tc::desc_sw128(tc::smem_u32(sB + b * N * 128) + 32 * w);
      tc::mma_ss(tS, da, db, idesc, kk > 0);
    }
    tc::mma_ss(tS, tc::desc_noswz(tc::smem_u32(sA16), 128, 256), tc::desc_noswz(tc::smem_u32(sB16), 128, 256), idesc,
               1);
    tc::mma_commit(&bar[0]);
  }
  if (!tc::mbar_wait(&bar[0], 0, kLimitNs)) atomicExch(err, 1);
  tc::fence_after_sync();
  const uint32_t lane_addr = ((uint32_t)(32 * warp)) << 16;
  const int row = tid;
  uint32_t r[32];
  for (int c = 0; c < N; c += 32) {
    tc::tmem_ld32(tS + lane_addr + c, r);
    tc::tmem_ld_wait();
    for (int i = 0; i < 32; i++) S_out[row * N + c + i] = __uint_as_float(r[i]);
  }
  // P (bf16, 128 keys -> 64 columns) written over S
  for (int c = 0; c < 64; c += 16) {
    uint32_t pw[16];
    for (int i = 0; i < 16; i++) {
      const __nv_bfloat16 lo = P[row * K + 2 * (c + i)], hi = P[row * K + 2 * (c + i) + 1];
      pw[i] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
    }
    tc::tmem_st16(tS + lane_addr + c, pw);
  }
  tc::tmem_st_wait();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0) {
    for (int kk = 0; kk < K / 16; kk++) {
      const int b = kk / 4, w = kk % 4;
      const uint64_t dv = tc::desc_sw128(tc::smem_u32(sV + b * N * 128) + 32 * w);
      tc::mma_ts(tO, tS + 8 * kk, dv, idesc, kk > 0);
    }
    tc::mma_commit(&bar[1]);
  }
  if (!tc::mbar_wait(&bar[1], 0, kLimitNs)) atomicExch(err, 2);
  tc::fence_after_sync();
  for (int c = 0; c < N; c += 32) {
    tc::tmem_ld32(tO + lane_addr + c, r);
    tc::tmem_ld_wait();
    for (int i = 0; i < 32; i++) O_out[row * N + c + i] = __uint_as_float(r[i]);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem_base, 256);
}
// O = P V with V [128 keys][128 d] row-major: in shared memory as two [128 keys][64 d] swizzled
// blocks (d 0-63, d 64-127); K-step kk (16 keys) starts 16 rows = 2048 bytes further; the two
// 64-element N atoms are one block (16 KB) apart; 8-key groups are 1024 bytes apart.
__global__ void __launch_bounds__(128) umma_mn_selftest_kernel(const __nv_bfloat16 *P, const __nv_bfloat16 *V,
                                                               float *O_out, int *err) {
  extern __shared__ __align__(16) unsigned char sm_raw[];
  unsigned char *sm = sm_raw + ((1024 - (tc::smem_u32(sm_raw) & 1023)) & 1023);
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid / 32;
  put_sw128(sm, V, K, N);  // rows = keys, columns = d
  tc::fence_proxy_async_smem();
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 256);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tP = tmem_base, tO = tmem_base + 128;
  const uint32_t lane_addr = ((uint32_t)(32 * warp)) << 16;
  const int row = tid;
  for (int c = 0; c < 64; c += 16) {
    uint32_t pw[16];
    for (int i = 0; i < 16; i++) {
      const __nv_bfloat16 lo = P[row * K + 2 * (c + i)], hi = P[row * K + 2 * (c + i) + 1];
      pw[i] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
    }
    tc::tmem_st16(tP + lane_addr + c, pw);
  }
  tc::tmem_st_wait();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_bf16_f32(M, N) | (1u << 16);  // B MN-major
    for (int kk = 0; kk < K / 16; kk++)
      tc::mma_ts(tO, tP + 8 * kk, tc::desc_sw128_mn(tc::smem_u32(sm) + 2048u * kk, K * 128, 1024), idesc, kk > 0);
    tc::mma_commit(&bar);
  }
  if (!tc::mbar_wait(&bar, 0, kLimitNs)) atomicExch(err, 3);
  tc::fence_after_sync();
  uint32_t r[32];
  for (int c = 0; c < N; c += 32) {
    tc::tmem_ld32(tO + lane_addr + c, r);
    tc::tmem_ld_wait();
    for (int i = 0; i < 32; i++) O_out[row * N + c + i] = __uint_as_float(r[i]);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem_base, 256);
}
// Columns [c0, c0 + 64) of a row-major bf16 matrix -> one [rows][64] 128-byte-swizzled block.
__device__ void put_sw128_64(unsigned char *base, const __nv_bfloat16 *src, int rows, int ld, int c0) {
  for (int r = threadIdx.x; r < rows; r += blockDim.x)
    for (int k = 0; k < 64; k++) *(__nv_bfloat16 *)(base + tc::sw128_offset(r, k)) = src[r * ld + c0 + k];
}

// CTA pair: S[256][128] = A B^T (+ the 16-column no-swizzle part) with A rows 128 c .. 128 c + 127
// and B rows 64 c .. 64 c + 63 held by CTA c; O[256][128] = P V with P rows in each CTA's tensor
// memory and V's d columns 64 c .. 64 c + 63 held by CTA c (MN-major).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128)
    umma_pair_selftest_kernel(const __nv_bfloat16 *A, const __nv_bfloat16 *B, const __nv_bfloat16 *P,
                              const __nv_bfloat16 *V, float *S_out, float *O_out, int *err) {
  extern __shared__ __align__(16) unsigned char sm_raw[];
  unsigned char *sm = sm_raw + ((1024 - (tc::smem_u32(sm_raw) & 1023)) & 1023);
  unsigned char *sA = sm;             // 2 x [128][64] = 32 KB
  unsigned char *sB = sA + 32768;     // 2 x [64][64] = 16 KB
  unsigned char *sV = sB + 16384;     // [128 keys][64 d] = 16 KB
  unsigned char *sA16 = sV + 16384;   // [128][16] = 4 KB
  unsigned char *sB16 = sA16 + 4096;  // [64][16] = 2 KB
  __shared__ uint64_t bar_in, bar_s, bar_p, bar_o;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid / 32;
  const uint32_t rank = tc::cluster_ctarank();
  for (int b = 0; b < 2; b++) {
    put_sw128_64(sA + b * 16384, A + (size_t)128 * rank * (K + 16), 128, K + 16, 64 * b);
    put_sw128_64(sB + b * 8192, B + (size_t)64 * rank * (K + 16), 64, K + 16, 64 * b);
  }
  put_sw128_64(sV, V, 128, N, 64 * (int)rank);
  put_noswz16(sA16, A + (size_t)128 * rank * (K + 16), 128, K + 16, K);
  put_noswz16(sB16, B + (size_t)64 * rank * (K + 16), 64, K + 16, K);
  tc::fence_proxy_async_smem();
  if (tid == 0) {
    tc::mbar_init(&bar_in, 2);
    tc::mbar_init(&bar_s, 1);
    tc::mbar_init(&bar_p, 2);
    tc::mbar_init(&bar_o, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc2(&tmem_base, 256);
    tc::tmem_relinquish2();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // both CTAs' barriers exist before any arrival from the peer
  tc::fence_after_sync();
  const uint32_t tS = tmem_base, tO = tmem_base + 128;
  const uint32_t bar_in0 = tc::mapa(tc::smem_u32(&bar_in), 0), bar_p0 = tc::mapa(tc::smem_u32(&bar_p), 0);
  if (tid == 0) tc::mbar_arrive_remote(bar_in0);
  if (rank == 0 && tid == 0) {
    if (!tc::mbar_wait_cluster(&bar_in, 0, kLimitNs)) atomicExch(err, 11);
    tc::fence_after_sync();
    const uint32_t idesc = tc::idesc_bf16_f32(2 * M, N);
    for (int kk = 0; kk < K / 16; kk++) {
      const int b = kk / 4, w = kk % 4;
      tc::mma2_ss(tS, tc::desc_sw128(tc::smem_u32(sA + b * 16384) + 32 * w),
                  tc::desc_sw128(tc::smem_u32(sB + b * 8192) + 32 * w), idesc, kk > 0);
    }
    tc::mma2_ss(tS, tc::desc_noswz(tc::smem_u32(sA16), 128, 256), tc::desc_noswz(tc::smem_u32(sB16), 128, 256),
                idesc, 1);
    tc::mma2_commit(&bar_s, 3);
  }
  if (!tc::mbar_wait(&bar_s, 0, kLimitNs)) atomicExch(err, 12);
  tc::fence_after_sync();
  const uint32_t lane_addr = ((uint32_t)(32 * warp)) << 16;
  const int row = 128 * (int)rank + tid;
  uint32_t r[32];
  for (int c = 0; c < N; c += 32) {
    tc::tmem_ld32(tS + lane_addr + c, r);
    tc::tmem_ld_wait();
    for (int i = 0; i < 32; i++) S_out[row * N + c + i] = __uint_as_float(r[i]);
  }
  for (int c = 0; c < 64; c += 16) {  // P (bf16) over S
    uint32_t pw[16];
    for (int i = 0; i < 16; i++) {
      const __nv_bfloat16 lo = P[row * K + 2 * (c + i)], hi = P[row * K + 2 * (c + i) + 1];
      pw[i] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
    }
    tc::tmem_st16(tS + lane_addr + c, pw);
  }
  tc::tmem_st_wait();
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0) tc::mbar_arrive_remote(bar_p0);
  if (rank == 0 && tid == 0) {
    if (!tc::mbar_wait_cluster(&bar_p, 0, kLimitNs)) atomicExch(err, 13);
    tc::fence_after_sync();
    const uint32_t idesc = tc::idesc_bf16_f32(2 * M, N) | (1u << 16);  // B MN-major
    for (int kk = 0; kk < K / 16; kk++)
      tc::mma2_ts(tO, tS + 8 * kk, tc::desc_sw128_mn(tc::smem_u32(sV) + 2048u * kk, 16384, 1024), idesc, kk > 0);
    tc::mma2_commit(&bar_o, 3);
  }
  if (!tc::mbar_wait(&bar_o, 0, kLimitNs)) atomicExch(err, 14);
  tc::fence_after_sync();
  for (int c = 0; c < N; c += 32) {
    tc::tmem_ld32(tO + lane_addr + c, r);
    tc::tmem_ld_wait();
    for (int i = 0; i < 32; i++) O_out[row * N + c + i] = __uint_as_float(r[i]);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // the peer is done with this CTA's shared and tensor memory
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc2(tmem_base, 256);
}
}  // namespace

extern "C" int umma_pair_selftest(const void *A, const void *B, const void *P, const void *V, float *S, float *O,
                                  int *err) {
  const int smem = 32768 + 16384 + 16384 + 4096 + 2048 + 1024;
  if (cudaFuncSetAttribute(umma_pair_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -1;
  umma_pair_selftest_kernel<<<2, 128, smem>>>((const __nv_bfloat16 *)A, (const __nv_bfloat16 *)B,
                                              (const __nv_bfloat16 *)P, (const __nv_bfloat16 *)V, S, O, err);
  if (cudaGetLastError() != cudaSuccess) return -2;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}

extern "C" int umma_mn_selftest(const void *P, const void *V, float *O, int *err) {
  const int smem = 32768 + 1024;
  if (cudaFuncSetAttribute(umma_mn_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -1;
  umma_mn_selftest_kernel<<<1, 128, smem>>>((const __nv_bfloat16 *)P, (const __nv_bfloat16 *)V, O, err);
  if (cudaGetLastError() != cudaSuccess) return -2;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}

extern "C" int umma_selftest(const void *A, const void *B, const void *P, const void *Vt, float *S, float *O,
                             int *err) {
  const int smem = 3 * 32768 + 2 * 4096 + 1024;
  if (cudaFuncSetAttribute(umma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -1;
  umma_selftest_kernel<<<1, 128, smem>>>((const __nv_bfloat16 *)A, (const __nv_bfloat16 *)B,
                                         (const __nv_bfloat16 *)P, (const __nv_bfloat16 *)Vt, S, O, err);
  if (cudaGetLastError() != cudaSuccess) return -2;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}
