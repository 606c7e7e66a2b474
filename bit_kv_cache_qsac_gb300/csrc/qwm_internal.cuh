// Internal declarations shared by the CUDA translation units of libqwm.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qwm.h"

#define QWM_D 128          // head_dim supported by the kernels
#define QWM_GROUP 64       // INT2 group size supported by the kernels
#define QWM_MAX_RANK 16
#define QWM_MAX_TOPM 16
#define QWM_MAX_RESIDENT_CENTROIDS 256  // larger codebooks (1024) stream through in slices

// One k-means workspace: a fit's fp32 centroids, per-CTA cluster sums and counts, operand image and
// kept assignments.  A context holds two, so that a chunk's Key and Value fits can run side by side.
struct KmWorkspace {
  uint8_t *prev;       // [H][kKmPrevTokens] assignments between iterations (resident codebooks), else NULL
  float *sum;          // [H][G][C][d] per-CTA cluster sums (G CTAs per head)
  int32_t *cnt;        // [H][G][C] per-CTA cluster counts
  float *cent;         // [H][C][d] fp32 centroids during the iterations
  unsigned char *img;  // the assignment kernel's operand image (hi/lo bf16 blocks) and squared norms
};

struct qwm_ctx {
  qwm_config cfg;
  int device;
  int num_sms;
  // device workspace (one allocation)
  void *ws;
  size_t ws_bytes;
  int32_t *status;       // [1] first device-side error (qwm_status), 0 if none
  float *stats_part;     // [splits][H][d][d] per-split partial sums of q q^T
  int stats_splits;
  KmWorkspace km[2];     // k-means workspaces: [0] qwm_fit_centroids and the Key fit, [1] the Value fit
  unsigned char *q_img;  // 1024-centroid codebooks: quantiser operand slices + maxima
  float *q_bfull;        // full-form ranking: b_j = M mu_j [H][C][d]
  float *q_mfull;        // full-form ranking: M = S / n [H][d][d]
  // a second stream (and fork / join events) on which the Value fit of qwm_fit_centroids_kv and the
  // Value pass of qwm_quantize_kv run beside the Key ones; the caller's stream waits for it before
  // anything it issues next
  cudaStream_t side;
  cudaEvent_t fork, join;
};

// record the first device-side error (kernels call this; never traps)
__device__ __forceinline__ void qwm_dev_error(int32_t *status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float f16_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// INT2 encoder shared by the QuantWM quantiser and the KIVI-style baseline (affine, per group):
// m = fp16 round-down of min r, s = fp16 round-up of (max r - m)/3 (0 when max r == m),
// q = clamp(rint((r - m) * (1/s)), 0, 3), so |r - (m + s q)| <= s/2.
// INT2 parameters of one group from its fp32 residual min and max.
static __device__ __forceinline__ void int2_params(float mn, float mx, float &m, float &s, float &inv, uint16_t &m_bits,
                                            uint16_t &s_bits, int32_t *status) {
  const __half mh = __float2half_rd(mn);
  m = __half2float(mh);
  const float range = __fsub_ru(mx, m);
  __half sh = __float2half_ru(__fdiv_ru(range, 3.0f));
  if (range == 0.f) sh = __float2half_rn(0.f);
  s = __half2float(sh);
  if (!isfinite(m) || !isfinite(s)) qwm_dev_error(status, QWM_ERR_RANGE);
  inv = s > 0.f ? __frcp_rn(s) : 0.f;
  m_bits = __half_as_ushort(mh);
  s_bits = __half_as_ushort(sh);
}
static __device__ __forceinline__ uint32_t int2_code(float r, float m, float s, float inv) {
  if (s == 0.f) return 0u;
  float qf = rintf(__fmul_rn(__fsub_rn(r, m), inv));
  qf = fminf(fmaxf(qf, 0.f), 3.f);
  return (uint32_t)qf;
}

// Where token `tok` (of a chunk with `tiles` 128-token tiles) of head h keeps its PSAC row in a
// QWM_C_PER_HEAD chunk: false when it keeps none (a sparse head, scale zero); else `row` = its row
// index in the head's region (the token itself for a dense head; for a sparse head the rows stored
// before its tile plus the set bits of its tile's bitmap below it).
__device__ __forceinline__ bool psac_row(const qwm_psac_head &hd, const uint32_t *c_mask, const int32_t *c_tile_rank,
                                         int64_t tiles, int h, int64_t tok, int64_t &row) {
  row = tok;
  if (hd.rank == 0) return false;
  if (!hd.sparse) return true;
  const int64_t t = tok >> 7;
  const int b = (int)(tok & 127), w = b >> 5, bit = b & 31;
  const uint4 m4 = *(const uint4 *)(c_mask + ((int64_t)h * tiles + t) * 4);
  const uint32_t word = w == 0 ? m4.x : (w == 1 ? m4.y : (w == 2 ? m4.z : m4.w));
  if (!((word >> bit) & 1u)) return false;
  const int below = __popc(word & ((1u << bit) - 1u)) + (w > 0 ? __popc(m4.x) : 0) + (w > 1 ? __popc(m4.y) : 0) +
                    (w > 2 ? __popc(m4.z) : 0);
  row = (int64_t)c_tile_rank[(int64_t)h * tiles + t] + below;
  return true;
}

// TMA tensor map (a 128-byte-aligned 128-byte blob, CUtensorMap) over rows of 128 bf16.
struct alignas(128) TensorMap128 {
  unsigned char bytes[128];
};
bool make_tmap_rows128_bf16(void *tmap_out, const void *base, uint64_t rows, uint32_t box_rows);

// Launchers (each returns cudaGetLastError() of its launch).
cudaError_t launch_stats_partial(const uint16_t *q, int64_t nq, int H, float *part, int splits, int32_t *status,
                                 cudaStream_t st);
cudaError_t launch_stats_finish(const float *part, int splits, int64_t nq, int H, float *S, int64_t *n, float *w,
                                cudaStream_t st);
cudaError_t launch_eig(const float *S, int64_t *n, int64_t nq, int H, int rank, float *eigvals, uint16_t *u_r,
                       int32_t *status, cudaStream_t st);
#define QWM_MAX_SMS 192  // workspace sizing bound on the SM count
constexpr int64_t kKmPrevTokens = 65536;  // tokens per head whose k-means assignments the workspace keeps
int kmeans_ctas_per_head(int H, int num_sms);
size_t kmeans_image_bytes(int H, int C);
// kmeans `prev`: [H][prev_cap] bytes for the assignments kept between Lloyd iterations (resident
// codebooks; chunks longer than prev_cap tokens recompute every iteration's sums in full).
cudaError_t launch_kmeans(const uint16_t *x, int64_t n, int H, int C, const uint16_t *init, int iters,
                          uint16_t *cent, float *km_cent, float *km_sum, int32_t *km_cnt, int num_sms,
                          int32_t *status, unsigned char *img, uint8_t *prev, int64_t prev_cap, cudaStream_t st);
size_t quantize_image_bytes(int H, int C);
cudaError_t launch_quantize(const qwm_config &cfg, const uint16_t *k, const uint16_t *v, int64_t n,
                            const float *w, const float *S, const int64_t *n_seen, float *Mq, float *Bq,
                            const uint16_t *u_r, const qwm_chunk &out, const qwm_debug *dbg, int32_t *status,
                            int num_sms, unsigned char *img, cudaStream_t st, cudaStream_t side, cudaEvent_t fork,
                            cudaEvent_t join);
cudaError_t launch_attend(const qwm_config &cfg, const uint16_t *q, int64_t nq, const qwm_chunk *chunks,
                          int n_chunks, float scale, float *out, float *lse, int merge, int num_sms, int32_t *status,
                          cudaStream_t st);
cudaError_t launch_dequantize(const qwm_config &cfg, const qwm_chunk *chunks, int n_chunks, uint16_t *k_hat,
                              uint16_t *v_hat, cudaStream_t st);
cudaError_t launch_select_rank(const float *eigvals, float energy, int H, int R, uint16_t *u_r, int32_t *head_rank,
                               cudaStream_t st);
cudaError_t launch_psac_kept(const uint16_t *c_scale, int64_t n, int H, int32_t *kept, cudaStream_t st);
cudaError_t launch_psac_pack(const int8_t *c_dense, const uint16_t *s_dense, int64_t n, int H, int R,
                             const qwm_psac_head *plan, int8_t *c_out, uint16_t *s_out, uint32_t *c_mask,
                             int32_t *c_tile_rank, cudaStream_t st);
void psac_plan_host(int H, int64_t n, const int32_t *head_rank, const int32_t *kept, qwm_psac_head *plan,
                    int64_t *c_bytes, int64_t *n_scales);
