// Step 1: per-head Query second moment, channel weights and principal basis.
//
// QuantWM (Chinese summary, "二阶Query统计与低秩分解" and step (1); English v2 summary §D.1):
// the statistics are a running sum S_h = sum q q^T with a count N_h, kept without the
// Queries themselves; M_h = S_h / N_h, w_{h,c} = diag(M_h), and the principal basis
// U_r (top-r eigenvectors of M_h) is recomputed at every chunk boundary.
//
// Kernels:
//   stats_partial_kernel  grid (H, splits): each CTA sums q q^T over a slice of the
//                         Queries into a private fp32 partial (deterministic; no atomics).
//   stats_finish_kernel   adds the partials to S in a fixed order and writes w.
//   jacobi_kernel         one CTA per head: parallel cyclic Jacobi on the 128x128 M_h in
//                         shared memory (round-robin pairing, 64 disjoint rotations per
//                         round), then sort, sign convention, U_r to bf16.
#include "qwm_internal.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int kStatsThreads = 256;
constexpr int kStatsTok = 32;  // Queries staged in shared memory per pass

// Each thread owns an 8x8 block of the 128x128 output: rows 8*(t/16), columns 8*(t%16).
__global__ void __launch_bounds__(kStatsThreads) stats_partial_kernel(const uint16_t *__restrict__ q, int64_t nq,
                                                                      float *__restrict__ part, int splits) {
  __shared__ __align__(16) float qs[kStatsTok][D];
  const int h = blockIdx.x, sp = blockIdx.y, H = gridDim.x;
  const int tid = threadIdx.x;
  const int r0 = 8 * (tid / 16), c0 = 8 * (tid % 16);
  const int64_t per = (nq + splits - 1) / splits;
  const int64_t t0 = (int64_t)sp * per;
  const int64_t t1 = (t0 + per < nq) ? t0 + per : nq;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; i++)
#pragma unroll
    for (int j = 0; j < 8; j++) acc[i][j] = 0.f;
  const uint16_t *qh = q + (int64_t)h * nq * D;
  for (int64_t base = t0; base < t1; base += kStatsTok) {
    const int cnt = (t1 - base < kStatsTok) ? (int)(t1 - base) : kStatsTok;
    __syncthreads();
    for (int e = tid; e < kStatsTok * D / 2; e += kStatsThreads) {
      const int tok = (2 * e) / D, c = (2 * e) % D;
      uint32_t pair = 0;
      if (tok < cnt) pair = *(const uint32_t *)(qh + (base + tok) * D + c);
      qs[tok][c] = __uint_as_float(pair << 16);
      qs[tok][c + 1] = __uint_as_float(pair & 0xFFFF0000u);
    }
    __syncthreads();
    for (int tok = 0; tok < cnt; tok++) {
      float a[8], b[8];
      const float4 a0 = *(const float4 *)&qs[tok][r0], a1 = *(const float4 *)&qs[tok][r0 + 4];
      const float4 b0 = *(const float4 *)&qs[tok][c0], b1 = *(const float4 *)&qs[tok][c0 + 4];
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w; a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 8; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
  }
  float *out = part + ((int64_t)sp * H + h) * D * D;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    float4 *o = (float4 *)(out + (r0 + i) * D + c0);
    o[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    o[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
}

// S += sum of the partials (split order fixed); w_c = S_cc / (n + nq), or 1 when that count is 0.
__global__ void stats_finish_kernel(const float *__restrict__ part, int splits, int64_t nq, int H,
                                    float *__restrict__ S, const int64_t *__restrict__ n, float *__restrict__ w) {
  const int h = blockIdx.y;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= D * D) return;
  float s = S[(int64_t)h * D * D + e];
  for (int sp = 0; sp < splits; sp++) s += part[((int64_t)sp * H + h) * D * D + e];
  if (splits > 0) S[(int64_t)h * D * D + e] = s;
  const int r = e / D, c = e % D;
  if (r == c) {
    const int64_t nn = n[h] + nq;
    w[(int64_t)h * D + c] = nn > 0 ? (float)((double)s / (double)nn) : 1.0f;
  }
}

constexpr int kJacThreads = 512;
constexpr int LD = D + 1;  // padded row stride of the shared matrices
constexpr int NP = D / 2;  // disjoint pairs per round
constexpr int kMaxSweeps = 30;
constexpr float kRotTol = 1e-6f;  // rotate (p,q) while |a_pq| > tol * sqrt(|a_pp a_qq|)

__global__ void __launch_bounds__(kJacThreads) jacobi_kernel(const float *__restrict__ S, int64_t *__restrict__ n,
                                                             int64_t nq, int rank, float *__restrict__ eigvals,
                                                             uint16_t *__restrict__ u_r, int32_t *status) {
  extern __shared__ __align__(16) float jsm[];
  float *A = jsm;           // [D][LD]
  float *V = jsm + D * LD;  // [D][LD]
  __shared__ float cs[NP], sn[NP];
  __shared__ int pp[NP], qq[NP];
  __shared__ int order[D];
  __shared__ int rotated;
  const int h = blockIdx.x, tid = threadIdx.x;
  const int64_t nn = n[h] + nq;
  if (nn == 0) {  // cold start: no statistics yet
    for (int i = tid; i < D; i += kJacThreads) eigvals[(int64_t)h * D + i] = 0.f;
    for (int i = tid; i < D * rank; i += kJacThreads) u_r[(int64_t)h * D * rank + i] = 0;
    return;
  }
  const float inv = (float)(1.0 / (double)nn);
  for (int i = tid; i < D * D; i += kJacThreads) {
    const int r = i / D, c = i % D;
    A[r * LD + c] = S[(int64_t)h * D * D + i] * inv;
    V[r * LD + c] = (r == c) ? 1.f : 0.f;
  }
  __syncthreads();
  bool converged = false;
  for (int sweep = 0; sweep < kMaxSweeps; sweep++) {
    if (tid == 0) rotated = 0;
    __syncthreads();
    for (int round = 0; round < D - 1; round++) {
      if (tid < NP) {
        // round-robin ("circle") schedule: player D-1 is fixed, the others rotate
        int a, b;
        if (tid == 0) { a = D - 1; b = round; }
        else { a = (round + tid) % (D - 1); b = (round - tid + (D - 1)) % (D - 1); }
        const int p = min(a, b), qd = max(a, b);
        const float apq = A[p * LD + qd], app = A[p * LD + p], aqq = A[qd * LD + qd];
        float c = 1.f, s = 0.f;
        if (apq != 0.f && fabsf(apq) > kRotTol * sqrtf(fabsf(app * aqq))) {
          // Golub & Van Loan, sym.schur2: the rotation that diagonalises [[app, apq], [apq, aqq]]
          const float tau = (aqq - app) / (2.f * apq);
          const float t = (tau >= 0.f ? 1.f : -1.f) / (fabsf(tau) + sqrtf(1.f + tau * tau));
          c = rsqrtf(1.f + t * t);
          s = t * c;
          rotated = 1;
        }
        cs[tid] = c; sn[tid] = s; pp[tid] = p; qq[tid] = qd;
      }
      __syncthreads();
      // A <- L A L^T block by block: 2x2 block (P,R) becomes L_P B L_R^T, L = [[c,-s],[s,c]].
      for (int b = tid; b < NP * NP; b += kJacThreads) {
        const int P = b / NP, R = b % NP;
        if (P > R) continue;
        const float c1 = cs[P], s1 = sn[P], c2 = cs[R], s2 = sn[R];
        if (s1 == 0.f && s2 == 0.f) continue;
        const int p1 = pp[P], q1 = qq[P], p2 = pp[R], q2 = qq[R];
        const float b00 = A[p1 * LD + p2], b01 = A[p1 * LD + q2], b10 = A[q1 * LD + p2], b11 = A[q1 * LD + q2];
        const float t00 = c1 * b00 - s1 * b10, t01 = c1 * b01 - s1 * b11;
        const float t10 = s1 * b00 + c1 * b10, t11 = s1 * b01 + c1 * b11;
        const float n00 = c2 * t00 - s2 * t01, n01 = s2 * t00 + c2 * t01;
        const float n10 = c2 * t10 - s2 * t11, n11 = s2 * t10 + c2 * t11;
        if (P == R) {
          A[p1 * LD + p1] = n00;
          A[q1 * LD + q1] = n11;
          A[p1 * LD + q1] = 0.f;
          A[q1 * LD + p1] = 0.f;
        } else {
          A[p1 * LD + p2] = n00; A[p1 * LD + q2] = n01; A[q1 * LD + p2] = n10; A[q1 * LD + q2] = n11;
          A[p2 * LD + p1] = n00; A[q2 * LD + p1] = n01; A[p2 * LD + q1] = n10; A[q2 * LD + q1] = n11;
        }
      }
      // V <- V L^T (column pairs)
      for (int i = tid; i < D * NP; i += kJacThreads) {
        const int row = i / NP, P = i % NP;
        const float s = sn[P];
        if (s == 0.f) continue;
        const float c = cs[P];
        const int p = pp[P], qd = qq[P];
        const float vp = V[row * LD + p], vq = V[row * LD + qd];
        V[row * LD + p] = c * vp - s * vq;
        V[row * LD + qd] = s * vp + c * vq;
      }
      __syncthreads();
    }
    const bool none = (rotated == 0);
    __syncthreads();
    if (none) { converged = true; break; }
  }
  if (!converged && tid == 0) qwm_dev_error(status, QWM_ERR_NOT_CONVERGED);
  // descending order, ties to the lower index
  if (tid < D) {
    const float li = A[tid * LD + tid];
    int rk = 0;
    for (int j = 0; j < D; j++) {
      const float lj = A[j * LD + j];
      rk += (lj > li) || (lj == li && j < tid);
    }
    order[rk] = tid;
  }
  __syncthreads();
  if (tid < D) eigvals[(int64_t)h * D + tid] = A[order[tid] * LD + order[tid]];
  // top-r eigenvectors: largest-magnitude component made positive (lowest channel on ties)
  const int warp = tid / 32, lane = tid % 32;
  for (int k = warp; k < rank; k += kJacThreads / 32) {
    const int src = order[k];
    float best = -1.f;
    int arg = D;
    for (int c = lane; c < D; c += 32) {
      const float a = fabsf(V[c * LD + src]);
      if (a > best) { best = a; arg = c; }
    }
    for (int off = 16; off > 0; off >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int oa = __shfl_xor_sync(0xffffffffu, arg, off);
      if (ob > best || (ob == best && oa < arg)) { best = ob; arg = oa; }
    }
    const float sg = V[arg * LD + src] < 0.f ? -1.f : 1.f;
    for (int c = lane; c < D; c += 32) u_r[((int64_t)h * D + c) * rank + k] = f32_to_bf16_rn(sg * V[c * LD + src]);
  }
  if (tid == 0) n[h] = nn;
}

}  // namespace

cudaError_t launch_stats_partial(const uint16_t *q, int64_t nq, int H, float *part, int splits, cudaStream_t st) {
  stats_partial_kernel<<<dim3(H, splits), kStatsThreads, 0, st>>>(q, nq, part, splits);
  return cudaGetLastError();
}

cudaError_t launch_stats_finish(const float *part, int splits, int64_t nq, int H, float *S, int64_t *n, float *w,
                                cudaStream_t st) {
  stats_finish_kernel<<<dim3(D * D / 256, H), 256, 0, st>>>(part, splits, nq, H, S, n, w);
  return cudaGetLastError();
}

cudaError_t launch_jacobi(const float *S, int64_t *n, int64_t nq, int H, int rank, float *eigvals, uint16_t *u_r,
                          int32_t *status, cudaStream_t st) {
  // n is read here and advanced by n += nq at the end of each head's solve
  const size_t smem = 2 * D * LD * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(jacobi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  jacobi_kernel<<<H, kJacThreads, smem, st>>>(S, n, nq, rank, eigvals, u_r, status);
  return cudaGetLastError();
}
