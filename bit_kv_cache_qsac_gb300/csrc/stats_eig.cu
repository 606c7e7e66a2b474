// Step 1: per-head Query second moment, channel weights and principal basis.
//
// QuantWM (Chinese summary, "二阶Query统计与低秩分解" and step (1); English v2 summary §D.1):
// the statistics are a running sum S_h = sum q q^T with a count N_h, kept without the
// Queries themselves; M_h = S_h / N_h, w_{h,c} = diag(M_h), and the principal basis
// U_r (top-r eigenvectors of M_h) is recomputed at every chunk boundary.
//
// Kernels:
//   stats_partial_kernel  grid (splits, H): each CTA sums q q^T over a slice of the Queries
//                         on the tensor cores into a private fp32 partial (no atomics).
//   stats_finish_kernel   adds the partials to S in a fixed order and writes w.
//   jacobi_kernel         one CTA per head: parallel cyclic Jacobi on the 128x128 M_h in
//                         shared memory (round-robin pairing, 64 disjoint rotations per
//                         round), then sort, sign convention, U_r to bf16.
#include "qwm_internal.cuh"
#include "tc.cuh"

namespace {

constexpr int D = QWM_D;
constexpr int kStatsThreads = 128;
constexpr int kStatsTile = 128;  // Queries per MMA (the K dimension of S += Q^T Q)
constexpr uint64_t kWaitNs = 1000000000ull;

// S_part = sum over this CTA's Queries of q q^T on the tensor cores.  Each 128-Query tile is
// written transposed into shared memory ([128 channels][128 Queries], 128-byte swizzle, K-major
// with K = Queries), and the same tile serves as both operands: D[c1][c2] += sum_t Q[t][c1] Q[t][c2].
// grid (splits, H); the CTA's partial goes to part[split][h] (no atomics: deterministic).
__global__ void __launch_bounds__(kStatsThreads, 1) stats_partial_kernel(const uint16_t *__restrict__ q, int64_t nq,
                                                                          float *__restrict__ part, int splits,
                                                                          int32_t *status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char *sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t done[2], fin;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  const int h = blockIdx.y, sp = blockIdx.x, H = gridDim.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t tiles = (nq + kStatsTile - 1) / kStatsTile;
  const int64_t per = (tiles + splits - 1) / splits;
  const int64_t t0 = (int64_t)sp * per;
  const int64_t t1 = t0 + per < tiles ? t0 + per : tiles;
  const int nt = t1 > t0 ? (int)(t1 - t0) : 0;
  if (tid == 0) {
    tc::mbar_init(&done[0], 1);
    tc::mbar_init(&done[1], 1);
    tc::mbar_init(&fin, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 128);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const uint16_t *qh = q + (int64_t)h * nq * D;
  const uint32_t idesc = tc::idesc_bf16_f32(128, 128);
  for (int i = 0; i < nt; i++) {
    const int s = i & 1;
    if (i >= 2 && !tc::mbar_wait(&done[s], ((i >> 1) - 1) & 1, kWaitNs)) abort_flag = 1;
    __syncthreads();
    if (abort_flag) break;
    unsigned char *stage = sm + s * 32768;
    const int64_t base = (t0 + i) * kStatsTile;
    // item = (Query pair, 8-channel block): 64 x 16 items, 8 per thread
    for (int it = tid; it < 64 * 16; it += kStatsThreads) {
      const int pr = it & 63, cb = it >> 6;
      const int64_t ta = base + 2 * pr, tb = ta + 1;
      uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
      if (ta < nq) a = *(const uint4 *)(qh + ta * D + 8 * cb);
      if (tb < nq) b = *(const uint4 *)(qh + tb * D + 8 * cb);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
      const int blk = (2 * pr) / 64, kin = (2 * pr) % 64;
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const uint32_t sel = (u & 1) ? 0x7632u : 0x5410u;
        const uint32_t word = __byte_perm(aw[u >> 1], bw[u >> 1], sel);  // (Query ta, Query tb) of channel 8cb+u
        *(uint32_t *)(stage + blk * 16384 + tc::sw128_offset(8 * cb + u, kin)) = word;
      }
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      const uint32_t sa = tc::smem_u32(stage);
#pragma unroll
      for (int kk = 0; kk < kStatsTile / 16; kk++) {
        const uint64_t dsc = tc::desc_sw128(sa + (kk / 4) * 16384 + 32 * (kk % 4));
        tc::mma_ss(tmem, dsc, dsc, idesc, (i > 0 || kk > 0) ? 1u : 0u);
      }
      tc::mma_commit(&done[s]);
    }
  }
  if (tid == 0) tc::mma_commit(&fin);
  const bool ok = !abort_flag && tc::mbar_wait(&fin, 0, kWaitNs);
  if (!ok && tid == 0) qwm_dev_error(status, QWM_ERR_DEVICE_TIMEOUT);
  tc::fence_after_sync();
  float *out = part + ((int64_t)sp * H + h) * D * D;
  const int row = tid;  // channel c1 = TMEM lane
  const uint32_t lane_addr = (uint32_t)(32 * warp) << 16;
  uint32_t r[32];
  for (int c0 = 0; c0 < D; c0 += 32) {
    tc::tmem_ld32(tmem + lane_addr + c0, r);
    tc::tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 32; k += 4) {
      const bool any = ok && nt > 0;
      *(float4 *)(out + row * D + c0 + k) =
          any ? make_float4(__uint_as_float(r[k]), __uint_as_float(r[k + 1]), __uint_as_float(r[k + 2]),
                            __uint_as_float(r[k + 3]))
              : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 128);
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
constexpr int LD = D + 4;  // padded row stride of the shared matrices (16-byte aligned rows)
constexpr int NP = D / 2;  // disjoint pairs per round
constexpr int kMaxSweeps = 30;
// rotate (p,q) while |a_pq| > kRotTol sqrt(|a_pp a_qq|) ...: a left-over off-diagonal entry at
// that level moves an eigenvalue by at most about 1e-5 of its size (the noise eigenvalues form a
// near-degenerate cluster, where the move is first order) and a well-separated eigenvector by
// far less
constexpr float kRotTol = 1e-5f;
constexpr float kAbsTol = 1.2e-7f;  // ... and |a_pq| > kAbsTol ||A||_F (fp32 rounding level of A)

// C = op(X) Y for 128x128 shared matrices (row stride LD), op(X) = X or X^T; 512 threads, each
// owning an 8x4 block of C.
__device__ __forceinline__ void smem_gemm128(const float *X, bool transX, const float *Y, float *Cm) {
  const int tid = threadIdx.x, ty = tid / 32, tx = tid % 32;
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; i++)
#pragma unroll
    for (int j = 0; j < 4; j++) acc[i][j] = 0.f;
  for (int k = 0; k < D; k++) {
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; i++) a[i] = transX ? X[k * LD + 8 * ty + i] : X[(8 * ty + i) * LD + k];
    const float4 b = *(const float4 *)(Y + k * LD + 4 * tx);
#pragma unroll
    for (int i = 0; i < 8; i++) {
      acc[i][0] = fmaf(a[i], b.x, acc[i][0]);
      acc[i][1] = fmaf(a[i], b.y, acc[i][1]);
      acc[i][2] = fmaf(a[i], b.z, acc[i][2]);
      acc[i][3] = fmaf(a[i], b.w, acc[i][3]);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; i++)
    *(float4 *)(Cm + (8 * ty + i) * LD + 4 * tx) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
}

// basis: [H][D][D] fp32 workspace holding each head's last full eigenbasis (columns sorted),
// valid: [H] flags.  When valid, the rotations start from that basis: A = U^T M U is nearly
// diagonal when the statistics moved little since the previous chunk, so few sweeps are needed.
__global__ void __launch_bounds__(kJacThreads) jacobi_kernel(const float *__restrict__ S, int64_t *__restrict__ n,
                                                             int64_t nq, int rank, float *__restrict__ eigvals,
                                                             uint16_t *__restrict__ u_r, int32_t *status,
                                                             float *__restrict__ basis, int32_t *__restrict__ valid) {
  extern __shared__ __align__(16) float jsm[];
  float *A = jsm;               // [D][LD]
  float *V = jsm + D * LD;      // [D][LD]
  float *T = jsm + 2 * D * LD;  // [D][LD] scratch for the warm start
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
  const bool warm = valid[h] != 0;
  float *Bh = basis + (int64_t)h * D * D;
  for (int i = tid; i < D * D; i += kJacThreads) {
    const int r = i / D, c = i % D;
    A[r * LD + c] = S[(int64_t)h * D * D + i] * inv;
    V[r * LD + c] = warm ? Bh[i] : ((r == c) ? 1.f : 0.f);
  }
  __syncthreads();
  if (warm) {  // A <- V^T A V, symmetrised
    smem_gemm128(A, false, V, T);
    __syncthreads();
    smem_gemm128(V, true, T, A);
    __syncthreads();
    for (int i = tid; i < D * D; i += kJacThreads) {
      const int r = i / D, c = i % D;
      if (r < c) {
        const float m = 0.5f * (A[r * LD + c] + A[c * LD + r]);
        A[r * LD + c] = m;
        A[c * LD + r] = m;
      }
    }
    __syncthreads();
  }
  // ||A||_F, reduced in a fixed order: off-diagonal entries at the rounding level of A carry no
  // information and would otherwise keep the sweeps going on rotation noise
  __shared__ float fro_part[kJacThreads / 32];
  __shared__ float abs_tol;
  {
    float f = 0.f;
    for (int i = tid; i < D * D; i += kJacThreads) {
      const float a = A[(i / D) * LD + i % D];
      f = fmaf(a, a, f);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) f += __shfl_xor_sync(0xffffffffu, f, o);
    if ((tid & 31) == 0) fro_part[tid / 32] = f;
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < kJacThreads / 32; w++) t += fro_part[w];
      abs_tol = kAbsTol * sqrtf(t);
    }
    __syncthreads();
  }
  const float atol = abs_tol;
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
        if (fabsf(apq) > atol && fabsf(apq) > kRotTol * sqrtf(fabsf(app * aqq))) {
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
  // full basis, sorted and sign-fixed like u_r, for the next call's warm start
  for (int k = warp; k < D; k += kJacThreads / 32) {
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
    for (int c = lane; c < D; c += 32) Bh[c * D + k] = sg * V[c * LD + src];
  }
  if (tid == 0) {
    valid[h] = 1;
    n[h] = nn;
  }
}

}  // namespace

cudaError_t launch_stats_partial(const uint16_t *q, int64_t nq, int H, float *part, int splits, int32_t *status,
                                 cudaStream_t st) {
  const int smem = 2 * 32768 + 1024;
  cudaError_t e = cudaFuncSetAttribute(stats_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  stats_partial_kernel<<<dim3(splits, H), kStatsThreads, smem, st>>>(q, nq, part, splits, status);
  return cudaGetLastError();
}

cudaError_t launch_stats_finish(const float *part, int splits, int64_t nq, int H, float *S, int64_t *n, float *w,
                                cudaStream_t st) {
  stats_finish_kernel<<<dim3(D * D / 256, H), 256, 0, st>>>(part, splits, nq, H, S, n, w);
  return cudaGetLastError();
}

cudaError_t launch_jacobi(const float *S, int64_t *n, int64_t nq, int H, int rank, float *eigvals, uint16_t *u_r,
                          int32_t *status, float *basis, int32_t *valid, cudaStream_t st) {
  // n is read here and advanced by n += nq at the end of each head's solve
  const size_t smem = 3 * D * LD * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(jacobi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  jacobi_kernel<<<H, kJacThreads, smem, st>>>(S, n, nq, rank, eigvals, u_r, status, basis, valid);
  return cudaGetLastError();
}
