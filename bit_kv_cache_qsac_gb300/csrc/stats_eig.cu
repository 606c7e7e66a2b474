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
//   eig_kernel            one CTA per head: Householder tridiagonalisation of M_h in shared
//                         memory, all eigenvalues by multisection on Sturm counts, the top-r
//                         eigenvectors by inverse iteration and back-transformation, sign
//                         convention, U_r to bf16.
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
  const int tid = threadIdx.x, warp = tid >> 5;
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

constexpr int kEigThreads = 512;
constexpr int LDA = D + 1;     // odd row stride: conflict-free row and column access
constexpr int kRounds = 14;    // multisection rounds: the Gershgorin interval shrinks 5x per round
constexpr int LU = 4 * D + 1;  // per-vector scratch of the tridiagonal solve (padded across banks)

__device__ __forceinline__ float warp_sum_f(float s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// Deterministic start vector of inverse iteration k (entries in [-0.5, 0.5)): a different vector per
// k, so that eigenvalues closer than the solve can separate still give independent vectors.
__device__ __forceinline__ float start_entry(int i, int k) {
  uint32_t x = (uint32_t)(i + 1) * 2654435761u ^ (uint32_t)(k + 1) * 40503u;
  x ^= x >> 15; x *= 2246822519u; x ^= x >> 13; x *= 3266489917u; x ^= x >> 16;
  return (float)(x >> 8) * (1.0f / 16777216.0f) - 0.5f;
}

// One CTA per head.  Eigenvalues of M = S / n, descending, and the top-r eigenvectors:
//  1. Householder reduction of M to a symmetric tridiagonal T = Q^T M Q (Golub & Van Loan,
//     Algorithm 8.3.1, with the reflector of Algorithm 5.1.1): 126 reflections in shared memory;
//     reflector k is kept in row k of the matrix for step 4.
//  2. Every eigenvalue of T by multisection on Sturm counts (the number of negative pivots of
//     T - x I): four threads per eigenvalue test four interior points per round.
//  3. Inverse iteration on T for each of the r largest eigenvalues (two solves with partial
//     pivoting, each from its own start vector; the back-substitution rescales the system when
//     near-zero pivots of a repeated eigenvalue make it grow), then modified Gram-Schmidt within
//     clusters of eigenvalues closer than 1e-3 ||T||.
//  4. Back-transformation u = Q z (one warp per vector) and the sign convention: the largest-
//     magnitude component is made positive, the lowest channel on ties.
__global__ void __launch_bounds__(kEigThreads) eig_kernel(const float *__restrict__ S, int64_t *__restrict__ n,
                                                          int64_t nq, int rank, float *__restrict__ eigvals,
                                                          uint16_t *__restrict__ u_r, int32_t *status) {
  extern __shared__ __align__(16) float esm[];
  float *A = esm;                    // [D][LDA]
  float *lu = A + D * LDA;           // [QWM_MAX_RANK][LU]: solve scratch, then the vectors z
  __shared__ float dg[D], e2[D], ev[D], tau[D], vv[D], pv[D], wv[D], lam[D];
  __shared__ float sc[4];            // tau_k, 1 / v0, K; Gershgorin and pivot bounds below
  __shared__ float gs[3];
  __shared__ int bad;
  const int h = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t nn = n[h] + nq;
  if (nn == 0) {  // cold start: no statistics yet
    for (int i = tid; i < D; i += kEigThreads) eigvals[(int64_t)h * D + i] = 0.f;
    for (int i = tid; i < D * rank; i += kEigThreads) u_r[(int64_t)h * D * rank + i] = 0;
    return;
  }
  const float inv = (float)(1.0 / (double)nn);
  for (int i = tid; i < D * D; i += kEigThreads) A[(i / D) * LDA + i % D] = S[(int64_t)h * D * D + i] * inv;
  if (tid == 0) bad = 0;
  __syncthreads();

  // ---- 1. tridiagonalisation ----
  for (int k = 0; k < D - 2; k++) {
    const int m = D - 1 - k;  // length of the column below the diagonal
    const float *xk = A + k * LDA + k + 1;
    if (warp == 0) {
      float sg = 0.f;
      for (int j = 1 + lane; j < m; j += 32) sg = fmaf(xk[j], xk[j], sg);
      sg = warp_sum_f(sg);
      if (lane == 0) {
        const float x0 = xk[0];
        dg[k] = A[k * LDA + k];
        if (sg == 0.f) {  // already reduced: no reflection
          sc[0] = 0.f; sc[1] = 0.f; ev[k] = x0;
        } else {
          const float mu = sqrtf(fmaf(x0, x0, sg));
          const float v0 = x0 <= 0.f ? x0 - mu : -sg / (x0 + mu);
          sc[0] = 2.f * v0 * v0 / (sg + v0 * v0);
          sc[1] = 1.f / v0;
          ev[k] = mu;
        }
        tau[k] = sc[0];
      }
    }
    __syncthreads();
    const float tk = sc[0], iv0 = sc[1];
    // p = tau A_t v, v = (1, x_1 / v0, ...): four threads per row
    {
      const int i = tid >> 2, part = tid & 3;
      float acc = 0.f;
      if (i < m && tk != 0.f) {
        const float *row = A + (k + 1 + i) * LDA + k + 1;
        for (int j = part; j < m; j += 4) acc = fmaf(row[j], j == 0 ? 1.f : xk[j] * iv0, acc);
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (i < m && part == 0) pv[i] = tk * acc;
    }
    __syncthreads();
    // K = tau / 2 (p . v); w = p - K v
    if (warp == 0) {
      float s2 = 0.f;
      for (int j = lane; j < m; j += 32) {
        const float v = j == 0 ? 1.f : xk[j] * iv0;
        vv[j] = v;
        s2 = fmaf(pv[j], v, s2);
      }
      const float K = 0.5f * tk * warp_sum_f(s2);
      for (int j = lane; j < m; j += 32) wv[j] = pv[j] - K * vv[j];
    }
    __syncthreads();
    // A_t -= v w^T + w v^T; row k keeps the reflector
    if (tk != 0.f) {
      for (int i = warp; i < m; i += kEigThreads / 32) {
        const float vi = vv[i], wi = wv[i];
        float *row = A + (k + 1 + i) * LDA + k + 1;
        for (int j = lane; j < m; j += 32) row[j] -= fmaf(vi, wv[j], wi * vv[j]);
      }
    }
    for (int j = tid; j < m; j += kEigThreads) A[k * LDA + k + 1 + j] = tk != 0.f ? vv[j] : (j == 0 ? 1.f : 0.f);
    __syncthreads();
  }
  if (tid == 0) {
    dg[D - 2] = A[(D - 2) * LDA + D - 2];
    dg[D - 1] = A[(D - 1) * LDA + D - 1];
    ev[D - 2] = A[(D - 2) * LDA + D - 1];
    ev[D - 1] = 0.f;
    tau[D - 2] = 0.f;
  }
  __syncthreads();
  if (tid < D) e2[tid] = ev[tid] * ev[tid];
  // Gershgorin interval and the pivot floor of the Sturm counts
  if (warp == 0) {
    float lo = INFINITY, hi = -INFINITY, emax = 0.f;
    for (int i = lane; i < D; i += 32) {
      const float r = fabsf(ev[i]) + (i > 0 ? fabsf(ev[i - 1]) : 0.f);
      lo = fminf(lo, dg[i] - r);
      hi = fmaxf(hi, dg[i] + r);
      emax = fmaxf(emax, ev[i] * ev[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      emax = fmaxf(emax, __shfl_xor_sync(0xffffffffu, emax, o));
    }
    if (lane == 0) {
      const float span = fmaxf(hi - lo, 1e-30f);
      gs[0] = lo - 1e-6f * span;
      gs[1] = hi + 1e-6f * span;
      gs[2] = 1e-30f * fmaxf(1.f, emax);
    }
  }
  __syncthreads();

  // ---- 2. eigenvalues: thread group of 4 per eigenvalue (ascending index a) ----
  {
    const int a = tid >> 2, s = tid & 3;
    const float pivmin = gs[2];
    float lo = gs[0], hi = gs[1];
    for (int r = 0; r < kRounds; r++) {
      float x[4];
#pragma unroll
      for (int u = 0; u < 4; u++) x[u] = lo + (hi - lo) * (0.2f * (float)(u + 1));
      const float xs = x[s];
      float qv = dg[0] - xs;
      if (fabsf(qv) < pivmin) qv = -pivmin;
      int c = qv < 0.f;
      for (int i = 1; i < D; i++) {
        qv = (dg[i] - xs) - __fdividef(e2[i - 1], qv);
        if (fabsf(qv) < pivmin) qv = -pivmin;
        c += qv < 0.f;
      }
      int cs[4];
#pragma unroll
      for (int u = 0; u < 4; u++) cs[u] = __shfl_sync(0xffffffffu, c, (lane & ~3) | u);
      // eigenvalue a lies in the first sub-interval whose right end counts more than a below it
      float nlo = lo, nhi = hi;
      bool found = false;
#pragma unroll
      for (int u = 0; u < 4; u++) {
        if (!found) {
          if (cs[u] > a) { nhi = x[u]; found = true; }
          else nlo = x[u];
        }
      }
      lo = nlo;
      hi = nhi;
    }
    if (s == 0) lam[a] = 0.5f * (lo + hi);
  }
  __syncthreads();
  if (tid < D) eigvals[(int64_t)h * D + tid] = lam[D - 1 - tid];
  if (rank == 0) {
    if (tid == 0) n[h] = nn;
    return;
  }
  const float tnorm = fmaxf(fabsf(gs[0]), fabsf(gs[1]));

  // ---- 3. inverse iteration, one thread per vector (vector k: k-th largest eigenvalue) ----
  if (tid < rank) {
    const int k = tid;
    const float sh = lam[D - 1 - k], tiny = fmaxf(1.2e-7f * tnorm, 1e-30f);
    float *dgv = lu + k * LU, *s1 = dgv + D, *s2 = s1 + D, *z = s2 + D;
    for (int i = 0; i < D; i++) z[i] = start_entry(i, k);
    for (int it = 0; it < 2; it++) {
      // Gaussian elimination with partial pivoting of T - sh I; U has two superdiagonals
      float cd = dg[0] - sh, c1 = ev[0], c2 = 0.f, cr = z[0];
      for (int i = 0; i < D - 1; i++) {
        const float sub = ev[i], nd = dg[i + 1] - sh, n1 = (i + 1 < D - 1) ? ev[i + 1] : 0.f, nr = z[i + 1];
        if (fabsf(sub) > fabsf(cd)) {  // swap rows i and i + 1
          const float f = cd / sub;
          dgv[i] = sub; s1[i] = nd; s2[i] = n1; z[i] = nr;
          cd = c1 - f * nd; c1 = c2 - f * n1; c2 = 0.f; cr = cr - f * nr;
        } else {
          if (cd == 0.f) cd = tiny;
          const float f = sub / cd;
          dgv[i] = cd; s1[i] = c1; s2[i] = c2; z[i] = cr;
          cd = nd - f * c1; c1 = n1 - f * c2; c2 = 0.f; cr = nr - f * cr;
        }
      }
      dgv[D - 1] = cd == 0.f ? tiny : cd; s1[D - 1] = 0.f; s2[D - 1] = 0.f; z[D - 1] = cr;
      float big = 0.f;
      for (int i = D - 1; i >= 0; i--) {
        float t = z[i];
        if (i + 1 < D) t -= s1[i] * z[i + 1];
        if (i + 2 < D) t -= s2[i] * z[i + 2];
        const float dd = dgv[i] == 0.f ? tiny : dgv[i];
        if (!(fabsf(t) <= 1e20f * fabsf(dd))) {
          // growth through near-zero pivots (an eigenvalue of high multiplicity, e.g. fewer Queries
          // than channels): scale the whole system down, solved part and remaining right-hand side
          const float f = (1e20f * fabsf(dd)) / fabsf(t);
          for (int j = 0; j < D; j++) z[j] *= f;
          big *= f;
          t *= f;
        }
        z[i] = t / dd;
        big = fmaxf(big, fabsf(z[i]));
      }
      const float sc2 = big > 0.f && big < INFINITY ? 1.f / big : 0.f;
      if (sc2 == 0.f) bad = 1;
      for (int i = 0; i < D; i++) z[i] *= sc2;
    }
  }
  __syncthreads();
  // modified Gram-Schmidt within clusters, in order of k (warp 0); then unit length
  if (warp == 0) {
    for (int k = 0; k < rank; k++) {
      float *zk = lu + k * LU + 3 * D;
      for (int j = 0; j < k; j++) {
        if (fabsf(lam[D - 1 - j] - lam[D - 1 - k]) > 1e-3f * tnorm) continue;
        const float *zj = lu + j * LU + 3 * D;
        float dt = 0.f;
        for (int i = lane; i < D; i += 32) dt = fmaf(zj[i], zk[i], dt);
        dt = warp_sum_f(dt);
        for (int i = lane; i < D; i += 32) zk[i] -= dt * zj[i];
        __syncwarp();
      }
      float nr = 0.f;
      for (int i = lane; i < D; i += 32) nr = fmaf(zk[i], zk[i], nr);
      nr = warp_sum_f(nr);
      const float in = nr > 0.f ? rsqrtf(nr) : 0.f;
      if (nr == 0.f && lane == 0) bad = 1;
      for (int i = lane; i < D; i += 32) zk[i] *= in;
      __syncwarp();
    }
  }
  __syncthreads();

  // ---- 4. back-transformation u = H_0 ... H_{D-3} z, one warp per vector; sign; bf16 ----
  if (warp < rank) {
    const int k = warp;
    float *u = lu + k * LU + 3 * D;
    for (int kk = D - 3; kk >= 0; kk--) {
      const float t = tau[kk];
      if (t == 0.f) continue;
      const float *v = A + kk * LDA + kk + 1;  // reflector kk acts on rows kk+1 .. D-1
      const int m = D - 1 - kk;
      float dt = 0.f;
      for (int j = lane; j < m; j += 32) dt = fmaf(v[j], u[kk + 1 + j], dt);
      dt = t * warp_sum_f(dt);
      for (int j = lane; j < m; j += 32) u[kk + 1 + j] -= dt * v[j];
      __syncwarp();
    }
    float best = -1.f;
    int arg = D;
    for (int c = lane; c < D; c += 32) {
      const float a = fabsf(u[c]);
      if (a > best) { best = a; arg = c; }
    }
    for (int off = 16; off > 0; off >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int oa = __shfl_xor_sync(0xffffffffu, arg, off);
      if (ob > best || (ob == best && oa < arg)) { best = ob; arg = oa; }
    }
    const float sg = u[arg] < 0.f ? -1.f : 1.f;
    for (int c = lane; c < D; c += 32) u_r[((int64_t)h * D + c) * rank + k] = f32_to_bf16_rn(sg * u[c]);
  }
  if (tid == 0) {
    if (bad) qwm_dev_error(status, QWM_ERR_NOT_CONVERGED);
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

cudaError_t launch_eig(const float *S, int64_t *n, int64_t nq, int H, int rank, float *eigvals, uint16_t *u_r,
                       int32_t *status, cudaStream_t st) {
  // n is read here and advanced by n += nq at the end of each head's solve
  const size_t smem = ((size_t)D * LDA + (size_t)QWM_MAX_RANK * LU) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(eig_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  eig_kernel<<<H, kEigThreads, smem, st>>>(S, n, nq, rank, eigvals, u_r, status);
  return cudaGetLastError();
}
