// qwm_update_query_stats_noalloc: the Query statistics / weights / basis update of
// qwm_update_query_stats for callers that cannot allocate device memory.
//
// The scratch the kernels need (per-split partial sums of q q^T) lives in one file-scope device
// array of fixed size instead of a context's workspace.
// Every GPU that loads this library holds that array until the process exits.  Host code only
// ever passes the array's device address, obtained once per device with cudaGetSymbolAddress.
#include <mutex>

#include "qwm_internal.cuh"

namespace {

constexpr int kMaxHeads = 64;  // largest head count this entry point accepts
constexpr int kSplits = 2;     // partial sums per head
constexpr size_t kPartFloats = (size_t)kSplits * kMaxHeads * QWM_D * QWM_D;  // 8 MiB
constexpr size_t kScratchBytes = kPartFloats * sizeof(float);

static __device__ __align__(256) unsigned char g_stats_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices];  // device address of g_stats_scratch, per device, set on first use

// Device address of the scratch array on the current device (first call on a device looks it up).
qwm_status scratch_on_current_device(unsigned char **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QWM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_stats_scratch) != cudaSuccess || p == nullptr) return QWM_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = (unsigned char *)g_scratch_addr[dev];
  return QWM_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" qwm_status qwm_update_query_stats_noalloc(const qwm_config *cfg, const uint16_t *q, int64_t nq, float *S,
                                                     int64_t *n, float *w, float *eigvals, uint16_t *u_r,
                                                     int32_t *dev_status, qwm_stream stream) {
  if (!cfg || !S || !n || !w || !eigvals || nq < 0) return QWM_ERR_ARG;
  if (nq > 0 && !q) return QWM_ERR_ARG;
  if (cfg->heads < 1 || cfg->rank < 0) return QWM_ERR_ARG;
  if (cfg->head_dim != QWM_D || cfg->rank > QWM_MAX_RANK) return QWM_ERR_SHAPE;
  if (cfg->heads > kMaxHeads) return QWM_ERR_SHAPE;  // beyond the fixed scratch array
  if (cfg->rank > 0 && !u_r) return QWM_ERR_ARG;
  if ((q && !aligned16(q)) || !aligned16(S) || !aligned16(n) || !aligned16(w) || !aligned16(eigvals) ||
      (u_r && !aligned16(u_r)))
    return QWM_ERR_ALIGN;
  unsigned char *base = nullptr;
  qwm_status s = scratch_on_current_device(&base);
  if (s != QWM_OK) return s;
  float *part = (float *)base;  // overwritten in full by every call
  cudaStream_t st = (cudaStream_t)stream;
  const int H = cfg->heads;
  cudaError_t e = cudaSuccess;
  if (nq > 0) e = launch_stats_partial(q, nq, H, part, kSplits, dev_status, st);
  if (e == cudaSuccess) e = launch_stats_finish(part, nq > 0 ? kSplits : 0, nq, H, S, n, w, st);
  if (e == cudaSuccess) e = launch_eig(S, n, nq, H, cfg->rank, eigvals, u_r, dev_status, st);
  return e == cudaSuccess ? QWM_OK : QWM_ERR_CUDA;
}
