// qwm_update_query_stats_noalloc: the Query statistics / weights / basis update of
// qwm_update_query_stats for callers that cannot allocate device memory.
//
// The scratch the kernels need (per-split partial sums of q q^T) lives in one file-scope device
// array of fixed size instead of a context's workspace.
// Every GPU that loads this library holds that array until the process exits.  Host code only
// ever passes the array's device address, obtained with cudaGetSymbolAddress once per CUDA
// context (a device's primary context, or a context the caller made current itself): the address
// belongs to the context the module was loaded into, so a new context (after cudaDeviceReset, or
// a caller's own context) gets its own lookup.  Contexts are told apart by the driver's unique
// context ID, which is never reused within a process.
#include <cuda.h>

#include <mutex>

#include "qwm_internal.cuh"

namespace {

constexpr int kMaxHeads = 64;   // largest head count this entry point accepts
constexpr int kSlots = 2 * kMaxHeads;  // partial-sum slots (splits x heads <= kSlots)
constexpr int kMaxSplits = 8;   // as many splits per head as the context version uses at most
constexpr size_t kPartFloats = (size_t)kSlots * QWM_D * QWM_D;  // 8 MiB
constexpr size_t kScratchBytes = kPartFloats * sizeof(float);

static __device__ __align__(256) unsigned char g_stats_scratch[kScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

struct CacheEntry {
  unsigned long long ctx_id;  // 0 = free
  void *addr;
};
constexpr int kCacheEntries = 64;
std::mutex g_setup_mutex;
CacheEntry g_cache[kCacheEntries];
int g_cache_next = 0;  // round-robin replacement once every entry is used
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

bool driver_fns() {
  if (g_ctx_current && g_ctx_id) return true;
  void *a = nullptr, *b = nullptr;
  cudaDriverEntryPointQueryResult qa, qb;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) != cudaSuccess ||
      qa != cudaDriverEntryPointSuccess)
    return false;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
      qb != cudaDriverEntryPointSuccess)
    return false;
  g_ctx_current = (CtxGetCurrentFn)a;
  g_ctx_id = (CtxGetIdFn)b;
  return true;
}

// Device address of the scratch array in the current context (the first call in a context looks
// it up; under lazy module loading that first lookup is also what loads the module and so reserves
// the array on the device).
qwm_status scratch_in_current_context(unsigned char **out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!driver_fns()) return QWM_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return QWM_ERR_CUDA;
  void *fresh = nullptr;
  if (!ctx) {  // no context current yet: the lookup itself initialises the device's primary context
    if (cudaGetSymbolAddress(&fresh, g_stats_scratch) != cudaSuccess || fresh == nullptr) return QWM_ERR_CUDA;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return QWM_ERR_CUDA;
  }
  unsigned long long id = 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS || id == 0) return QWM_ERR_CUDA;
  for (const CacheEntry &e : g_cache)
    if (e.ctx_id == id) {
      *out = (unsigned char *)e.addr;
      return QWM_OK;
    }
  if (!fresh && (cudaGetSymbolAddress(&fresh, g_stats_scratch) != cudaSuccess || fresh == nullptr))
    return QWM_ERR_CUDA;
  g_cache[g_cache_next] = CacheEntry{id, fresh};
  g_cache_next = (g_cache_next + 1) % kCacheEntries;
  *out = (unsigned char *)fresh;
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
      (u_r && !aligned16(u_r)) || (dev_status && ((uintptr_t)dev_status & 3u)))
    return QWM_ERR_ALIGN;
  unsigned char *base = nullptr;
  qwm_status s = scratch_in_current_context(&base);
  if (s != QWM_OK) return s;
  const int H = cfg->heads;
  int dev = 0, sms = 1;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return QWM_ERR_CUDA;
  // splits: enough CTAs to cover the SMs, as the context version does, within the array's slots
  int splits = (sms + H - 1) / H;
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (splits > kSlots / H) splits = kSlots / H;
  if (splits < 1) splits = 1;
  float *part = (float *)base;  // the slots this call uses are written in full before they are read
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  if (nq > 0) e = launch_stats_partial(q, nq, H, part, splits, dev_status, st);
  if (e == cudaSuccess) e = launch_stats_finish(part, nq > 0 ? splits : 0, nq, H, S, n, w, st);
  if (e == cudaSuccess) e = launch_eig(S, n, nq, H, cfg->rank, eigvals, u_r, dev_status, st);
  return e == cudaSuccess ? QWM_OK : QWM_ERR_CUDA;
}
