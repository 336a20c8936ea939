// gbo_clip_norm_noalloc: the global gradient norm and clip coefficient of
// gbo_clip_norm, for callers that cannot hand the library a scratch buffer.
//
// Some callers own none of the device memory they run in: every byte of
// HBM already belongs to another allocator (a framework's caching pool that
// reserved the device up front), or they run on a path where a cudaMalloc
// -- which can synchronise the whole device -- is not allowed.  Such a
// caller cannot provide the clip norm's scratch.  This entry point keeps
// that scratch (one fp32 partial sum per reduction block) in a fixed array
// of the library's own device memory instead, so it allocates nothing.
//
// The array is compiled into the library: every GPU that loads it holds the
// array until the process exits.  All calls share it, so two calls whose
// work overlaps on the GPU (different streams, or different host threads)
// race on it; calls in one stream are ordered and safe.  The array keeps
// the last call's partial sums; nothing needs clearing, because every slot
// a call reads is written earlier in that same call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <mutex>

#include "gbo.h"
#include "internal.h"

namespace gbo {

// One partial sum per clip reduction block (kClipBlocks fp32 = 4 KB).
static __device__ __align__(256) float g_clip_scratch[kClipBlocks];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
// Per device: the CUDA context the address was looked up in (its
// process-unique ID, never reused) and the address.  A device reset, or
// anything else that replaces the context, makes the next call look the
// address up again instead of using one from a context that is gone.
struct ScratchAddr {
  unsigned long long ctx_id = 0;
  bool known = false;
  float *addr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name) {
  void *p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

// ID of the context current on this thread (the runtime has made the
// device's primary context current by the time this runs).
int current_context_id(unsigned long long *id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, id) != CUDA_SUCCESS)
    return report_error(GBO_ERR_CUDA, "cannot identify the current CUDA context");
  return GBO_OK;
}

// Device address of g_clip_scratch on the current device.  The set-up --
// cudaGetSymbolAddress with that device current -- runs on the first call
// in each context of a device and is cached for the later ones.
int scratch_on_device(int dev, float **out) {
  if (dev < 0 || dev >= kMaxDevices) return report_error(GBO_ERR_UNSUPPORTED, "device index above 63");
  unsigned long long ctx_id = 0;
  int rc = current_context_id(&ctx_id);
  if (rc != GBO_OK) return rc;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchAddr &c = g_scratch[dev];
  if (!c.known || c.ctx_id != ctx_id) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_clip_scratch);
    if (e != cudaSuccess) {
      char msg[256];
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress(clip scratch): %s", cudaGetErrorString(e));
      return report_error(GBO_ERR_CUDA, msg);
    }
    c.addr = static_cast<float *>(p);
    c.ctx_id = ctx_id;
    c.known = true;
  }
  *out = c.addr;
  return GBO_OK;
}

bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace gbo

using namespace gbo;

extern "C" int gbo_clip_norm_noalloc(const gbo_tensor *grads, int32_t n, float max_norm, float *dev_total_norm,
                                     float *dev_coef, int32_t *dev_status, gbo_stream_t stream) {
  if (n < 0 || (n > 0 && !grads)) return report_error(GBO_ERR_INVALID_ARG, "bad gradient table");
  if (n > GBO_CLIP_NOALLOC_MAX_TENSORS) {
    char msg[200];
    snprintf(msg, sizeof msg,
             "%d tensors: the fixed scratch of %d partial sums serves at most %d tensors per call", n,
             kClipBlocks, GBO_CLIP_NOALLOC_MAX_TENSORS);
    return report_error(GBO_ERR_INVALID_ARG, msg);
  }
  // the same rule as gbo_clip_norm: any finite positive max_norm
  if (!(max_norm > 0.f) || !std::isfinite(max_norm)) return report_error(GBO_ERR_INVALID_ARG, "max_norm must be > 0");
  for (int32_t i = 0; i < n; ++i) {
    const gbo_tensor &t = grads[i];
    if (t.dtype != GBO_F32 && t.dtype != GBO_BF16) return report_error(GBO_ERR_DTYPE, "bad gradient dtype");
    if (t.numel < 0) return report_error(GBO_ERR_INVALID_ARG, "negative numel");
    if (t.numel > 0 && (!t.ptr || !aligned_to(t.ptr, t.dtype == GBO_BF16 ? 2 : 4)))
      return report_error(GBO_ERR_INVALID_ARG, "NULL or misaligned gradient pointer");
  }
  int dev = -1, sm = 0;
  int rc = require_device(&dev, &sm);
  if (rc != GBO_OK) return rc;
  float *scratch = nullptr;
  rc = scratch_on_device(dev, &scratch);
  if (rc != GBO_OK) return rc;
  const int err = launch_clip_norm(grads, n, max_norm, dev_total_norm, dev_coef, dev_status, scratch, sm, stream);
  if (err) {
    char msg[200];
    snprintf(msg, sizeof msg, "clip-norm kernels: %s", cudaGetErrorString((cudaError_t)err));
    return report_error(GBO_ERR_CUDA, msg);
  }
  return report_ok();
}
