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
#include <cuda_runtime.h>

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
float *g_scratch_addr[kMaxDevices] = {};

// Device address of g_clip_scratch on the current device, looked up once
// per device (with that device current) and cached.
int scratch_on_device(int dev, float **out) {
  if (dev < 0 || dev >= kMaxDevices) return report_error(GBO_ERR_UNSUPPORTED, "device index above 63");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_clip_scratch);
    if (e != cudaSuccess) {
      char msg[256];
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress(clip scratch): %s", cudaGetErrorString(e));
      return report_error(GBO_ERR_CUDA, msg);
    }
    g_scratch_addr[dev] = static_cast<float *>(p);
  }
  *out = g_scratch_addr[dev];
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
  if (!(max_norm > 0.f) || !(max_norm < 3.4e38f)) return report_error(GBO_ERR_INVALID_ARG, "max_norm must be > 0");
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
