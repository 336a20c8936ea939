// gbo_h2d_copy: a host-to-device copy made by SM loads of page-locked host
// memory rather than by a copy engine.
//
// A GB300's GPU reaches its Grace CPU's memory over NVLink-C2C.  Measured on
// a GB300 host (one 3.5 GB gradient upload per step, from page-locked memory
// on 2 MB pages): copy-engine uploads and SM loads both move ~211 GB/s, but
// on some hosts 3 to 4 copy-engine uploads in 40 stalled for 40-140 ms (more
// under a concurrent GEMM load), while the same 40 uploads made by a kernel
// never took more than 17.2 ms (16.6 ms median).  The stalls are in the
// copy engine's path, not in the link.
//
// A copy kernel competes with the step's kernels for SMs.  Spread thinly
// over every SM it slowed the Newton-Schulz GEMMs by a third, because their
// persistent, statically scheduled launches wait for their slowest CTA
// pair.  So the copy runs on SMs of its own: each block is 1024 threads
// with eight 16-byte loads in flight per thread, and it reserves kCopySmem
// of shared memory that it does not use, so that no SM holds two copy
// blocks, or a copy block beside a Newton-Schulz CTA (226 KB each).  A plan
// that leaves as many SMs free (gbo_muon_plan_set_free_sms) runs its GEMMs
// beside the copy.  Measured: a block moves ~50 GB/s from the host alone
// (four: 203 GB/s), ~27 GB/s beside a step's GEMMs, so overlapping a 3.5 GB
// upload with a 20 ms step takes more SMs than the GEMMs can spare, and the
// copy engine stays the better route there.  Stores are marked evict-first:
// nothing reads the copy before the next step.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "gbo.h"
#include "internal.h"

namespace gbo {
namespace {

constexpr int kCopyThreads = 1024;
constexpr int kCopyUnroll = 8;
constexpr int kCopySmem = 120 * 1024;  // reserved, unused: more than half an SM's 228 KB

__global__ void __launch_bounds__(kCopyThreads, 1)
    h2d_copy_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src, int64_t n16,
                    unsigned char *__restrict__ dst_tail, const unsigned char *__restrict__ src_tail, int tail) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (kCopyUnroll - 1) * stride < n16; i += kCopyUnroll * stride) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) v[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) __stcs(dst + i + u * stride, v[u]);
  }
  for (; i < n16; i += stride) __stcs(dst + i, src[i]);
  if (blockIdx.x == 0 && (int)threadIdx.x < tail) dst_tail[threadIdx.x] = src_tail[threadIdx.x];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The device address of host byte p, if p lies in page-locked host memory
// mapped for this device; nullptr otherwise.
const void *mapped_host(const void *p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

bool device_memory(const void *p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

}  // namespace
}  // namespace gbo

using namespace gbo;

extern "C" int gbo_h2d_copy(void *dst, const void *src, int64_t nbytes, int32_t blocks, gbo_stream_t stream) {
  if (nbytes < 0) return report_error(GBO_ERR_INVALID_ARG, "nbytes must be >= 0");
  if (blocks < 0) return report_error(GBO_ERR_INVALID_ARG, "blocks must be >= 0");
  if (nbytes == 0) return report_ok();
  if (!dst || !src) return report_error(GBO_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(dst) || !aligned16(src))
    return report_error(GBO_ERR_INVALID_ARG, "dst and src must be 16-byte aligned");
  int dev = -1, sm = 0;
  int rc = require_device(&dev, &sm);
  if (rc != GBO_OK) return rc;
  const char *last = static_cast<const char *>(src) + (nbytes - 1);
  const void *dsrc = mapped_host(src);
  const void *dlast = mapped_host(last);
  if (!dsrc || !dlast || static_cast<const char *>(dlast) - static_cast<const char *>(dsrc) != nbytes - 1)
    return report_error(GBO_ERR_INVALID_ARG,
                        "src .. src + nbytes must lie in page-locked host memory mapped for the device "
                        "(cudaHostRegister or cudaMallocHost)");
  if (!device_memory(dst) || !device_memory(static_cast<char *>(dst) + (nbytes - 1)))
    return report_error(GBO_ERR_INVALID_ARG, "dst .. dst + nbytes must lie in device memory");
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(h2d_copy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCopySmem);
  });
  if (attr_err != cudaSuccess) return report_error(GBO_ERR_CUDA, "cudaFuncSetAttribute(h2d copy kernel)");
  const int64_t n16 = nbytes / 16;
  const int tail = (int)(nbytes % 16);
  const int64_t per_block = (int64_t)kCopyThreads * kCopyUnroll;
  const int64_t want = blocks > 0 ? std::min<int64_t>(blocks, sm) : sm;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (n16 + per_block - 1) / per_block));
  h2d_copy_kernel<<<grid, kCopyThreads, kCopySmem, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4 *>(dst), static_cast<const uint4 *>(dsrc), n16, static_cast<unsigned char *>(dst) + n16 * 16,
      static_cast<const unsigned char *>(dsrc) + n16 * 16, tail);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    char msg[200];
    snprintf(msg, sizeof msg, "h2d copy kernel: %s", cudaGetErrorString(e));
    return report_error(GBO_ERR_CUDA, msg);
  }
  count_launches(1);
  return report_ok();
}
