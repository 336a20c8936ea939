// Device helpers shared by the library's kernels: element conversion,
// block reductions, and the Newton-Schulz epilogue arithmetic.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "internal.h"

namespace gbo {

// Programmatic dependent launch.  Every kernel of the library calls
// pdl_launch() as it starts, letting the next kernel on the stream be
// scheduled as SMs free up, and pdl_wait() after its prologue (barrier
// set-up, TMEM allocation) and before its first access to global memory,
// which returns once the previous kernel has completed and its writes are
// visible.  These take effect only when the launch carries
// cudaLaunchAttributeProgrammaticStreamSerialization, which launch_kernel
// below sets when pdl_enabled(stream): by default only while the stream is
// being captured into a CUDA graph.  Measured on a GB300, in graph replays it
// made the one-layer step ~1.7% faster (and the others slightly), while with
// kernels launched directly on a stream it made the many-small-matrix step
// 12.7% slower.  Without the attribute both calls return at once.
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kernel` (with programmatic stream serialization when enabled, and,
// with cluster > 1, clusters of that many CTAs along x).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 int cluster, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = pdl_enabled(stream);
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ float ld_elem(const void *base, int32_t dtype, int64_t idx) {
  if (dtype == GBO_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
  return reinterpret_cast<const float *>(base)[idx];
}

__device__ __forceinline__ void st_elem(void *base, int32_t dtype, int64_t idx, float v) {
  if (dtype == GBO_BF16)
    reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float *>(base)[idx] = v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum / max for blockDim.x a multiple of 32 (<= 1024).  `red`
// is shared scratch of >= 32 floats.  Every thread gets the result.  The
// combination order is fixed, so results are reproducible.
__device__ __forceinline__ float block_sum(float v, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  t = warp_sum(t);
  return t;
}

__device__ __forceinline__ float block_max(float v, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  t = warp_max(t);
  return t;
}

__device__ __forceinline__ void flag_status(int32_t *status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

// Index of the matrix owning global item `t`, given each matrix's first
// item in `first` (non-decreasing).  Binary search; `n` >= 1.
template <typename GetFirst>
__device__ __forceinline__ int find_owner(int64_t t, int n, GetFirst first) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (first(mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Eight consecutive elements of a row as fp32: one 16-byte load (bf16) or
// two (fp32) when `vec`, else element by element under `valid`.
__device__ __forceinline__ void load8(const void *base, int32_t dtype, int64_t idx, int valid, bool vec,
                                      float *out) {
  if (vec && valid == 8) {
    if (dtype == GBO_BF16) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(base) + idx);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[h]);
        out[2 * h] = __low2float(b);
        out[2 * h + 1] = __high2float(b);
      }
    } else {
      const float4 *f = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(base) + idx);
      const float4 a = f[0], b = f[1];
      out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
      out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) out[e] = e < valid ? ld_elem(base, dtype, idx + e) : 0.f;
  }
}

// Eight consecutive elements: 16-byte store(s) when `vec` (the caller
// guarantees alignment) and the segment is whole, else element by element.
template <typename XT>
__device__ __forceinline__ void store8(XT *dst, const float *v, int valid, bool vec) {
  if (vec && valid == 8) {
    if constexpr (sizeof(XT) == 2) {
      uint4 u;
      __nv_bfloat162 h[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) h[q] = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
      u.x = *reinterpret_cast<uint32_t *>(&h[0]);
      u.y = *reinterpret_cast<uint32_t *>(&h[1]);
      u.z = *reinterpret_cast<uint32_t *>(&h[2]);
      u.w = *reinterpret_cast<uint32_t *>(&h[3]);
      *reinterpret_cast<uint4 *>(dst) = u;
    } else {
      float4 *f = reinterpret_cast<float4 *>(dst);
      f[0] = make_float4(v[0], v[1], v[2], v[3]);
      f[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (e < valid) {
        if constexpr (sizeof(XT) == 2) dst[e] = __float2bfloat16_rn(v[e]);
        else dst[e] = v[e];
      }
  }
}

}  // namespace gbo
