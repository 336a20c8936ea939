// AdamW path: the global gradient norm of the AdamW gradients (clip at
// max_norm, OMN page AdamW paragraph) and the bias-corrected AdamW update
// with decoupled decay (Qwen3.8 optimizer notes, Adam/AdamW history).
//
// Both kernels stream HBM: 128-bit loads where the pointers allow, several
// independent vectors in flight per thread, grid sized in multiples of the
// SM count.  Tensor tables travel in the kernel parameters (up to
// kMaxTensors per launch), so no device table is needed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "device_common.cuh"
#include "internal.h"

namespace gbo {

namespace {

constexpr int kMaxTensors = 64;
constexpr int kChunk = 16384;  // elements per work item
constexpr int kThreads = 256;

struct ClipTable {
  const void *ptr[kMaxTensors];
  int64_t numel[kMaxTensors];
  int64_t chunk0[kMaxTensors + 1];
  int32_t dtype[kMaxTensors];
  int32_t vec[kMaxTensors];
  int32_t n;
};

struct AdamTable {
  float *p[kMaxTensors];
  const void *g[kMaxTensors];
  float *m[kMaxTensors];
  float *v[kMaxTensors];
  int64_t numel[kMaxTensors];
  int64_t chunk0[kMaxTensors + 1];
  int32_t gdtype[kMaxTensors];
  int32_t vec[kMaxTensors];
  int32_t n;
};

struct AdamScalars {
  float lr, beta1, beta2, eps, wd;
  float step_size;     // lr / (1 - beta1^t)
  float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^t)
};

// Compensated (Kahan) accumulation keeps the fp32 sum of ~1e3 terms per
// thread at about one rounding of error.
struct Kahan {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
};

__device__ __forceinline__ float4 load_g4(const void *g, int32_t dtype, int64_t idx) {
  if (dtype == GBO_BF16) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(g) + idx));
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
    return make_float4(__low2float(lo), __high2float(lo), __low2float(hi), __high2float(hi));
  }
  return __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(g) + idx));
}

__global__ void __launch_bounds__(kThreads)
clip_partial_kernel(const __grid_constant__ ClipTable T, float *__restrict__ partials) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up
  pdl_wait();    // the previous kernel has completed and its writes are visible
  __shared__ float red[32];
  Kahan acc;
  const int64_t n_chunks = T.chunk0[T.n];
  for (int64_t ch = blockIdx.x; ch < n_chunks; ch += gridDim.x) {
    const int ti = find_owner(ch, T.n, [&](int k) { return T.chunk0[k]; });
    const int64_t start = (ch - T.chunk0[ti]) * kChunk;
    const int64_t end = min(start + (int64_t)kChunk, T.numel[ti]);
    const void *g = T.ptr[ti];
    const int32_t dt = T.dtype[ti];
    if (T.vec[ti]) {
      const int64_t vend = start + ((end - start) & ~(int64_t)3);
      for (int64_t i = start + 4 * threadIdx.x; i < vend; i += 4 * kThreads) {
        const float4 x = load_g4(g, dt, i);
        acc.add(fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, x.w * x.w))));
      }
      for (int64_t i = vend + threadIdx.x; i < end; i += kThreads) {
        const float x = ld_elem(g, dt, i);
        acc.add(x * x);
      }
    } else {
      for (int64_t i = start + threadIdx.x; i < end; i += kThreads) {
        const float x = ld_elem(g, dt, i);
        acc.add(x * x);
      }
    }
  }
  const float s = block_sum(acc.s - acc.c, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = s;
}

__global__ void __launch_bounds__(kThreads)
clip_finalize_kernel(const float *__restrict__ partials, int n_partials, float max_norm,
                     float *total_out, float *coef_out, int32_t *status) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up
  pdl_wait();    // the previous kernel has completed and its writes are visible
  __shared__ float red[32];
  Kahan acc;
  for (int i = threadIdx.x; i < n_partials; i += kThreads) acc.add(partials[i]);
  const float sum = block_sum(acc.s - acc.c, red);
  if (threadIdx.x == 0) {
    const float N = sqrtf(sum);
    float coef = 1.0f;
    if (!isfinite(N)) {
      coef = __int_as_float(0x7fc00000);
      flag_status(status, GBO_STATUS_NONFINITE);
    } else if (N > max_norm) {
      coef = max_norm / N;
    }
    if (total_out) *total_out = N;
    if (coef_out) *coef_out = coef;
  }
}

__device__ __forceinline__ void adam_elem(float &p, float g, float &m, float &v, float coef,
                                          const AdamScalars &s) {
  const float gg = coef * g;
  m = fmaf(s.beta1, m, (1.0f - s.beta1) * gg);
  v = fmaf(s.beta2, v, (1.0f - s.beta2) * gg * gg);
  const float denom = sqrtf(v) * s.inv_sqrt_bc2 + s.eps;
  // the decay and the Adam step summed first (at their own, small,
  // magnitude), so p itself is rounded once
  p = p + fmaf(-s.lr * s.wd, p, -s.step_size * (m / denom));
}

#ifndef GBO_ADAM_MIN_BLOCKS
#define GBO_ADAM_MIN_BLOCKS 1  // compiler choice (80 regs, 3 blocks/SM): forcing 4 measured 1.39 ms against 1.26
#endif
__global__ void __launch_bounds__(kThreads, GBO_ADAM_MIN_BLOCKS)
adamw_kernel(const __grid_constant__ AdamTable T, const __grid_constant__ AdamScalars s0,
             const float *__restrict__ coef_ptr, const int32_t *__restrict__ dev_step) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up
  pdl_wait();    // the previous kernel has completed and its writes are visible
  const float coef = coef_ptr ? __ldg(coef_ptr) : 1.0f;
  // the bias corrections, from a device step count when one is given
  // (computed as on the host, in double, once per block)
  __shared__ float bc[2];
  AdamScalars s = s0;
  if (dev_step) {
    if (threadIdx.x == 0) {
      const double t = (double)*dev_step;
      bc[0] = (float)((double)s.lr / (1.0 - pow((double)s.beta1, t)));
      bc[1] = (float)(1.0 / sqrt(1.0 - pow((double)s.beta2, t)));
    }
    __syncthreads();
    s.step_size = bc[0];
    s.inv_sqrt_bc2 = bc[1];
  }
  const int64_t n_chunks = T.chunk0[T.n];
  for (int64_t ch = blockIdx.x; ch < n_chunks; ch += gridDim.x) {
    const int ti = find_owner(ch, T.n, [&](int k) { return T.chunk0[k]; });
    const int64_t start = (ch - T.chunk0[ti]) * kChunk;
    const int64_t end = min(start + (int64_t)kChunk, T.numel[ti]);
    float *P = T.p[ti];
    float *M = T.m[ti];
    float *V = T.v[ti];
    const void *G = T.g[ti];
    const int32_t dt = T.gdtype[ti];
    int64_t vend = start;
    if (T.vec[ti]) {
      vend = start + ((end - start) & ~(int64_t)7);
      // two independent float4 groups per thread per trip
      for (int64_t i = start + 8 * threadIdx.x; i < vend; i += 8 * kThreads) {
        float4 p0 = *reinterpret_cast<float4 *>(P + i);
        float4 p1 = *reinterpret_cast<float4 *>(P + i + 4);
        float4 m0 = *reinterpret_cast<float4 *>(M + i);
        float4 m1 = *reinterpret_cast<float4 *>(M + i + 4);
        float4 v0 = *reinterpret_cast<float4 *>(V + i);
        float4 v1 = *reinterpret_cast<float4 *>(V + i + 4);
        const float4 g0 = load_g4(G, dt, i);
        const float4 g1 = load_g4(G, dt, i + 4);
        adam_elem(p0.x, g0.x, m0.x, v0.x, coef, s);
        adam_elem(p0.y, g0.y, m0.y, v0.y, coef, s);
        adam_elem(p0.z, g0.z, m0.z, v0.z, coef, s);
        adam_elem(p0.w, g0.w, m0.w, v0.w, coef, s);
        adam_elem(p1.x, g1.x, m1.x, v1.x, coef, s);
        adam_elem(p1.y, g1.y, m1.y, v1.y, coef, s);
        adam_elem(p1.z, g1.z, m1.z, v1.z, coef, s);
        adam_elem(p1.w, g1.w, m1.w, v1.w, coef, s);
        *reinterpret_cast<float4 *>(P + i) = p0;
        *reinterpret_cast<float4 *>(P + i + 4) = p1;
        *reinterpret_cast<float4 *>(M + i) = m0;
        *reinterpret_cast<float4 *>(M + i + 4) = m1;
        *reinterpret_cast<float4 *>(V + i) = v0;
        *reinterpret_cast<float4 *>(V + i + 4) = v1;
      }
    }
    for (int64_t i = vend + threadIdx.x; i < end; i += kThreads) {
      float p = P[i], m = M[i], v = V[i];
      adam_elem(p, ld_elem(G, dt, i), m, v, coef, s);
      P[i] = p;
      M[i] = m;
      V[i] = v;
    }
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int launch_clip_norm(const gbo_tensor *grads, int32_t n, float max_norm, float *total, float *coef,
                     int32_t *status, float *partials, int sm_count, void *stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int n_launch = (n + kMaxTensors - 1) / kMaxTensors;
  // Each launch owns an equal slice of the partial-sum array; unused
  // entries are written as zero so the finalize can sum all of them.
  const int per_launch = n_launch > 0 ? kClipBlocks / n_launch : kClipBlocks;
  int used = 0;
  for (int l = 0; l < n_launch; ++l) {
    ClipTable T{};
    T.n = min(kMaxTensors, n - l * kMaxTensors);
    T.chunk0[0] = 0;
    for (int k = 0; k < T.n; ++k) {
      const gbo_tensor &t = grads[l * kMaxTensors + k];
      T.ptr[k] = t.ptr;
      T.numel[k] = t.numel;
      T.dtype[k] = t.dtype;
      T.vec[k] = t.dtype == GBO_BF16 ? ((reinterpret_cast<uintptr_t>(t.ptr) & 7) == 0) : aligned16(t.ptr);
      T.chunk0[k + 1] = T.chunk0[k] + (t.numel + kChunk - 1) / kChunk;
    }
    const int grid = per_launch;
    const cudaError_t err = launch_kernel(clip_partial_kernel, dim3(grid), dim3(kThreads), 0, st, 1, T, partials + used);
    count_launches(1);
    used += grid;
    if (err != cudaSuccess) return (int)err;
  }
  (void)sm_count;
  const cudaError_t err =
      launch_kernel(clip_finalize_kernel, dim3(1), dim3(kThreads), 0, st, 1, (const float *)partials, used, max_norm,
                    total, coef, status);
  count_launches(1);
  return (int)err;
}

int launch_adamw(const gbo_adamw_desc *descs, int32_t n, const gbo_adamw_opts *opts,
                 const float *coef, int32_t *status, int sm_count, void *stream) {
  (void)status;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  AdamScalars s;
  s.lr = opts->lr;
  s.beta1 = opts->beta1;
  s.beta2 = opts->beta2;
  s.eps = opts->eps;
  s.wd = opts->weight_decay;
  if (!opts->dev_step) {
    const double bc1 = 1.0 - std::pow((double)opts->beta1, (double)opts->step);
    const double bc2 = 1.0 - std::pow((double)opts->beta2, (double)opts->step);
    s.step_size = (float)((double)opts->lr / bc1);
    s.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
  }
  for (int l = 0; l * kMaxTensors < n; ++l) {
    AdamTable T{};
    T.n = min(kMaxTensors, n - l * kMaxTensors);
    T.chunk0[0] = 0;
    for (int k = 0; k < T.n; ++k) {
      const gbo_adamw_desc &d = descs[l * kMaxTensors + k];
      T.p[k] = d.p;
      T.g[k] = d.g;
      T.m[k] = d.m;
      T.v[k] = d.v;
      T.numel[k] = d.numel;
      T.gdtype[k] = d.g_dtype;
      const bool gal = d.g_dtype == GBO_BF16 ? ((reinterpret_cast<uintptr_t>(d.g) & 7) == 0) : aligned16(d.g);
      T.vec[k] = aligned16(d.p) && aligned16(d.m) && aligned16(d.v) && gal;
      T.chunk0[k + 1] = T.chunk0[k] + (d.numel + kChunk - 1) / kChunk;
    }
    const int64_t chunks = T.chunk0[T.n];
    if (chunks == 0) continue;
    const unsigned grid = (unsigned)std::min<int64_t>(chunks, (int64_t)sm_count * 8);
    const cudaError_t err = launch_kernel(adamw_kernel, dim3(grid), dim3(kThreads), 0, st, 1, T, s, coef, opts->dev_step);
    count_launches(1);
    if (err != cudaSuccess) return (int)err;
  }
  return 0;
}

}  // namespace gbo
