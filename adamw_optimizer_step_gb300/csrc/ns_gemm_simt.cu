// Newton-Schulz GEMMs on CUDA cores (FFMA), used for fp32 arithmetic.
//
// One persistent launch covers every matrix of up to kMaxClassesPerLaunch
// shape classes.  Each 64 x 64 output tile is one loop trip; the epilogue
// (ns_epilogue) does the polynomial combination, the product scaling or the
// weight write.  Iteration of eq. (5) of the NorMuon paper (zskr.cn, section
// 2.2): Gram A = X X^T, optional square A A, product (a I + b A + c A^2) X.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "device_common.cuh"
#include "internal.h"

namespace gbo {

namespace {

constexpr int kBM = 64, kBN = 64, kBK = 16, kThreads = 256;

struct SimtLaunch {
  ShapeClass cls[kMaxClassesPerLaunch];
  int64_t tile_start[kMaxClassesPerLaunch + 1];
  int32_t tiles_m[kMaxClassesPerLaunch];
  int32_t tiles_n[kMaxClassesPerLaunch];
  int32_t n;
};

template <typename T>
__device__ __forceinline__ float to_f(T v) {
  if constexpr (sizeof(T) == 2) return __bfloat162float(v);
  else return v;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
ns_gemm_simt_kernel(const __grid_constant__ SimtLaunch L, const __grid_constant__ PhaseArgs A) {
  __shared__ float As[kBK][kBM + 4];
  __shared__ float Bs[kBK][kBN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int64_t total = L.tile_start[L.n];
  const bool gram = (A.mode == kGram || A.mode == kGramA);
  const bool square = (A.mode == kSquare);
  for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
    int c = 0;
    while (c + 1 < L.n && L.tile_start[c + 1] <= t) ++c;
    const ShapeClass &C = L.cls[c];
    const int64_t local = t - L.tile_start[c];
    const int64_t per = (int64_t)L.tiles_m[c] * L.tiles_n[c];
    const int mat = (int)(local / per);
    const int rem = (int)(local % per);
    const int tm = rem / L.tiles_n[c], tn = rem % L.tiles_n[c];
    const int sub = C.sub0 + mat;
    const DevSub &S = A.subs[sub];
    const int Mdim = S.p;
    const int Ndim = (gram || square) ? S.p : S.q;
    const int Kdim = gram ? S.q : S.p;
    const T *X = reinterpret_cast<const T *>(A.x_in) + S.x_off;
    const T *Pm = reinterpret_cast<const T *>(square ? A.abuf : A.pbuf) + S.p_off;
    const int m0 = tm * kBM, n0 = tn * kBN;
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;

    for (int k0 = 0; k0 < Kdim; k0 += kBK) {
      {  // A tile: rows m0 .. m0+63, k k0 .. k0+15; thread: row tid/4, k 4*(tid%4)..+3
        const int r = tid >> 2, kk = (tid & 3) * 4;
        const int i = m0 + r;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = k0 + kk + e;
          float v = 0.f;
          if (i < Mdim && k < Kdim)
            v = gram ? to_f(X[(int64_t)i * S.ld + k]) : to_f(Pm[(int64_t)i * S.ldp + k]);
          As[kk + e][r] = v;
        }
      }
      if (gram) {  // B(k, j) = X[j][k]
        const int r = tid >> 2, kk = (tid & 3) * 4;
        const int j = n0 + r;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = k0 + kk + e;
          Bs[kk + e][r] = (j < Ndim && k < Kdim) ? to_f(X[(int64_t)j * S.ld + k]) : 0.f;
        }
      } else {  // B(k, j) = X[k][j] (product) or A[k][j] (square)
        const int kk = tid >> 4, jj = (tid & 15) * 4;
        const int k = k0 + kk;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = n0 + jj + e;
          float v = 0.f;
          if (k < Kdim && j < Ndim)
            v = square ? to_f(Pm[(int64_t)k * S.ldp + j]) : to_f(X[(int64_t)k * S.ld + j]);
          Bs[kk][jj + e] = v;
        }
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < kBK; ++kk) {
        float a[4], b[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          a[e] = As[kk][ty * 4 + e];
          b[e] = Bs[kk][tx * 4 + e];
        }
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
      }
      __syncthreads();
    }
    const EpiScalars e = epi_scalars(A, sub);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int i = m0 + ty * 4 + x;
      if (i >= Mdim) continue;
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int j = n0 + tx * 4 + y;
        if (j < Ndim) ns_epilogue(A, S, e, i, j, acc[x][y]);
      }
    }
  }
}

}  // namespace

int launch_ns_gemm_simt(const ShapeClass *classes, int32_t n_classes, const PhaseArgs &args,
                        int sm_count, void *stream) {
  const bool gram = (args.mode == kGram || args.mode == kGramA);
  const bool square = (args.mode == kSquare);
  for (int32_t c0 = 0; c0 < n_classes; c0 += kMaxClassesPerLaunch) {
    SimtLaunch L{};
    L.n = std::min(kMaxClassesPerLaunch, n_classes - c0);
    L.tile_start[0] = 0;
    for (int k = 0; k < L.n; ++k) {
      const ShapeClass &C = classes[c0 + k];
      L.cls[k] = C;
      const int Ndim = (gram || square) ? C.p : C.q;
      L.tiles_m[k] = (C.p + kBM - 1) / kBM;
      L.tiles_n[k] = (Ndim + kBN - 1) / kBN;
      L.tile_start[k + 1] = L.tile_start[k] + (int64_t)C.count * L.tiles_m[k] * L.tiles_n[k];
    }
    const int64_t total = L.tile_start[L.n];
    if (total == 0) continue;
    const unsigned grid = (unsigned)std::min<int64_t>(total, (int64_t)sm_count * 6);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (args.x_dtype == GBO_BF16)
      ns_gemm_simt_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(L, args);
    else
      ns_gemm_simt_kernel<float><<<grid, kThreads, 0, st>>>(L, args);
    count_launches(1);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return (int)err;
  }
  return 0;
}

}  // namespace gbo
