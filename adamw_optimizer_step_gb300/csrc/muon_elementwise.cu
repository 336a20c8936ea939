// Memory-bound kernels of the Muon path:
//   - momentum + Nesterov direction + per-tile max|D| / sum-of-squares, with
//     the direction written (transposed for tall matrices) into the
//     Newton-Schulz workspace;
//   - the per-matrix reduction of those partials into the pre-normalisation
//     factor;
//   - NorMuon row statistics, row normalisation and the weight write.
//
// Momentum and direction: NorMuon paper (zskr.cn) section 2.2 eq. (1); OMN
// page, Muon path (buffer at 0.95, Nesterov adds the scaled buffer back).
// Pre-normalisation: OMN page, Muon path (max-abs rescale clamped at 1e-7,
// then the Frobenius norm with an additive 1e-7).  NorMuon rows: NorMuon
// paper section 3.1.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "device_common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace gbo {

namespace {

constexpr int kMomThreads = 256;
constexpr int kMomWarps = kMomThreads / 32;  // one partial pair per warp and tile

// One 64 x 64 tile of one matrix per loop trip.  256 threads: thread t
// covers columns 8*(t%8) .. +7 of tile rows t/8 and t/8 + 32.  Every load
// of the tile is issued before any arithmetic, so each thread keeps four
// 16-byte requests in flight.
#ifndef GBO_MOM_MIN_BLOCKS
#define GBO_MOM_MIN_BLOCKS 5  // 5 x 256 threads per SM: measured 3.27 ms vs 4.03 ms at 4 (1.23B set)
#endif
template <typename XT>
__global__ void __launch_bounds__(kMomThreads, GBO_MOM_MIN_BLOCKS)
momentum_kernel(const DevSub *__restrict__ subs, int32_t n_subs, int64_t n_tiles, float mu,
                int32_t nesterov, XT *__restrict__ x0, XT *__restrict__ x0t, float *__restrict__ partials) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up
  pdl_wait();    // the previous kernel has completed and its writes are visible
  __shared__ float tile[kMomTile][kMomTile + 1];
  const int cg = threadIdx.x & 7;
  const int rr = threadIdx.x >> 3;
  // Each block takes a contiguous range of tiles, so the owning matrix is
  // found once and then only advanced.
  const int64_t per = (n_tiles + gridDim.x - 1) / gridDim.x;
  const int64_t t_begin = (int64_t)blockIdx.x * per;
  const int64_t t_end = min(n_tiles, t_begin + per);
  if (t_begin >= t_end) return;
  int si = find_owner(t_begin, n_subs, [&](int k) { return subs[k].tile0; });
  for (int64_t t = t_begin; t < t_end; ++t) {
    while (si + 1 < n_subs && subs[si + 1].tile0 <= t) ++si;
    const DevSub &S = subs[si];
    const int64_t lt = t - S.tile0;
    const bool vec = S.vec_ok != 0;
    float g[2][8], b[2][8], d[2][8];
    float lmax = 0.f;
    if (S.tiles_c == 0) {
      // flat tile: elements [lt * 4096, +4096) of the contiguous matrix;
      // thread t covers 8 consecutive elements in each half
      const int64_t nel = (int64_t)S.m * S.n;
      const int64_t e0 = lt * kMomFlat;
      const int64_t wbase = S.r0 * S.cols;
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        const int64_t e = e0 + ps * (kMomFlat / 2) + threadIdx.x * 8;
        const int valid = (int)max((int64_t)0, min((int64_t)8, nel - e));
        if (valid > 0) {
          load8(S.g, S.g_dtype, wbase + e, valid, vec, g[ps]);
          load8(S.mom, GBO_F32, wbase + e, valid, vec, b[ps]);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) g[ps][k] = b[ps][k] = 0.f;
        }
      }
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        const int64_t e = e0 + ps * (kMomFlat / 2) + threadIdx.x * 8;
        const int valid = (int)max((int64_t)0, min((int64_t)8, nel - e));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float nb = mu * b[ps][k] + g[ps][k];
          b[ps][k] = nb;
          d[ps][k] = k < valid ? (nesterov ? g[ps][k] + mu * nb : nb) : 0.f;
          lmax = fmaxf(lmax, fabsf(d[ps][k]));
        }
        if (valid > 0) {
          store8(S.mom + wbase + e, b[ps], valid, vec);
          store8(x0 + S.x_off + e, d[ps], valid, true);
        }
      }
    } else {
      // 2-D tile (tall matrices, or rows that do not allow 16-byte access)
      const int tr = (int)(lt / S.tiles_c), tc = (int)(lt % S.tiles_c);
      const int rb = tr * kMomTile, cb = tc * kMomTile;
      const int j = cb + cg * 8;
      const int valid = max(0, min(8, S.n - j));
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        const int i = rb + ps * 32 + rr;
        if (i < S.m && valid > 0) {
          const int64_t widx = (S.r0 + i) * S.cols + j;
          load8(S.g, S.g_dtype, widx, valid, vec, g[ps]);
          load8(S.mom, GBO_F32, widx, valid, vec, b[ps]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) g[ps][e] = b[ps][e] = 0.f;
        }
      }
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        const int i = rb + ps * 32 + rr;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float nb = mu * b[ps][e] + g[ps][e];
          b[ps][e] = nb;
          d[ps][e] = nesterov ? g[ps][e] + mu * nb : nb;
          lmax = fmaxf(lmax, fabsf(d[ps][e]));
        }
        if (i < S.m && valid > 0) store8(S.mom + (S.r0 + i) * S.cols + j, b[ps], valid, vec);
      }
      // D itself goes to X, or with a transposed twin (fp32 mode) to XT when X
      // holds D^T; D^T goes to X when transposed, else to XT when it exists.
      // The bf16 mode holds every X in stored orientation: D to X only.
      XT *direct = x0 + S.x_off, *trans = nullptr;
      int ld_direct = S.ld, ld_trans = 0;
      if constexpr (sizeof(XT) == 4) {
        direct = S.transposed ? (S.has_xt ? x0t + S.xt_off : nullptr) : x0 + S.x_off;
        ld_direct = S.transposed ? S.ldt : S.ld;
        trans = S.transposed ? x0 + S.x_off : (S.has_xt ? x0t + S.xt_off : nullptr);
        ld_trans = S.transposed ? S.ld : S.ldt;
      }
      if (direct) {
#pragma unroll
        for (int ps = 0; ps < 2; ++ps) {
          const int i = rb + ps * 32 + rr;
          if (i < S.m && valid > 0) store8(direct + (int64_t)i * ld_direct + j, d[ps], valid, true);
        }
      }
      if (trans) {
        // D^T: stage the tile, then write rows of D^T (columns of D).
        __syncthreads();  // the previous transposed tile's reads are done
#pragma unroll
        for (int ps = 0; ps < 2; ++ps)
#pragma unroll
          for (int e = 0; e < 8; ++e) tile[ps * 32 + rr][cg * 8 + e] = d[ps][e];
        __syncthreads();
#pragma unroll
        for (int ps = 0; ps < 2; ++ps) {
          const int xr = cb + ps * 32 + rr;  // row of X = column of D
          const int xc = rb + cg * 8;        // first column of X = row of D
          const int xvalid = max(0, min(8, S.m - xc));
          if (xr < S.n && xvalid > 0) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = tile[cg * 8 + e][ps * 32 + rr];
            store8(trans + (int64_t)xr * ld_trans + xc, v, xvalid, true);
          }
        }
      }
    }
    // Partials, one pair per warp: the max |D| of the warp's part of the tile
    // and the sum of squares of D / max, so that the per-matrix combination
    // cannot overflow.  Warp shuffles only: no block-wide barrier.
    const float M = warp_max(lmax);
    float ss = 0.f;
    if (M > 0.f) {
      const float inv = 1.0f / M;
#pragma unroll
      for (int ps = 0; ps < 2; ++ps)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float y = d[ps][e] * inv;
          ss = fmaf(y, y, ss);
        }
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) {
      float *pp = partials + 2 * (t * kMomWarps + (threadIdx.x >> 5));
      pp[0] = M;
      pp[1] = ss;
    }
  }
}

// One bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// into shared memory, completing on the mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// The momentum pass streamed through shared memory, for tables whose every
// matrix has flat tiles (bf16 X in stored orientation, G and B rows on
// 16-byte boundaries).  One block per SM, taking either tiles dealt out
// across the blocks (tables of large matrices: all SMs then stream from one
// narrow window of each array at a time) or a contiguous range of tiles
// (tables of many small matrices, where that measured faster).  A block's
// producer warp finds each of its tiles' matrix, moves the tile's
// G and B into shared memory by bulk copies, running ahead of the consumers
// without holding registers, and leaves the tile's destinations and extent
// in a small header beside the stage.  The consumers are kMsGroups groups
// of eight warps: the block's tile i goes to group i % kMsGroups, as that
// group's tile j = i / kMsGroups, into the group's own ring of kPer stages
// (stage j % kPer).  A stage is thus waited on by one group in order, never
// a full phase ahead of its barrier (a parity wait cannot tell that phase
// from the one before it).  Each group takes momentum_kernel's flat-tile
// path on its landed stage, with the same elements per thread, the same
// operations in the same order and the same per-warp partials, so B, X_0
// and the partials are bitwise those of momentum_kernel.  kG is G's element
// size: 2 when every G is bf16 (24 KB stages), else 4 (32 KB stages; a bf16
// G fills half of its slot).
#ifndef GBO_MS_GROUPS
#define GBO_MS_GROUPS 3
#endif
constexpr int kMsGroups = GBO_MS_GROUPS;
constexpr int kMsThreads = kMsGroups * kMomThreads + 32;  // the consumer groups and the producer warp
constexpr int kMsBudget = 216 * 1024;                     // shared memory for stages
constexpr int kMsInterleaveTiles = 512;  // average tiles a matrix from which blocks take dealt-out tiles
template <int kG>
struct MsRing {
  static constexpr int kGBytes = kMomFlat * kG;
  static constexpr int kStageBytes = kGBytes + kMomFlat * 4;
  static constexpr int kPer = kMsBudget / (kMsGroups * kStageBytes);  // stages per group
  static constexpr int kStages = kPer * kMsGroups;
  static constexpr int kSmem = 128 /*align*/ + kStages * kStageBytes;
  static_assert(kPer >= 2, "each consumer group needs two stages at least");
};

// What the producer tells a stage's consumers about the tile in it.
struct MsHdr {
  float *b;            // B at the tile's first element
  __nv_bfloat16 *x;    // X_0 at the tile's first element
  int64_t rem;         // elements from the tile's first to the matrix's end
  int32_t g_bf16, pad;
};

template <int kG>
__global__ void __launch_bounds__(kMsThreads, 1)
momentum_stream_kernel(const DevSub *__restrict__ subs, int32_t n_subs, int64_t n_tiles, float mu,
                       int32_t nesterov, __nv_bfloat16 *__restrict__ x0, float *__restrict__ partials,
                       int32_t *status, int32_t interleave) {
  using R = MsRing<kG>;
  pdl_launch();  // the next kernel may be scheduled as SMs free up
  pdl_wait();    // the previous kernel has completed and its writes are visible
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[R::kStages], empty[R::kStages];
  __shared__ MsHdr hdr[R::kStages];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
  const uint32_t ring = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int st = 0; st < R::kStages; ++st) {
      mbar_init(smem_u32(&full[st]), 1);
      mbar_init(smem_u32(&empty[st]), kMomWarps);  // one arrival per warp of the stage's group
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // the stage of the block's tile i, and the use of that stage it is (its barriers' phase)
  auto stage_of = [](uint32_t i) { return (i % kMsGroups) * R::kPer + (i / kMsGroups) % R::kPer; };
  auto use_of = [](uint32_t i) { return (i / kMsGroups) / R::kPer; };
  // The block's tile i: with `interleave`, tiles are dealt out across the
  // blocks (block b takes b, b + gridDim.x, ...), so all SMs stream from one
  // narrow window of each array at a time; else each block takes a
  // contiguous range.
  const int64_t G = gridDim.x;
  int64_t t_begin, t_step;
  uint32_t n_mine;
  if (interleave) {
    t_begin = blockIdx.x;
    t_step = G;
    n_mine = n_tiles > t_begin ? (uint32_t)((n_tiles - t_begin + G - 1) / G) : 0u;
  } else {
    const int64_t per = (n_tiles + G - 1) / G;
    t_begin = (int64_t)blockIdx.x * per;
    t_step = 1;
    n_mine = n_tiles > t_begin ? (uint32_t)min(per, n_tiles - t_begin) : 0u;
  }
  if (n_mine == 0) return;
  if (warp == kMsGroups * kMomWarps) {  // the producer warp; lane 0 issues every copy
    // The block's tiles are resolved 32 at a time, one per lane (its
    // matrix by binary search, then the copy's sources and the header),
    // while the ring is full; lane 0 then issues them in order.
    int si = find_owner(t_begin, n_subs, [&](int k) { return subs[k].tile0; });
    uint32_t issued = 0;
    bool timed_out = false;
    while (issued < n_mine && !timed_out) {
      const uint32_t ij = min(issued + (uint32_t)lane, n_mine - 1);
      const int64_t tj = t_begin + (int64_t)ij * t_step;
      int lo = si, hi = n_subs - 1;  // the last matrix whose first tile is <= tj
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (subs[mid].tile0 <= tj) lo = mid;
        else hi = mid - 1;
      }
      const DevSub &S = subs[lo];
      const uint32_t gsz = S.g_dtype == GBO_BF16 ? 2u : 4u;
      const int64_t e0 = (tj - S.tile0) * kMomFlat, w = S.r0 * S.cols + e0;
      const uint64_t gsrc = reinterpret_cast<uint64_t>(reinterpret_cast<const uint8_t *>(S.g) + w * gsz);
      const uint64_t bsrc = reinterpret_cast<uint64_t>(S.mom + w);
      const uint64_t xdst = reinterpret_cast<uint64_t>(x0 + S.x_off + e0);
      const int64_t rem = (int64_t)S.m * S.n - e0;
      si = __shfl_sync(0xffffffffu, lo, 31);  // owners are nondecreasing over the lanes
      const uint32_t batch = min(32u, n_mine - issued);
      for (uint32_t j = 0; j < batch; ++j) {
        const uint64_t g_j = __shfl_sync(0xffffffffu, gsrc, j), b_j = __shfl_sync(0xffffffffu, bsrc, j);
        const uint64_t x_j = __shfl_sync(0xffffffffu, xdst, j);
        const int64_t r_j = __shfl_sync(0xffffffffu, rem, j);
        const uint32_t gz_j = __shfl_sync(0xffffffffu, gsz, j);
        if (lane == 0) {
          const uint32_t i = issued, st = stage_of(i), use = use_of(i);
          if (use > 0 && !mbar_wait(smem_u32(&empty[st]), (use - 1) & 1u)) {
            flag_status(status, GBO_STATUS_TIMEOUT);
            timed_out = true;
          } else {
            const uint32_t n = (uint32_t)min((int64_t)kMomFlat, r_j);
            hdr[st] = MsHdr{reinterpret_cast<float *>(b_j), reinterpret_cast<__nv_bfloat16 *>(x_j), r_j,
                            gz_j == 2u ? 1 : 0};
            const uint32_t bar = smem_u32(&full[st]), dst = ring + st * R::kStageBytes;
            mbar_expect_tx(bar, n * (gz_j + 4u));  // releases the header to the stage's consumers
            bulk_load(dst, reinterpret_cast<const void *>(g_j), n * gz_j, bar);
            bulk_load(dst + R::kGBytes, reinterpret_cast<const void *>(b_j), n * 4u, bar);
          }
        }
        timed_out = __shfl_sync(0xffffffffu, timed_out ? 1 : 0, 0) != 0;
        if (timed_out) break;
        ++issued;
      }
    }
    // after a timeout: the copies in flight land before shared memory goes
    // away (tiles are issued round-robin over the groups, so the last kStages
    // issued use each stage once, each its latest use)
    if (lane == 0 && timed_out)
      for (uint32_t k = issued > (uint32_t)R::kStages ? issued - R::kStages : 0u; k < issued; ++k)
        (void)mbar_wait(smem_u32(&full[stage_of(k)]), use_of(k) & 1u);
    return;
  }
  const int grp = warp / kMomWarps, cw = warp % kMomWarps, ct = threadIdx.x % kMomThreads;
  for (uint32_t i = (uint32_t)grp; i < n_mine; i += kMsGroups) {
    const int64_t t = t_begin + (int64_t)i * t_step;
    const uint32_t st = stage_of(i);
    if (!mbar_wait(smem_u32(&full[st]), use_of(i) & 1u)) {
      flag_status(status, GBO_STATUS_TIMEOUT);
      break;
    }
    const MsHdr hd = hdr[st];  // the tile's destinations and extent, from the producer
    const uint32_t gs = ring + st * R::kStageBytes, bs = gs + R::kGBytes;
    const bool gbf = hd.g_bf16 != 0;
    float g[2][8], b[2][8], d[2][8];
    float lmax = 0.f;
#pragma unroll
    for (int ps = 0; ps < 2; ++ps) {
      const int el = ps * (kMomFlat / 2) + ct * 8;  // element within the tile
      const int valid = (int)max((int64_t)0, min((int64_t)8, hd.rem - el));
      uint32_t r[8];
      if (gbf) {
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(gs + el * 2)
                     : "memory");
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&r[h]);
          g[ps][2 * h] = __low2float(v);
          g[ps][2 * h + 1] = __high2float(v);
        }
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(g[ps][4 * h]), "=f"(g[ps][4 * h + 1]), "=f"(g[ps][4 * h + 2]), "=f"(g[ps][4 * h + 3])
                       : "r"(gs + el * 4 + 16 * h)
                       : "memory");
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(b[ps][4 * h]), "=f"(b[ps][4 * h + 1]), "=f"(b[ps][4 * h + 2]), "=f"(b[ps][4 * h + 3])
                     : "r"(bs + el * 4 + 16 * h)
                     : "memory");
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k >= valid) g[ps][k] = b[ps][k] = 0.f;  // past the matrix: what landed there is stale
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[st]));  // the warp has read the stage
#pragma unroll
    for (int ps = 0; ps < 2; ++ps) {
      const int el = ps * (kMomFlat / 2) + ct * 8;
      const int valid = (int)max((int64_t)0, min((int64_t)8, hd.rem - el));
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float nb = mu * b[ps][k] + g[ps][k];
        b[ps][k] = nb;
        d[ps][k] = k < valid ? (nesterov ? g[ps][k] + mu * nb : nb) : 0.f;
        lmax = fmaxf(lmax, fabsf(d[ps][k]));
      }
      if (valid > 0) {
        store8(hd.b + el, b[ps], valid, true);
        store8(hd.x + el, d[ps], valid, true);
      }
    }
    const float M = warp_max(lmax);
    float ss = 0.f;
    if (M > 0.f) {
      const float inv = 1.0f / M;
#pragma unroll
      for (int ps = 0; ps < 2; ++ps)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float y = d[ps][k] * inv;
          ss = fmaf(y, y, ss);
        }
    }
    ss = warp_sum(ss);
    if (lane == 0) {
      float *pp = partials + 2 * (t * kMomWarps + cw);
      pp[0] = M;
      pp[1] = ss;
    }
  }
}

// The finalize sums each matrix's partials as kFinLanes virtual lanes (lane v
// takes partials v, v + kFinLanes, ... in order), then in a fixed tree: the
// 32 lanes of each virtual warp, then the 32 warps.  A block of kT threads
// runs kFinLanes / kT lanes per thread, so the sums do not depend on kT
// (1024 threads when there are fewer matrices than SMs, so that a few large
// matrices are reduced by many threads; 256 when there are many).  The max
// comes first, from a block reduction (a max is the same in any order).
constexpr int kFinLanes = 1024;

// One block per matrix: combine the tile partials (max |D| and the sum of
// (D / max)^2 of each warp's elements) in that fixed order into
// alpha = 1 / (s * (||D / s||_F + 1e-7)), s = max(max|D|, 1e-7), so that
// X0 = alpha * D.
template <int kT>
__global__ void __launch_bounds__(kT)
prenorm_finalize_kernel(const DevSub *__restrict__ subs, const float *__restrict__ partials,
                        float *__restrict__ alpha, int32_t *status, float *__restrict__ stats) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up
  pdl_wait();    // the previous kernel has completed and its writes are visible
  constexpr int R = kFinLanes / kT;  // virtual lanes per thread
  static_assert(R >= 1 && kFinLanes % kT == 0 && kFinLanes / 32 == 32, "lane layout");
  __shared__ float red[32];
  const DevSub &S = subs[blockIdx.x];
  if (S.mom_fused) return;  // the chain kernel forms this matrix's factor
  const int64_t nt = (int64_t)S.ntiles * kMomWarps;
  const float2 *P = reinterpret_cast<const float2 *>(partials) + S.tile0 * kMomWarps;
  // the max, four partials in flight per thread
  float M = 0.f;
  {
    int64_t k = threadIdx.x;
    for (; k + 3 * kT < nt; k += 4 * kT) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = P[k + u * kT].x;
#pragma unroll
      for (int u = 0; u < 4; ++u) M = fmaxf(M, v[u]);
    }
    for (; k < nt; k += kT) M = fmaxf(M, P[k].x);
  }
  M = block_max(M, red);
  // the sum of squares relative to M, lane by lane
  float ss[R];
#pragma unroll
  for (int r = 0; r < R; ++r) ss[r] = 0.f;
  if (M > 0.f) {
    const float inv = 1.0f / M;
    if constexpr (R == 1) {  // four of the lane's partials in flight, summed in order
      int64_t k = threadIdx.x;
      for (; k + 3 * kFinLanes < nt; k += 4 * kFinLanes) {
        float2 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = P[k + u * kFinLanes];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float x = v[u].x * inv;
          ss[0] = fmaf(v[u].y, x * x, ss[0]);
        }
      }
      for (; k < nt; k += kFinLanes) {
        const float2 v = P[k];
        const float x = v.x * inv;
        ss[0] = fmaf(v.y, x * x, ss[0]);
      }
    } else {  // one partial of each of the thread's R lanes in flight
      for (int64_t k = threadIdx.x; k < nt; k += kFinLanes) {
        float2 v[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (k + r * kT < nt) v[r] = P[k + r * kT];
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (k + r * kT < nt) {
            const float x = v[r].x * inv;
            ss[r] = fmaf(v[r].y, x * x, ss[r]);
          }
      }
    }
  }
  // each virtual warp's 32 lanes (the physical warp's lanes), then the
  // warps; warps without partials hold zeros and skip their shuffles
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();  // red is free again
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int vw = warp + r * (kT / 32);
    float t = ss[r];
    if ((int64_t)vw * 32 < nt) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_down_sync(0xffffffffu, t, o);
    }
    if (lane == 0) red[vw] = t;
  }
  __syncthreads();
  if (warp != 0) return;
  float t = red[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_down_sync(0xffffffffu, t, o);
  if (lane == 0) {
    const float s = fmaxf(M, 1e-7f);
    const float normY = (M / s) * sqrtf(t);
    float a = 1.0f / (s * (normY + 1e-7f));
    if (!isfinite(M) || !isfinite(t) || !isfinite(a)) {
      flag_status(status, GBO_STATUS_NONFINITE);
      a = __int_as_float(0x7fc00000);
    }
    alpha[blockIdx.x] = a;
    if (stats) stats[2 * S.mat_idx] = M > 0.f ? M * sqrtf(t) : (isfinite(M) ? 0.f : M);  // ||D||_F
  }
}

// ||U||_F of every matrix (one block each), from partial sums the step left
// in the workspace, combined in a fixed order:
//   without NorMuon  the last product's per-(stored row, 128 columns) sums of
//                    U^2 (rowss, m x ss_ntn values from ss_off)
//   NorMuon          the rows pass's per-row-block sums of
//                    (1 / (sqrt(v) + eps))^2 ||X_i||^2 = ||O_hat||_F^2 of the
//                    block (rowpart, from rb0); U = scale * O_hat, or with
//                    the RMS-keeping scale rms sqrt(m n) O_hat / ||O_hat||_F
__global__ void __launch_bounds__(256)
stats_finalize_kernel(const DevSub *__restrict__ subs, int32_t normuon, float rms_target,
                      const float *__restrict__ rowss, const float *__restrict__ rowpart,
                      float *__restrict__ stats) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up
  pdl_wait();    // the previous kernel has completed and its writes are visible
  __shared__ float red[32];
  const DevSub &S = subs[blockIdx.x];
  float t = 0.f;
  if (normuon) {
    const int nb = (S.m + kRowBlock - 1) / kRowBlock;
    for (int k = threadIdx.x; k < nb; k += blockDim.x) t += rowpart[S.rb0 + k];
  } else {
    const int64_t n = (int64_t)S.m * S.ss_ntn;
    for (int64_t k = threadIdx.x; k < n; k += blockDim.x) t += rowss[S.ss_off + k];
  }
  t = block_sum(t, red);
  if (threadIdx.x == 0) {
    float u;
    if (!normuon) u = sqrtf(t);
    else if (rms_target > 0.f) u = t > 0.f ? rms_target * sqrtf((float)S.m * (float)S.n) : (t == 0.f ? 0.f : t);
    else u = S.scale * sqrtf(t);
    stats[2 * S.mat_idx + 1] = u;
  }
}

// Eight consecutive fp32 values from X (bf16 or fp32 workspace): 16-byte
// loads when the segment is whole (the workspace rows are 16-element
// aligned), else element by element.
template <typename XT>
__device__ __forceinline__ void load8x(const XT *src, int valid, float *out) {
  if (valid == 8) {
    if constexpr (sizeof(XT) == 2) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(src);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[h]);
        out[2 * h] = __low2float(b);
        out[2 * h + 1] = __high2float(b);
      }
    } else {
      const float4 a = reinterpret_cast<const float4 *>(src)[0], b = reinterpret_cast<const float4 *>(src)[1];
      out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
      out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if constexpr (sizeof(XT) == 2) out[e] = e < valid ? __bfloat162float(src[e]) : 0.f;
      else out[e] = e < valid ? src[e] : 0.f;
    }
  }
}

// W[widx .. widx + valid) <- W - lrm * (wd * W + f * o), and the update f * o
// to dbg; 16-byte accesses when `vec` and the segment is whole.
__device__ __forceinline__ void weight_rmw8(const DevSub &S, int64_t widx, int valid, bool vec, float lrm, float f,
                                            const float *o, float *dbg) {
  float w[8], u[8];
  load8(S.w, S.w_dtype, widx, valid, vec, w);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    u[e] = f * o[e];
    w[e] = w[e] - lrm * (S.wd * w[e] + u[e]);
  }
  if (S.w_dtype == GBO_BF16) store8(reinterpret_cast<__nv_bfloat16 *>(S.w) + widx, w, valid, vec);
  else store8(reinterpret_cast<float *>(S.w) + widx, w, valid, vec);
  if (dbg) {
    float *d = dbg + S.dbg_off + widx;
    store8(d, u, valid, (reinterpret_cast<uintptr_t>(d) & 15) == 0);
  }
}

// NorMuon rows of the plan's matrices: one block of 256 threads per
// kRowBlock stored rows of one matrix.  O (the unscaled orthogonalised
// update) is read from the workspace.  Row statistics, v update, then the
// weight write, with 16-byte accesses throughout.
//   untransposed: warp w takes stored rows w, w + 8, ... of the block; a
//     row is X's row.  Its statistics come from the last product's partial
//     sums of squares (rowss, bf16 mode: one per 128 columns of the row,
//     summed in a fixed order), or from a first read of the row; the
//     write reads it (again), two 256-element segments per step with every
//     load issued before the stores (two segments kept 64 registers; four
//     took 119 and were slower)
//   transposed (fp32 mode): stored row i is column i of X; the block reads
//     32 x 64 tiles of X (8 threads per 64-column row segment), keeps
//     per-column sums, then transposes tiles through shared memory for the
//     write
// kMode selects the pass (NorMuon paper, section 3.1):
//   0  statistics and write, f_i = scale / (sqrt(v_i) + eps)
//   1  statistics only, for the RMS-keeping scale: f_i = 1 / (sqrt(v_i) + eps)
//      to rowf, and the block's sum of f_i^2 * sum_j X_ij^2 (its share of
//      ||O_hat||_F^2) to rowpart
//   2  write only, f_i = mscale[matrix] * rowf[i]
template <typename XT, int kMode>
__global__ void __launch_bounds__(256)
normuon_rows_kernel(const DevSub *__restrict__ subs, int32_t n_subs, int64_t n_blocks,
                    const XT *__restrict__ xbuf0, const XT *__restrict__ xbuf1, float beta2, float eps, float lr,
                    float *__restrict__ dbg, int32_t *status, float *__restrict__ rowf,
                    float *__restrict__ rowpart, const float *__restrict__ mscale,
                    const float *__restrict__ rowss) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up
  pdl_wait();    // the previous kernel has completed and its writes are visible
  __shared__ float tileT[32][kRowBlock + 1];
  __shared__ float colsum[32][kRowBlock + 1];
  __shared__ float rfac[kRowBlock];
  __shared__ float red[kRowBlock];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t b = blockIdx.x; b < n_blocks; b += gridDim.x) {
    const int si = find_owner(b, n_subs, [&](int k) { return subs[k].rb0; });
    const DevSub &S = subs[si];
    const int i0 = (int)(b - S.rb0) * kRowBlock;
    const int nrows = min(kRowBlock, S.m - i0);
    const XT *X = (S.x_sel ? xbuf1 : xbuf0) + S.x_off;  // the buffer holding the last iterate
    const float lrm = lr * S.lr_mult;
    const bool wvec = S.w_vec != 0;
    float *rf = rowf + b * kRowBlock;  // per-row factors of this block (modes 1, 2)
    if (!S.transposed) {
      float part = 0.f;  // mode 1: this warp's share of the block partial
      for (int r = warp; r < nrows; r += 8) {
        const int row = i0 + r;
        const XT *xr = X + (int64_t)row * S.ld;
        const int64_t vrow = S.r0 + row;
        float f;
        if constexpr (kMode != 2) {
          float ss = 0.f;
          int j = rowss ? S.n : lane * 8;  // with the partials, X is not read here
          if (rowss) {
            const float *part = rowss + S.ss_off + (int64_t)row * S.ss_ntn;
            for (int t = lane; t < S.ss_ntn; t += 32) ss += part[t];
          }
          for (; j + 1 * 256 + 8 <= S.n; j += 2 * 256) {  // two whole segments: loads first
            float o[2][8];
#pragma unroll
            for (int u = 0; u < 2; ++u) load8x(xr + j + u * 256, 8, o[u]);
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
              for (int e = 0; e < 8; ++e) ss = fmaf(o[u][e], o[u][e], ss);
          }
          for (; j < S.n; j += 256) {
            float o[8];
            load8x(xr + j, min(8, S.n - j), o);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(o[e], o[e], ss);
          }
          ss = warp_sum(ss);
          const float v = beta2 * S.row_v[vrow] + (1.0f - beta2) * (ss / (float)S.n);
          f = (kMode == 0 ? S.scale : 1.0f) / (sqrtf(v) + eps);
          if (!isfinite(f)) flag_status(status, GBO_STATUS_NONFINITE);
          __syncwarp();
          if (lane == 0) S.row_v[vrow] = v;
          if constexpr (kMode == 1) {
            if (lane == 0) rf[r] = f;
            part = fmaf(f * f, ss, part);
          } else {
            const float g = 1.0f / (sqrtf(v) + eps);  // the row's factor without the scale
            part = fmaf(g * g, ss, part);             // (its share of ||O_hat||_F^2, for the norms)
          }
        } else {
          f = mscale[si] * rf[r];
        }
        if constexpr (kMode != 1) {
          int j = lane * 8;
          for (; j + 1 * 256 + 8 <= S.n; j += 2 * 256) {  // two whole segments: all loads, then the stores
            float o[2][8], w[2][8];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              load8x(xr + j + u * 256, 8, o[u]);
              load8(S.w, S.w_dtype, vrow * S.cols + j + u * 256, 8, wvec, w[u]);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              float uu[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                uu[e] = f * o[u][e];
                w[u][e] = w[u][e] - lrm * (S.wd * w[u][e] + uu[e]);
              }
              const int64_t widx = vrow * S.cols + j + u * 256;
              if (S.w_dtype == GBO_BF16) store8(reinterpret_cast<__nv_bfloat16 *>(S.w) + widx, w[u], 8, wvec);
              else store8(reinterpret_cast<float *>(S.w) + widx, w[u], 8, wvec);
              if (dbg) {
                float *d = dbg + S.dbg_off + widx;
                store8(d, uu, 8, (reinterpret_cast<uintptr_t>(d) & 15) == 0);
              }
            }
          }
          for (; j < S.n; j += 256) {
            const int valid = min(8, S.n - j);
            float o[8];
            load8x(xr + j, valid, o);
            weight_rmw8(S, vrow * S.cols + j, valid, wvec, lrm, f, o, dbg);
          }
        }
      }
      if (kMode == 1 || (kMode == 0 && rowpart)) {  // fixed-order block sum of the warps' shares
        if (lane == 0) red[warp] = part;
        __syncthreads();
        if (threadIdx.x == 0) {
          float t = 0.f;
          for (int w = 0; w < 8; ++w) t += red[w];
          rowpart[b] = t;
        }
      }
    } else {
      const int cg = threadIdx.x & 7, rr = threadIdx.x >> 3;  // 8 columns x 32 rows of X per pass
      const int c = i0 + cg * 8;                                // first X column (stored row)
      const int cvalid = max(0, min(8, i0 + nrows - c));
      if constexpr (kMode != 2) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int j = rr; j < S.n; j += 32) {
          if (cvalid > 0) {
            float o[8];
            load8x(X + (int64_t)j * S.ld + c, cvalid, o);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(o[e], o[e], acc[e]);
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) colsum[rr][cg * 8 + e] = acc[e];
        __syncthreads();
        float part = 0.f;
        if (threadIdx.x < nrows) {
          float ss = 0.f;
          for (int k = 0; k < 32; ++k) ss += colsum[k][threadIdx.x];  // fixed order
          const int64_t vrow = S.r0 + i0 + threadIdx.x;
          const float v = beta2 * S.row_v[vrow] + (1.0f - beta2) * (ss / (float)S.n);
          S.row_v[vrow] = v;
          const float f = (kMode == 0 ? S.scale : 1.0f) / (sqrtf(v) + eps);
          if (!isfinite(f)) flag_status(status, GBO_STATUS_NONFINITE);
          rfac[threadIdx.x] = f;
          if constexpr (kMode == 1) {
            rf[threadIdx.x] = f;
            part = f * f * ss;
          } else {
            const float g = 1.0f / (sqrtf(v) + eps);
            part = g * g * ss;
          }
        }
        if (kMode == 1 || rowpart) {
          if (threadIdx.x < kRowBlock) red[threadIdx.x] = part;
          __syncthreads();
          if (threadIdx.x == 0) {
            float t = 0.f;
            for (int k = 0; k < kRowBlock; ++k) t += red[k];  // fixed order
            rowpart[b] = t;
          }
        }
      } else {
        if (threadIdx.x < nrows) rfac[threadIdx.x] = mscale[si] * rf[threadIdx.x];
      }
      __syncthreads();
      if constexpr (kMode != 1) {
        // write: stored rows i0 + k (k < nrows), stored columns j0 .. j0 + 31
        const int k = threadIdx.x >> 2, seg = threadIdx.x & 3;  // 64 rows x 4 segments of 8
        for (int j0 = 0; j0 < S.n; j0 += 32) {
          {
            const int j = j0 + rr;
            float o[8];
            if (j < S.n && cvalid > 0) load8x(X + (int64_t)j * S.ld + c, cvalid, o);
            else
#pragma unroll
              for (int e = 0; e < 8; ++e) o[e] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) tileT[rr][cg * 8 + e] = o[e];
          }
          __syncthreads();
          const int jc = j0 + seg * 8;
          const int valid = max(0, min(8, S.n - jc));
          if (k < nrows && valid > 0) {
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = tileT[seg * 8 + e][k];
            weight_rmw8(S, (S.r0 + i0 + k) * S.cols + jc, valid, wvec, lrm, rfac[k], o, dbg);
          }
          __syncthreads();
        }
      }
    }
    __syncthreads();
  }
}

// The NorMuon write pass streamed through shared memory (bf16 X and bf16
// weights whose rows start on 16-byte boundaries): each warp takes whole
// stored rows and moves them in 512-element segments, X's and W's, by bulk
// copies into a ring of kWStages stages of its own, kept full across its
// rows, so the loads run ahead without holding registers; the warp reads a
// landed stage, computes the new weights and stores them with 16-byte vector
// stores.  The row factors come from the statistics pass (rowf, 1 / (sqrt(v)
// + eps)), times the rectangular scale (kMode 0) or the RMS scale (kMode 2);
// each is read when its row's first segment is loaded, so no row waits for
// it (NorMuon paper, section 3.1, as normuon_rows_kernel).
constexpr int kSeg = 512;
constexpr int kWStages = 3;
constexpr int kWWarps = 32;  // 1024 threads, 192 KB of copies in flight per SM
constexpr int kWStageBytes = 2 * kSeg * 2;  // a segment of X and of W, bf16
constexpr int kWSmem = 128 /*align*/ + kWWarps * kWStages * kWStageBytes;

// A warp's walk over stored rows: row slots slot, slot + stride, ... of the
// plan's row blocks (kRowBlock slots each), skipping slots past a matrix's
// rows.
struct RowCursor {
  int64_t slot;
  int si, row, seg;  // matrix, row within it, segment
};

__device__ __forceinline__ bool row_at(const DevSub *subs, int32_t n_subs, int64_t n_slots, int64_t stride,
                                       RowCursor &c) {
  for (; c.slot < n_slots; c.slot += stride) {
    const int64_t b = c.slot / kRowBlock;
    c.si = find_owner(b, n_subs, [&](int k) { return subs[k].rb0; });
    c.row = (int)(b - subs[c.si].rb0) * kRowBlock + (int)(c.slot % kRowBlock);
    if (c.row < subs[c.si].m) {
      c.seg = 0;
      return true;
    }
  }
  return false;
}

__device__ __forceinline__ bool row_next(const DevSub *subs, int32_t n_subs, int64_t n_slots, int64_t stride,
                                         RowCursor &c) {
  if (++c.seg * kSeg < subs[c.si].n) return true;
  c.slot += stride;
  return row_at(subs, n_subs, n_slots, stride, c);
}

template <int kMode>
__global__ void __launch_bounds__(kWWarps * 32, 1)
normuon_write_kernel(const DevSub *__restrict__ subs, int32_t n_subs, int64_t n_slots,
                     const __nv_bfloat16 *__restrict__ xbuf0, const __nv_bfloat16 *__restrict__ xbuf1, float beta2,
                     float eps, float lr, float *__restrict__ dbg, int32_t *status, const float *__restrict__ rowf,
                     const float *__restrict__ mscale) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up
  pdl_wait();    // the previous kernel has completed and its writes are visible
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[kWWarps * kWStages];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring = smem_u32(smem) + (uint32_t)(warp * kWStages * kWStageBytes);
  const uint32_t bar0 = smem_u32(&bars[warp * kWStages]);
  if (lane == 0) {
    for (int st = 0; st < kWStages; ++st) mbar_init(bar0 + 8 * st, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  const int64_t stride = (int64_t)gridDim.x * kWWarps;
  RowCursor ic{(int64_t)blockIdx.x * kWWarps + warp, 0, 0, 0};
  bool ic_ok = row_at(subs, n_subs, n_slots, stride, ic);
  RowCursor cc = ic;
  bool cc_ok = ic_ok;
  uint32_t issued = 0, consumed = 0;
  float fq[kWStages];  // lane 0: the row factor of each stage's segment
  // lane 0 loads the stream's next segment into its stage
  auto issue = [&]() {
    const DevSub &S = subs[ic.si];
    const __nv_bfloat16 *X = (S.x_sel ? xbuf1 : xbuf0) + S.x_off + (int64_t)ic.row * S.ld + (int64_t)ic.seg * kSeg;
    const __nv_bfloat16 *W =
        reinterpret_cast<const __nv_bfloat16 *>(S.w) + (S.r0 + ic.row) * S.cols + (int64_t)ic.seg * kSeg;
    const uint32_t bytes = (uint32_t)min(kSeg, S.n - ic.seg * kSeg) * 2u;
    const uint32_t st = issued % kWStages, bar = bar0 + 8 * st, dst = ring + st * kWStageBytes;
    mbar_expect_tx(bar, 2 * bytes);
    bulk_load(dst, X, bytes, bar);
    bulk_load(dst + kSeg * 2, W, bytes, bar);
    const float g = ic.seg == 0 ? rowf[ic.slot] * (kMode == 0 ? S.scale : mscale[ic.si]) : 0.f;
#pragma unroll
    for (int k = 0; k < kWStages; ++k)
      if (k == (int)st) fq[k] = g;
  };
  while (ic_ok && issued < (uint32_t)kWStages) {
    if (lane == 0) issue();
    ++issued;
    ic_ok = row_next(subs, n_subs, n_slots, stride, ic);
  }
  float f = 0.f;
  bool timed_out = false;
  while (cc_ok) {
    const DevSub &S = subs[cc.si];
    const int64_t vrow = S.r0 + cc.row;
    const uint32_t st = consumed % kWStages;
    if (cc.seg == 0) {  // the row's factor, loaded with its first segment
      float g = 0.f;
#pragma unroll
      for (int k = 0; k < kWStages; ++k)
        if (k == (int)st) g = fq[k];
      f = __shfl_sync(0xffffffffu, g, 0);
    }
    if (!mbar_wait(bar0 + 8 * st, (consumed / kWStages) & 1u)) {
      flag_status(status, GBO_STATUS_TIMEOUT);
      timed_out = true;
      break;
    }
    const uint32_t xs = ring + st * kWStageBytes, ws = xs + kSeg * 2;
    const int base = cc.seg * kSeg, len = min(kSeg, S.n - base);
    const float lrm = lr * S.lr_mult;
    __nv_bfloat16 *W = reinterpret_cast<__nv_bfloat16 *>(S.w) + vrow * S.cols + base;
    for (int g = lane; g * 8 < len; g += 32) {  // eight elements per lane and step
      uint32_t xr[4], wr[4];
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(xr[0]), "=r"(xr[1]), "=r"(xr[2]), "=r"(xr[3])
                   : "r"(xs + g * 16)
                   : "memory");
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(wr[0]), "=r"(wr[1]), "=r"(wr[2]), "=r"(wr[3])
                   : "r"(ws + g * 16)
                   : "memory");
      float o[8], w[8], u[8];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const __nv_bfloat162 xb = *reinterpret_cast<const __nv_bfloat162 *>(&xr[h]);
        const __nv_bfloat162 wb = *reinterpret_cast<const __nv_bfloat162 *>(&wr[h]);
        o[2 * h] = __low2float(xb);
        o[2 * h + 1] = __high2float(xb);
        w[2 * h] = __low2float(wb);
        w[2 * h + 1] = __high2float(wb);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        u[e] = f * o[e];
        w[e] = w[e] - lrm * (S.wd * w[e] + u[e]);
      }
      store8(W + g * 8, w, 8, true);
      if (dbg) {
        float *d = dbg + S.dbg_off + vrow * S.cols + base + g * 8;
        store8(d, u, 8, (reinterpret_cast<uintptr_t>(d) & 15) == 0);
      }
    }
    __syncwarp();  // every lane has read the stage
    ++consumed;
    cc_ok = row_next(subs, n_subs, n_slots, stride, cc);
    if (ic_ok) {
      if (lane == 0) issue();
      ++issued;
      ic_ok = row_next(subs, n_subs, n_slots, stride, ic);
    }
  }
  if (timed_out)  // the copies in flight land before shared memory goes away
    for (uint32_t k = consumed; k < issued; ++k) (void)mbar_wait(bar0 + 8 * (k % kWStages), (k / kWStages) & 1u);
}

// The RMS-keeping scale of each matrix (one block per matrix): the row-block
// partials of ||O_hat||_F^2 summed in a fixed order, then
// rho * sqrt(m n) / ||O_hat||_F; an all-zero update keeps a zero scale.
__global__ void __launch_bounds__(256)
normuon_scale_kernel(const DevSub *__restrict__ subs, const float *__restrict__ rowpart, float rho,
                     float *__restrict__ mscale, int32_t *status) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up
  pdl_wait();    // the previous kernel has completed and its writes are visible
  __shared__ float red[32];
  const DevSub &S = subs[blockIdx.x];
  const int nb = (S.m + kRowBlock - 1) / kRowBlock;
  float t = 0.f;
  for (int k = threadIdx.x; k < nb; k += blockDim.x) t += rowpart[S.rb0 + k];
  t = block_sum(t, red);
  if (threadIdx.x == 0) {
    float g = t > 0.f ? rho * sqrtf((float)S.m * (float)S.n) / sqrtf(t) : 0.f;
    if (!isfinite(t) || !isfinite(g)) {
      flag_status(status, GBO_STATUS_NONFINITE);
      g = __int_as_float(0x7fc00000);
    }
    mscale[blockIdx.x] = g;
  }
}

// Stand-alone NorMuon rows on a plain fp32 O (rows x cols): one block per
// kRowBlock rows.
__global__ void __launch_bounds__(256)
rownorm_plain_kernel(const float *__restrict__ O, int64_t rows, int64_t cols, float *__restrict__ row_v,
                     void *w, int32_t w_dtype, float beta2, float eps, float scale, float lr,
                     float wd, float *__restrict__ dbg) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up
  pdl_wait();    // the previous kernel has completed and its writes are visible
  __shared__ float rinv[kRowBlock];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t b = blockIdx.x; b * kRowBlock < rows; b += gridDim.x) {
    const int64_t i0 = b * kRowBlock;
    const int nrows = (int)min((int64_t)kRowBlock, rows - i0);
    for (int r = warp; r < nrows; r += 8) {
      const float *o = O + (i0 + r) * cols;
      float ss = 0.f;
      for (int64_t j = lane; j < cols; j += 32) ss = fmaf(o[j], o[j], ss);
      ss = warp_sum(ss);
      if (lane == 0) {
        const float v = beta2 * row_v[i0 + r] + (1.0f - beta2) * (ss / (float)cols);
        row_v[i0 + r] = v;
        rinv[r] = scale / (sqrtf(v) + eps);
      }
    }
    __syncthreads();
    for (int r = warp; r < nrows; r += 8) {
      const int64_t base = (i0 + r) * cols;
      for (int64_t j = lane; j < cols; j += 32) {
        const float u = rinv[r] * O[base + j];
        const float wv = ld_elem(w, w_dtype, base + j);
        st_elem(w, w_dtype, base + j, wv - lr * (wd * wv + u));
        if (dbg) dbg[base + j] = u;
      }
    }
    __syncthreads();
  }
}

}  // namespace

namespace {
std::atomic<int32_t> g_mom_stream{1};  // see gbo_testing_set_momentum_stream
}  // namespace

int32_t set_momentum_stream(int32_t enable) { return g_mom_stream.exchange(enable != 0 ? 1 : 0); }

int launch_momentum(const DevSub *subs, int32_t n_subs, int64_t n_tiles, float mu, int32_t nesterov,
                    void *x0, void *x0t, int32_t x_dtype, float *partials, int32_t stream_g, int32_t *status,
                    int sm_count, void *stream) {
  if (n_tiles == 0) return 0;
  if (stream_g && x_dtype == GBO_BF16 && g_mom_stream.load()) {
    static const cudaError_t attr_err = [] {
      cudaError_t e = cudaFuncSetAttribute(momentum_stream_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           MsRing<2>::kSmem);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(momentum_stream_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 MsRing<4>::kSmem);
      return e;
    }();
    if (attr_err != cudaSuccess) return (int)attr_err;
    const int64_t grid = std::min<int64_t>(n_tiles, (int64_t)sm_count);
    // tiles dealt out across the blocks when the matrices average at least
    // kMsInterleaveTiles tiles: bench set (1792 a matrix) momentum 2.49 ->
    // 2.37-2.43 ms, 7B set 13.2 -> 12.5 ms; the 9216 MLA/KDA matrices (82 a
    // matrix) 5.85 -> 6.25 ms, so they keep contiguous ranges
    const int32_t interleave = n_tiles >= (int64_t)kMsInterleaveTiles * n_subs ? 1 : 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    __nv_bfloat16 *x = reinterpret_cast<__nv_bfloat16 *>(x0);
    const cudaError_t err =
        stream_g == 2
            ? launch_kernel(momentum_stream_kernel<2>, dim3((unsigned)grid), dim3(kMsThreads), MsRing<2>::kSmem, st, 1,
                            subs, n_subs, n_tiles, mu, nesterov, x, partials, status, interleave)
            : launch_kernel(momentum_stream_kernel<4>, dim3((unsigned)grid), dim3(kMsThreads), MsRing<4>::kSmem, st, 1,
                            subs, n_subs, n_tiles, mu, nesterov, x, partials, status, interleave);
    count_launches(1);
    return (int)err;
  }
  // one wave: as many blocks as can be resident, each a contiguous tile range
  static int resident[2] = {0, 0};
  const int which = x_dtype == GBO_BF16 ? 0 : 1;
  if (!resident[which]) {
    int r = 0;
    const cudaError_t e = x_dtype == GBO_BF16
        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, momentum_kernel<__nv_bfloat16>, kMomThreads, 0)
        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, momentum_kernel<float>, kMomThreads, 0);
    resident[which] = (e == cudaSuccess && r > 0) ? r : 4;
  }
  const int64_t grid = std::min<int64_t>(n_tiles, (int64_t)sm_count * resident[which]);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t err =
      x_dtype == GBO_BF16
          ? launch_kernel(momentum_kernel<__nv_bfloat16>, dim3((unsigned)grid), dim3(kMomThreads), 0, st, 1, subs,
                          n_subs, n_tiles, mu, nesterov, reinterpret_cast<__nv_bfloat16 *>(x0),
                          reinterpret_cast<__nv_bfloat16 *>(x0t), partials)
          : launch_kernel(momentum_kernel<float>, dim3((unsigned)grid), dim3(kMomThreads), 0, st, 1, subs, n_subs,
                          n_tiles, mu, nesterov, reinterpret_cast<float *>(x0), reinterpret_cast<float *>(x0t),
                          partials);
  count_launches(1);
  return (int)err;
}

int launch_prenorm_finalize(const DevSub *subs, int32_t n_subs, const float *partials, float *alpha,
                            int32_t *status, float *stats, int sm_count, void *stream) {
  if (n_subs == 0) return 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t err =
      n_subs < sm_count
          ? launch_kernel(prenorm_finalize_kernel<1024>, dim3(n_subs), dim3(1024), 0, st, 1, subs, partials, alpha,
                          status, stats)
          : launch_kernel(prenorm_finalize_kernel<256>, dim3(n_subs), dim3(256), 0, st, 1, subs, partials, alpha,
                          status, stats);
  count_launches(1);
  return (int)err;
}

int launch_stats_finalize(const DevSub *subs, int32_t n_subs, int32_t normuon, float rms_target,
                          const float *rowss, const float *rowpart, float *stats, void *stream) {
  if (n_subs == 0) return 0;
  const cudaError_t err = launch_kernel(stats_finalize_kernel, dim3(n_subs), dim3(256), 0,
                                        reinterpret_cast<cudaStream_t>(stream), 1, subs, normuon, rms_target, rowss,
                                        rowpart, stats);
  count_launches(1);
  return (int)err;
}

int launch_normuon_rows(const DevSub *subs, int32_t n_subs, int64_t n_row_blocks, const void *x0,
                        const void *x1, int32_t x_dtype, float beta2, float eps, float lr, float *dbg,
                        int32_t *status, float rms_target, float *rowf, float *rowpart, float *mscale,
                        const float *rowss, bool streamed, bool stats, int sm_count, void *stream) {
  if (n_row_blocks == 0) return 0;
  const int64_t grid = std::min<int64_t>(n_row_blocks, (int64_t)sm_count * 8);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  static cudaError_t attr_err = [] {
    cudaError_t e = cudaFuncSetAttribute(normuon_write_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(normuon_write_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem);
    return e;
  }();
  if (streamed && attr_err != cudaSuccess) return (int)attr_err;
  cudaError_t err = cudaSuccess;
  auto rows = [&](auto mode) {
    constexpr int kMode = decltype(mode)::value;
    if (err != cudaSuccess) return;
    if (streamed && kMode != 1)
      err = launch_kernel(normuon_write_kernel<kMode>, dim3((unsigned)sm_count), dim3(kWWarps * 32), kWSmem, st, 1,
                          subs, n_subs, n_row_blocks * kRowBlock, reinterpret_cast<const __nv_bfloat16 *>(x0),
                          reinterpret_cast<const __nv_bfloat16 *>(x1), beta2, eps, lr, dbg, status, rowf,
                          (const float *)mscale);
    else if (x_dtype == GBO_BF16)
      err = launch_kernel(normuon_rows_kernel<__nv_bfloat16, kMode>, dim3((unsigned)grid), dim3(256), 0, st, 1, subs,
                          n_subs, n_row_blocks, reinterpret_cast<const __nv_bfloat16 *>(x0),
                          reinterpret_cast<const __nv_bfloat16 *>(x1), beta2, eps, lr, dbg, status, rowf,
                          (kMode == 0 && !stats) ? nullptr : rowpart, (const float *)mscale, rowss);
    else
      err = launch_kernel(normuon_rows_kernel<float, kMode>, dim3((unsigned)grid), dim3(256), 0, st, 1, subs, n_subs,
                          n_row_blocks, reinterpret_cast<const float *>(x0), reinterpret_cast<const float *>(x1),
                          beta2, eps, lr, dbg, status, rowf, (kMode == 0 && !stats) ? nullptr : rowpart,
                          (const float *)mscale, (const float *)nullptr);
    count_launches(1);
  };
  if (rms_target > 0.f) {
    rows(std::integral_constant<int, 1>());
    if (err == cudaSuccess)
      err = launch_kernel(normuon_scale_kernel, dim3((unsigned)n_subs), dim3(256), 0, st, 1, subs,
                          (const float *)rowpart, rms_target, mscale, status);
    count_launches(1);
    rows(std::integral_constant<int, 2>());
  } else if (streamed) {  // the statistics pass (row factors), then the streamed write
    rows(std::integral_constant<int, 1>());
    rows(std::integral_constant<int, 0>());
  } else {
    rows(std::integral_constant<int, 0>());
  }
  return (int)err;
}

int launch_normuon_rownorm_plain(const float *O, int64_t rows, int64_t cols, float *row_v, void *w,
                                 int32_t w_dtype, float beta2, float eps, float scale, float lr,
                                 float wd, float *dbg, void *stream) {
  if (rows == 0 || cols == 0) return 0;
  const int64_t nb = (rows + kRowBlock - 1) / kRowBlock;
  const unsigned grid = (unsigned)std::min<int64_t>(nb, 65535);
  const cudaError_t err = launch_kernel(rownorm_plain_kernel, dim3(grid), dim3(256), 0,
                                        reinterpret_cast<cudaStream_t>(stream), 1, O, rows, cols, row_v, w, w_dtype,
                                        beta2, eps, scale, lr, wd, dbg);
  count_launches(1);
  return (int)err;
}

}  // namespace gbo
