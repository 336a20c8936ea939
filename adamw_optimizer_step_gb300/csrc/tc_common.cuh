// Pieces shared by the tensor-core Newton-Schulz kernels (bf16 operands, and
// fp32 operands as three TF32 products): tile geometry, the per-launch job
// table, PTX wrappers for mbarriers, TMA loads and bulk stores, tcgen05
// commits and TMEM loads, tile decoding, the weight write of the last
// product, and tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"

namespace gbo {

namespace {

constexpr int BM = 128;  // accumulator rows per CTA
constexpr int BN = 256;  // tile columns (a pair tile is 256 x BN, split by rows)
constexpr int kTmemCols = 512;                   // two 128 x 256 fp32 accumulators
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s per wait


// What one class of a launch computes, as the kernel sees it.
struct TcJob {
  int32_t mode;   // GemmMode
  int32_t kind;   // GemmKind: the products have full outputs, the others a
                  // symmetric p x p output (upper-triangle tiles only)
  int32_t first;  // s = alpha of the matrix (pre-normalisation folded in), else 1
  float a, b, c;
  void *out, *out2;
  const void *aux;
};

struct TcParams {
  CUtensorMap mapA[kMaxClassesPerLaunch];  // A operand: one 128-byte row of K x 128 rows, or MN-major boxes
  CUtensorMap mapB[kMaxClassesPerLaunch];  // B operand, likewise
  CUtensorMap mapO[kMaxClassesPerLaunch];  // output (TMA store), box 32 x 32
  CUtensorMap mapO2[kMaxClassesPerLaunch]; // second output: A of kGramAP, or X'T of an fp32 product
  CUtensorMap mapBh[kMaxClassesPerLaunch]; // bf16 pair kernel: K-major B in 64-row boxes, for half tiles
  int64_t tile_start[kMaxClassesPerLaunch + 1];
  int32_t tiles_n[kMaxClassesPerLaunch];
  int32_t k_iters[kMaxClassesPerLaunch];
  int32_t sub0[kMaxClassesPerLaunch];
  int32_t tiles_per_mat[kMaxClassesPerLaunch];
  TcJob job[kMaxClassesPerLaunch];
  int32_t n;
  // tail split (bf16 pair kernel only): work items split_base .. of the
  // launch's tile_start[n] items run as two halves of 128 columns each, so
  // the launch has n_items = tile_start[n] + (tile_start[n] - split_base)
  // work items; without a split, split_base = n_items = tile_start[n]
  int64_t split_base;
  int64_t n_items;
};

// ---------------------------------------------------------------------------
// PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of a phase (mbarrier.try_wait may suspend the thread for
// a while when the phase is incomplete; a loop that polls several barriers
// in turn wants an answer at once).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete: gives up
// (returns false) after `limit_ns` of the global timer.
__device__ __forceinline__ bool mbar_wait_ns(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t spin = 0;; ++spin) {
    if (mbar_try(bar, parity)) return true;
    if ((spin & 255u) == 255u && global_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) { return mbar_wait_ns(bar, parity, kWaitNs); }

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Copy into this CTA's shared memory and signal the mbarrier at the
// shared::cluster address `bar`, which may be in either CTA of the pair.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y,
                                                 int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Bulk tensor store of one box from this CTA's shared memory; completion is
// tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed their writes.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make this thread's shared-memory writes visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// shared::cluster address of the same shared::cta offset in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on a local barrier that CTAs of the cluster arrive on.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  if (mbar_try_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t spin = 0;; ++spin) {
    if (mbar_try_cluster(bar, parity)) return true;
    if ((spin & 255u) == 255u && global_ns() - t0 > kWaitNs) return false;
  }
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of both CTAs of the pair.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05), 128-byte swizzle.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-47  descriptor version (1)
//   bits 61-63  layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

__device__ __forceinline__ void mma_commit_one(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Arrive on the mbarrier at offset `bar` in every CTA of `mask` once the
// pair MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
}

struct TileCoord {
  int c, mat, tm, tn;  // tm: work-item row (a pair of tile rows in pair mode)
};

// First computed column tile of tile row tm in a symmetric launch: the
// tile holds an element on or above the diagonal iff BN*tn + BN - 1 >= BM*tm.
__host__ __device__ __forceinline__ int tri_tn_min(int tm) { return (tm * BM) / BN; }

// Work items: kRows consecutive 128-row tiles of one column tile tn (the two
// CTAs of a pair take rows kRows * r and kRows * r + 1).  In a symmetric
// launch only items touching the upper triangle exist.
template <int kRows>
__device__ __forceinline__ TileCoord decode(const TcParams &P, int64_t t) {
  TileCoord tc;
  int c = 0;
  while (c + 1 < P.n && P.tile_start[c + 1] <= t) ++c;
  const int64_t local = t - P.tile_start[c];
  tc.c = c;
  tc.mat = (int)(local / P.tiles_per_mat[c]);
  int rem = (int)(local % P.tiles_per_mat[c]);
  const int tn_all = P.tiles_n[c];
  if (is_product_kind(P.job[c].kind)) {
    tc.tm = rem / tn_all;
    tc.tn = rem % tn_all;
  } else {
    int r = 0;
    for (;; ++r) {
      const int cnt = max(0, tn_all - tri_tn_min(kRows * r));
      if (rem < cnt) break;
      rem -= cnt;
    }
    tc.tm = r;
    tc.tn = tri_tn_min(kRows * r) + rem;
  }
  return tc;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// 32 consecutive values of one row: vector store when the row segment is
// whole and aligned, else element by element under the mask.
template <typename T>
__device__ __forceinline__ void store_row32(T *dst, const float (&o)[32], bool vec, uint32_t mask) {
  if constexpr (sizeof(T) == 2) {
    if (vec) {
      uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        d[q] = make_uint4(pack_bf16(o[8 * q], o[8 * q + 1]), pack_bf16(o[8 * q + 2], o[8 * q + 3]),
                          pack_bf16(o[8 * q + 4], o[8 * q + 5]), pack_bf16(o[8 * q + 6], o[8 * q + 7]));
      return;
    }
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (mask >> k & 1u) dst[k] = __float2bfloat16_rn(o[k]);
  } else {
    if (vec) {
      float4 *d = reinterpret_cast<float4 *>(dst);
#pragma unroll
      for (int q = 0; q < 8; ++q) d[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      return;
    }
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (mask >> k & 1u) dst[k] = o[k];
  }
}

template <typename T>
__device__ __forceinline__ void load_row32(const T *src, float (&o)[32], bool vec, uint32_t mask) {
  if constexpr (sizeof(T) == 2) {
    if (vec) {
      const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = s4[q];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[h]);
          o[8 * q + 2 * h] = __low2float(b);
          o[8 * q + 2 * h + 1] = __high2float(b);
        }
      }
      return;
    }
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = (mask >> k & 1u) ? __bfloat162float(src[k]) : 0.f;
  } else {
    if (vec) {
      const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 f = s4[q];
        o[4 * q] = f.x; o[4 * q + 1] = f.y; o[4 * q + 2] = f.z; o[4 * q + 3] = f.w;
      }
      return;
    }
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = (mask >> k & 1u) ? src[k] : 0.f;
  }
}

__device__ __forceinline__ uint32_t prefix_mask(int n) {  // the low n bits, n in [0, 32]
  return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
}

// bf16 staging of the bf16 kernel's epilogue: per warp two slots of
// kSlotBytes, each a 32 x 32 bf16 block and its transpose.
constexpr int kSlotBytes = 4096;

// Byte offset of 16-byte chunk q of row r in a 32-row x 64-byte bf16 block in
// the 64-byte swizzle layout of TMA (chunk index XOR bits 7-8 of the offset).
__device__ __forceinline__ uint32_t sw64(int r, int q) { return (uint32_t)(r * 64 + ((q ^ ((r >> 1) & 3)) << 4)); }

// Lane r holds row r of a 32 x 32 block: write it as bf16 row r.
__device__ __forceinline__ void stage_rows(uint32_t dst, const float (&o)[32], int lane) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + sw64(lane, q)),
                 "r"(pack_bf16(o[8 * q], o[8 * q + 1])), "r"(pack_bf16(o[8 * q + 2], o[8 * q + 3])),
                 "r"(pack_bf16(o[8 * q + 4], o[8 * q + 5])), "r"(pack_bf16(o[8 * q + 6], o[8 * q + 7]))
                 : "memory");
}

// The transpose: element (lane, k) goes to row k, column lane.  For each k
// the warp writes one 64-byte row, two lanes per 32-bit word.
__device__ __forceinline__ void stage_cols(uint32_t dst, const float (&o)[32], int lane) {
  const uint32_t col = (uint32_t)((lane & 7) * 2);
#pragma unroll
  for (int k = 0; k < 32; ++k)
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(dst + sw64(k, lane >> 3) + col),
                 "h"(__bfloat16_as_ushort(__float2bfloat16_rn(o[k])))
                 : "memory");
}

// Store a warp's 32 x 32 block at (x0, y0) of matrix z, and with `mirror`
// its transpose at (y0, x0), through the next of the warp's kSlots staging
// slots (two, or one); TMA drops whatever falls outside the tensor.
template <int kSlots = 2>
__device__ __forceinline__ void tma_store_block(const CUtensorMap *map, uint32_t stage, int &slot,
                                                const float (&o)[32], bool mirror, int x0, int y0, int z, int lane) {
  const uint32_t dst = stage + (uint32_t)(slot * kSlotBytes);
  if constexpr (kSlots == 2) slot ^= 1;
  if (lane == 0) bulk_wait_read<kSlots - 1>();  // the stores that last used this slot have read it
  __syncwarp();
  stage_rows(dst, o, lane);
  if (mirror) stage_cols(dst + 2048, o, lane);
  fence_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_3d(map, dst, x0, y0, z);
    if (mirror) tma_store_3d(map, dst + 2048, y0, x0, z);
    bulk_commit();
  }
}

// Weight write of 32 consecutive elements of one stored row: W[row][c0..c0+31]
// with the update directions u[0..31] (valid under `mask`).
template <typename WT>
__device__ __forceinline__ void weight_rmw32(const PhaseArgs &A, const DevSub &S, int64_t row, int c0,
                                             const float (&u)[32], uint32_t mask) {
  const int64_t widx = row * S.cols + c0;
  WT *w = reinterpret_cast<WT *>(S.w) + widx;
  const bool vec = S.w_vec && mask == 0xffffffffu;
  float wv[32];
  load_row32(w, wv, vec, mask);
  const float lr = A.lr * S.lr_mult;
#pragma unroll
  for (int k = 0; k < 32; ++k) wv[k] = wv[k] - lr * (S.wd * wv[k] + u[k]);
  store_row32(w, wv, vec, mask);
  if (A.dbg) {
    float *d = A.dbg + S.dbg_off + widx;
    const bool dvec = mask == 0xffffffffu && (reinterpret_cast<uintptr_t>(d) & 15) == 0;
    store_row32(d, u, dvec, mask);
  }
}

// 32 consecutive bf16 weights of one row, as raw bits.
struct WSeg {
  uint4 q[4];
};

__device__ __forceinline__ void wseg_load(WSeg &r, const __nv_bfloat16 *w, bool vec, uint32_t mask) {
  if (vec) {
    const uint4 *p = reinterpret_cast<const uint4 *>(w);
#pragma unroll
    for (int q = 0; q < 4; ++q) r.q[q] = p[q];
    return;
  }
  uint32_t h[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t lo = (mask >> (2 * k) & 1u) ? __bfloat16_as_ushort(w[2 * k]) : 0u;
    const uint32_t hi = (mask >> (2 * k + 1) & 1u) ? __bfloat16_as_ushort(w[2 * k + 1]) : 0u;
    h[k] = lo | (hi << 16);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) r.q[q] = make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
}

__device__ __forceinline__ void wseg_unpack(const WSeg &r, float (&o)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w[4] = {r.q[q].x, r.q[q].y, r.q[q].z, r.q[q].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[h]);
      o[8 * q + 2 * h] = __low2float(b);
      o[8 * q + 2 * h + 1] = __high2float(b);
    }
  }
}

// The last product's epilogue of one warp for one tile when W is bf16 and
// no TMA map covers the block (rows past the end of the matrix, or weight
// rows that do not start on 16-byte boundaries).  The output is in stored
// orientation (rows x cols of the matrix); lane r owns stored row
// r0 + i0 + r.  The weights of chunk ch + 1 are loaded before chunk ch is
// computed, so a load of each lane's row segment is always in flight.
// rss (nullable): per 128 columns of the span, this lane's sum of squares of
// the update direction, added to.
__device__ __forceinline__ void final_tile_bf16(const PhaseArgs &A, const DevSub &S, float s, int i0, int tile_col0,
                                                int rows, int cols, uint32_t trow, int lane, int span = BN,
                                                float *rss = nullptr) {
  const int nch = min(span / 32, (cols - tile_col0 + 31) / 32);  // chunks holding columns < cols
  const float lr = A.lr * S.lr_mult, su = S.scale * s;
  __nv_bfloat16 *W = reinterpret_cast<__nv_bfloat16 *>(S.w);
  const bool ok = i0 + lane < rows;
  const int64_t wrow = (S.r0 + i0 + lane) * S.cols;
  WSeg nxt;
  if (ok) {
    const uint32_t m0 = prefix_mask(cols - tile_col0);
    wseg_load(nxt, W + wrow + tile_col0, S.w_vec && m0 == 0xffffffffu, m0);
  }
#pragma unroll 1
  for (int ch = 0; ch < nch; ++ch) {
    const WSeg cur = nxt;
    const int col0 = tile_col0 + ch * 32;
    const uint32_t mask = prefix_mask(cols - col0);
    if (ok && ch + 1 < nch) {
      const uint32_t mn = prefix_mask(cols - col0 - 32);
      wseg_load(nxt, W + wrow + col0 + 32, S.w_vec && mn == 0xffffffffu, mn);
    }
    float u[32];
    tmem_ld32(trow + ch * 32, u);
    if (ok) {
      float w[32];
      wseg_unpack(cur, w);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        u[k] *= su;
        w[k] = w[k] - lr * (S.wd * w[k] + u[k]);
      }
      if (rss) {
        float a = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) a = fmaf(u[k], u[k], a);  // columns past the matrix hold zeros
        rss[ch >> 2] += a;
      }
      store_row32(W + wrow + col0, w, S.w_vec && mask == 0xffffffffu, mask);
      if (A.dbg) {
        float *d = A.dbg + S.dbg_off + wrow + col0;
        store_row32(d, u, mask == 0xffffffffu && (reinterpret_cast<uintptr_t>(d) & 15) == 0, mask);
      }
    }
  }
}

// The same epilogue for a block of 32 whole rows of a bf16 weight with a TMA
// map (`wmap`: the whole weight, 32 x 32 boxes, 64-byte swizzle): the weights
// travel by TMA both ways.  Column chunk c (a 32 x 32 block) is loaded into
// buffer c % kWBufs of the warp's staging area, updated in place and stored
// from there.  Loads run kWBufs - 1 chunks ahead of the chunk being updated;
// the first ones are issued before the accumulator is ready
// (weight_loads_begin).  Each buffer has an mbarrier (wbar0 + 8 b); wpar
// holds the parity each waits for next (bit b) and winfl the buffers with a
// load in flight (bit b).  The warp's state is uniform across its lanes.
constexpr int kWBufBytes = 2048;

template <int kWBufs>
__device__ __forceinline__ void weight_load_chunk(const CUtensorMap *wmap, uint32_t stage, uint32_t wbar0, int c,
                                                  int col0, int row0) {
  const uint32_t b = (uint32_t)(c & (kWBufs - 1));
  mbar_expect_tx(wbar0 + 8 * b, kWBufBytes);
  tma_load_3d(stage + b * kWBufBytes, wmap, wbar0 + 8 * b, col0, row0, 0);
}

__device__ __forceinline__ int weight_chunks(int tile_col0, int cols, int span) {
  return min(span / 32, (cols - tile_col0 + 31) / 32);
}

// kWBufs buffers: kWBufs - 1 chunks are loaded here, ahead of the first
// update (final_tile_bf16_tma).
template <int kWBufs>
__device__ __forceinline__ void weight_loads_begin(const CUtensorMap *wmap, uint32_t stage, uint32_t wbar0,
                                                   int tile_col0, int cols, int row0, int lane, uint32_t &winfl,
                                                   int span) {
  const int n0 = min(kWBufs - 1, weight_chunks(tile_col0, cols, span));
  if (lane == 0) {
    bulk_wait_read<0>();  // earlier stores from the staging area have read it
    for (int c = 0; c < n0; ++c) weight_load_chunk<kWBufs>(wmap, stage, wbar0, c, tile_col0 + 32 * c, row0);
  }
  __syncwarp();
  winfl |= (1u << n0) - 1u;
}

// Lane r reads bf16 row r of a 32 x 32 block in the 64-byte swizzle layout.
__device__ __forceinline__ void stage_read_row(uint32_t src, float (&o)[32], int lane) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(src + sw64(lane, q))
                 : "memory");
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[h]);
      o[8 * q + 2 * h] = __low2float(b);
      o[8 * q + 2 * h + 1] = __high2float(b);
    }
  }
}

// kWBufs buffers, loads kWBufs - 1 chunks ahead of the update.  `span`: the
// columns of the tile this warp covers, from tile_col0.  Returns false on a
// time-out of a load wait.
template <int kWBufs>
__device__ __forceinline__ bool final_tile_bf16_tma(const PhaseArgs &A, const DevSub &S, float s, int i0,
                                                    int tile_col0, int cols, uint32_t trow, int lane,
                                                    const CUtensorMap *wmap, uint32_t stage, uint32_t wbar0,
                                                    uint32_t &wpar, uint32_t &winfl, int span, float *rss = nullptr) {
  constexpr int kWAhead = kWBufs - 1;
  const int nch = weight_chunks(tile_col0, cols, span);
  const float lr = A.lr * S.lr_mult, su = S.scale * s;
  // W - lr (wd W + su C) as one multiply-add per element: decay factor and
  // update factor folded (the same result up to one fp32 rounding)
  const float keep = 1.0f - lr * S.wd, step = lr * su;
  const bool decay = S.wd != 0.f;
  const int row0 = (int)(S.r0 + i0);
  const int64_t wrow = (S.r0 + i0 + lane) * S.cols;
#pragma unroll 1
  for (int ch = 0; ch < nch; ++ch) {
    const uint32_t b = (uint32_t)(ch & (kWBufs - 1));
    const uint32_t buf = stage + b * kWBufBytes;
    const int col0 = tile_col0 + ch * 32;
    float u[32];
    tmem_ld32(trow + ch * 32, u);
    if (rss) {  // the update direction is su * u; columns past the matrix hold zeros
      float a = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) a = fmaf(u[k], u[k], a);
      rss[ch >> 2] += su * su * a;
    }
    if (!mbar_wait(wbar0 + 8 * b, (wpar >> b) & 1u)) return false;
    wpar ^= 1u << b;
    winfl &= ~(1u << b);
    float w[32];
    stage_read_row(buf, w, lane);
    if (decay) {
#pragma unroll
      for (int k = 0; k < 32; ++k) w[k] = fmaf(-step, u[k], keep * w[k]);
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) w[k] = fmaf(-step, u[k], w[k]);
    }
    stage_rows(buf, w, lane);
    fence_async_smem();
    __syncwarp();
    const bool more = ch + kWAhead < nch;
    if (lane == 0) {
      tma_store_3d(wmap, buf, col0, row0, 0);
      bulk_commit();
      if (more) {
        // the buffer of chunk ch + kWAhead was last stored from by chunk
        // ch - 1: at most this chunk's store may still read the staging area
        bulk_wait_read<1>();
        weight_load_chunk<kWBufs>(wmap, stage, wbar0, ch + kWAhead, col0 + 32 * kWAhead, row0);
      }
    }
    if (more) winfl |= 1u << ((ch + kWAhead) & (kWBufs - 1));
    if (A.dbg) {
#pragma unroll
      for (int k = 0; k < 32; ++k) u[k] *= su;
      const uint32_t mask = prefix_mask(cols - col0);
      float *d = A.dbg + S.dbg_off + wrow + col0;
      store_row32(d, u, mask == 0xffffffffu && (reinterpret_cast<uintptr_t>(d) & 15) == 0, mask);
    }
  }
  if (lane == 0) bulk_wait_read<0>();  // the staging area is free for the other epilogues
  __syncwarp();
  return true;
}

__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Bring into L2 the weight elements the last product's epilogue of this
// warp will read-modify-write for the tile at (i0.., col0 .. col0 + BN) of
// the stored-orientation output (rows x cols).
__device__ __forceinline__ void prefetch_weight_tile(const DevSub &S, int i0, int col0, int rows, int cols,
                                                     int lane, int span = BN) {
  const int64_t es = S.w_dtype == GBO_BF16 ? 2 : 4;
  const char *w = static_cast<const char *>(S.w);
  const int i = i0 + lane;
  if (i >= rows) return;
  const int c1 = min(cols, col0 + span);
  for (int c = col0; c < c1; c += (int)(128 / es)) prefetch_l2(w + ((S.r0 + i) * S.cols + c) * es);
}

// ---------------------------------------------------------------------------
// host: tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D map over `count` row-major rows x cols matrices with row stride `ld`
// elements of `esize` bytes (bf16 unless given), stored back to back; box =
// box_cols x box_rows x 1.  Loads use the 128-byte swizzle the MMA
// descriptors expect; the bf16 kernel's stores (32 x 32 boxes) use the
// 64-byte swizzle of its staging slots.
bool encode_map(CUtensorMap *map, void *base, int64_t cols, int64_t rows, int64_t count, int64_t ld,
                uint32_t box_cols, uint32_t box_rows,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
                CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, int esize = 2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)count};
  const cuuint64_t strides[2] = {(cuuint64_t)(ld * esize), (cuuint64_t)(ld * rows * esize)};
  const cuuint32_t box[3] = {box_cols, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dtype, 3, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace

}  // namespace gbo
