// Newton-Schulz GEMMs of the fp32 mode on the 5th-generation tensor cores
// (sm_103a).  The same jobs as the bf16 kernel (ns_gemm_tc.cu), with fp32
// operands and outputs; each product is formed from three TF32 products,
//   x y ~ hi(x) hi(y) + hi(x) lo(y) + lo(x) hi(y),
// where hi(x) keeps the 10 explicit mantissa bits TF32 carries and
// lo(x) = x - hi(x) is exact.  The omitted lo(x) lo(y) term and the TF32
// reading of lo(x) leave a relative error of about 2^-20 per product,
// against the 2^-8 of a bf16 operand.
//
// Every operand is loaded K-major (no MN-major TF32 operand is used): an X
// iterate is held both as X (p x q) and as its transpose XT (q x p), and
// the products take XT where they need X with K along its rows.
//
// Persistent, warp-specialised CTA (320 threads, one CTA per SM):
//   warp 0      TMA producer (one lane): each CTA loads its own A rows and
//               its half of B into the raw part of a stage
//   warp 1      TMEM owner and MMA issuer (one lane, the pair's even CTA)
//   warps 2..5  epilogue, one per TMEM lane quarter: TMEM -> registers ->
//               a 128-byte-swizzled staging slot -> TMA store
//   warps 6..9  split: once a stage has landed, each of its fp32 values x
//               becomes hi(x) in place and lo(x) in the stage's lo part;
//               the split warps of both CTAs then arrive on the leader's
//               split barrier, which the MMA issuer waits on
// Every wait is bounded: on time-out the kernel flags GBO_STATUS_TIMEOUT,
// waits (bounded) for its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "device_common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace gbo {

namespace {

constexpr int FK = 32;                      // 32 fp32 = one 128-byte swizzle row
constexpr int FA_BYTES = BM * FK * 4;       // 16 KB: this CTA's rows of A
constexpr int FB_HALF = (BN / 2) * FK * 4;  // 16 KB: 128 rows of B
// pair:   each CTA stages A 16 KB + half of B 16 KB, 3 stages
// single: A 16 KB + all of B 32 KB, 2 stages
template <bool kPair>
struct FMode {
  static constexpr int kRawBytes = FA_BYTES + (kPair ? FB_HALF : 2 * FB_HALF);
  static constexpr int kStages = kPair ? 3 : 2;
  static constexpr int kRows = kPair ? 2 : 1;
};
constexpr int kFRing = 3 * (FA_BYTES + FB_HALF);  // raw parts; the lo parts follow at +kFRing
static_assert(FMode<true>::kStages * FMode<true>::kRawBytes == kFRing, "ring size");
static_assert(FMode<false>::kStages * FMode<false>::kRawBytes == kFRing, "ring size");
constexpr int kFEpiWarps = 4;
constexpr int kFSplitWarps = 4;  // A/B on the 1.23B set: 140 ms per step with 2, 115 with 4, 114.5 with 6
constexpr int kFThreads = 32 * (2 + kFEpiWarps + kFSplitWarps);
// Per epilogue warp: one 8 KB slot, a 32 x 32 fp32 block and its transpose.
constexpr int kFSlotBytes = 8192;
constexpr int kFStageBytes = kFEpiWarps * kFSlotBytes;
constexpr int kFSmemBytes = 1024 /*align*/ + 2 * kFRing + kFStageBytes + 256 /*barriers*/;
static_assert(kFSmemBytes <= 232448, "shared memory per CTA");

// Instruction descriptor of kind::tf32: fp32 accumulator, TF32 A and B (format
// code 2 in both fields), both K-major, N = 256, M = 128 (one CTA) or 256 (pair).
__host__ __device__ constexpr uint32_t make_idesc_tf32(int m) {
  return (1u << 4)                      // D format: f32
         | (2u << 7)                    // A format: tf32
         | (2u << 10)                   // B format: tf32
         | ((uint32_t)(BN >> 3) << 17)  // N / 8
         | ((uint32_t)(m >> 4) << 24);  // M / 16
}

// One 128 x 256 x 8 MMA of this CTA (cta_group::1).
__device__ __forceinline__ void mma_tf32_one(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One 256 x 256 x 8 MMA over the CTA pair (issued by the even CTA).
__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Byte offset of 16-byte chunk q of row r in a 32-row x 128-byte fp32 block in
// the 128-byte swizzle layout of TMA (chunk index XOR the row's low 3 bits).
__device__ __forceinline__ uint32_t sw128(int r, int q) { return (uint32_t)(r * 128 + ((q ^ (r & 7)) << 4)); }

// Lane r holds row r of a 32 x 32 block: write it as fp32 row r.
__device__ __forceinline__ void stage_rows_f32(uint32_t dst, const float (&o)[32], int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst + sw128(lane, q)), "f"(o[4 * q]),
                 "f"(o[4 * q + 1]), "f"(o[4 * q + 2]), "f"(o[4 * q + 3])
                 : "memory");
}

// The transpose: element (lane, k) goes to row k, column lane.
__device__ __forceinline__ void stage_cols_f32(uint32_t dst, const float (&o)[32], int lane) {
  const uint32_t col = (uint32_t)((lane & 3) * 4);
#pragma unroll
  for (int k = 0; k < 32; ++k)
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst + sw128(k, lane >> 2) + col), "f"(o[k]) : "memory");
}

// Store a warp's 32 x 32 block at (x0, y0) of matrix z through `map`, and
// with `tmap` its transpose at (y0, x0) through `tmap` (the same tensor for
// a symmetric output's mirror, X's twin XT for a product); TMA drops what
// falls outside the tensor.  One slot per warp: the previous stores must
// have read it.
__device__ __forceinline__ void tma_store_block_f32(const CUtensorMap *map, const CUtensorMap *tmap, uint32_t slot,
                                                    const float (&o)[32], int x0, int y0, int z, int lane) {
  if (lane == 0) bulk_wait_read<0>();
  __syncwarp();
  stage_rows_f32(slot, o, lane);
  if (tmap) stage_cols_f32(slot + 4096, o, lane);
  fence_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_3d(map, slot, x0, y0, z);
    if (tmap) tma_store_3d(tmap, slot + 4096, y0, x0, z);
    bulk_commit();
  }
}

// Epilogue of one warp's 32 rows x 32 columns of the accumulator (lane r
// holds row i0 + r, columns col0 ..); s is the matrix's folded
// pre-normalisation factor.
__device__ __forceinline__ void epilogue_block_f32(const TcParams &P, const PhaseArgs &A, int c, int mat,
                                                   const DevSub &S, float s, int i0, int col0, float (&v)[32],
                                                   uint32_t slot, int lane) {
  const TcJob &J = P.job[c];
  const int i = i0 + lane;
  if (J.mode == kProduct) {  // X' and its twin X'T
    float o[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = s * v[k];
    tma_store_block_f32(&P.mapO[c], &P.mapO2[c], slot, o, col0, i0, mat, lane);
    return;
  }
  if (J.mode == kFinal) {  // fp32 weights (bf16 weights take final_tile_bf16)
    const int rows = kind_rows(J.kind, S.p, S.q), cols = kind_cols(J.kind, S.p, S.q);
    if (i >= rows) return;
    float u[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) u[k] = S.scale * s * v[k];
    weight_rmw32<float>(A, S, S.r0 + i, col0, u, prefix_mask(cols - col0));
    return;
  }
  // symmetric outputs, as in the bf16 kernel: a block above the diagonal is
  // stored with its mirror, a block on it whole, a block below it skipped
  if (col0 + 32 <= i0) return;
  const CUtensorMap *mirror = col0 >= i0 + 32 ? &P.mapO[c] : nullptr;
  const int p = S.p;
  const float s2 = s * s;
  float o[32];
  if (J.mode == kSquare) {
    float am[32];
    const bool full = i < p && col0 + 32 <= p;
    if (i < p)
      load_row32(reinterpret_cast<const float *>(J.aux) + S.p_off + (int64_t)i * S.ldp + col0, am, full,
                 prefix_mask(p - col0));
    else
#pragma unroll
      for (int k = 0; k < 32; ++k) am[k] = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = J.c * v[k] + J.b * am[k] + (i == col0 + k ? J.a : 0.f);
  } else if (J.mode == kGram || J.mode == kGramAP) {
    const float bs2 = J.b * s2;
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = bs2 * v[k] + (i == col0 + k ? J.a : 0.f);
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = s2 * v[k];
  }
  tma_store_block_f32(&P.mapO[c], mirror, slot, o, col0, i0, mat, lane);
  if (J.mode == kGramAP) {  // and A = s^2 C
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = s2 * v[k];
    tma_store_block_f32(&P.mapO2[c], mirror ? &P.mapO2[c] : nullptr, slot, o, col0, i0, mat, lane);
  }
}

template <bool kPair>
__global__ void __launch_bounds__(kFThreads, 1)
ns_gemm_tf32_kernel(const __grid_constant__ TcParams P, const __grid_constant__ PhaseArgs A) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up (see device_common.cuh)
  constexpr int STAGES = FMode<kPair>::kStages;
  constexpr int RAW = FMode<kPair>::kRawBytes;
  constexpr int kRows = FMode<kPair>::kRows;
  constexpr int kSplitArrivals = kFSplitWarps * (kPair ? 2 : 1);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t *stage_base = smem + 2 * kFRing;  // epilogue slots, 1024-byte aligned
  uint64_t *bars = reinterpret_cast<uint64_t *>(stage_base + kFStageBytes);
  // bars: full[STAGES], split[STAGES], empty[STAGES], accf[2], acce[2], drain
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * STAGES + 5);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
  const uint32_t full0 = smem_u32(bars), split0 = smem_u32(bars + STAGES), empty0 = smem_u32(bars + 2 * STAGES);
  const uint32_t accf0 = smem_u32(bars + 3 * STAGES), acce0 = smem_u32(bars + 3 * STAGES + 2);
  const uint32_t drain = smem_u32(bars + 3 * STAGES + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = kPair ? cluster_rank() : 0u;
  const bool leader = crank == 0;

  // Barrier protocol (pair mode: the even CTA leads):
  //   full[s]   each CTA: its own copies of stage s complete_tx on it
  //   split[s]  leader only: one arrival per split warp of both CTAs once
  //             stage s holds hi and lo parts
  //   empty[s]  each CTA: the leader's MMA commit (multicast) frees slot s
  //   accf[a]   each CTA: the leader's commit says accumulator a is complete
  //   acce[a]   leader only: one arrival per epilogue warp of both CTAs
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(split0 + 8 * s, kSplitArrivals);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf0 + 8 * a, 1);
      mbar_init(acce0 + 8 * a, (kPair ? 2 : 1) * kFEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    if constexpr (kPair) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (kPair) cluster_sync();  // both CTAs' barriers exist before any remote arrive
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int64_t total = P.tile_start[P.n];
  const int64_t cid = kPair ? (blockIdx.x >> 1) : blockIdx.x;
  const int64_t ncl = kPair ? (gridDim.x >> 1) : gridDim.x;
  const uint32_t split_lead0 = kPair ? map_to_rank(split0, 0) : split0;
  const uint32_t acce_lead0 = kPair ? map_to_rank(acce0, 0) : acce0;

  auto give_up = [&]() {
    *abort_flag = 1;
    flag_status(A.status, GBO_STATUS_TIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed_parity[STAGES];
      bool armed[STAGES];
      for (int s = 0; s < STAGES; ++s) armed[s] = false, armed_parity[s] = 0;
      for (int64_t t = cid; t < total && !*abort_flag; t += ncl) {
        const TileCoord tc = decode<kRows>(P, t);
        const int m0 = (kRows * tc.tm + (int)crank) * BM;
        const int n0 = tc.tn * BN + (kPair ? (int)crank * (BN / 2) : 0);
        const CUtensorMap *ma = &P.mapA[tc.c], *mb = &P.mapB[tc.c];
        const int kit = P.k_iters[tc.c];
        bool bad = false;
        for (int kb = 0; kb < kit; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1)) { give_up(); bad = true; break; }
          if (*abort_flag) break;
          const uint32_t fb = full0 + 8 * stage;
          mbar_expect_tx(fb, RAW);
          armed[stage] = true;
          armed_parity[stage] = phase;
          const uint32_t sa = smem_u32(smem + stage * RAW);
          const uint32_t sb = sa + FA_BYTES;
          const int k0 = kb * FK;
          tma_load_3d(sa, ma, fb, k0, m0, tc.mat);
          if constexpr (kPair) {
            tma_load_3d(sb, mb, fb, k0, n0, tc.mat);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) tma_load_3d(sb + h * FB_HALF, mb, fb, k0, n0 + h * (BN / 2), tc.mat);
          }
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
        if (bad) break;
      }
      if (*abort_flag) {
        // let every copy armed here land before shared memory goes away
        for (int s = 0; s < STAGES; ++s)
          if (armed[s]) (void)mbar_wait(full0 + 8 * s, armed_parity[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = make_idesc_tf32(kRows * BM);
      // descriptors of stage 0, K step 0 (K-major, 128-byte swizzle); a K
      // step of 8 fp32 is 32 bytes, a stage RAW bytes, the lo parts kFRing
      const uint64_t hi0 = smem_desc(smem_u32(smem), 16, 1024);
      const uint64_t lo0 = smem_desc(smem_u32(smem) + kFRing, 16, 1024);
      constexpr uint32_t kB = FA_BYTES >> 4;  // B follows A within a stage
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool issued = false;
      for (int64_t t = cid; t < total && !*abort_flag; t += ncl) {
        const TileCoord tc = decode<kRows>(P, t);
        const int kit = P.k_iters[tc.c];
        const bool freed = kPair ? mbar_wait_cluster(acce0 + 8 * acc, acc_phase ^ 1)
                                 : mbar_wait(acce0 + 8 * acc, acc_phase ^ 1);
        if (!freed) { give_up(); break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        bool bad = false;
        for (int kb = 0; kb < kit; ++kb) {
          const bool ready = kPair ? mbar_wait_cluster(split0 + 8 * stage, phase) : mbar_wait(split0 + 8 * stage, phase);
          if (!ready) { give_up(); bad = true; break; }
          tc_fence_after();
          const uint32_t soff = (uint32_t)(stage * RAW) >> 4;
#pragma unroll
          for (int k = 0; k < FK / 8; ++k) {
            const uint32_t ko = soff + 2u * k;  // 32 bytes per K step of 8
            const uint64_t ah = hi0 + ko, al = lo0 + ko, bh = hi0 + ko + kB, bl = lo0 + ko + kB;
            if constexpr (kPair) {
              mma_tf32_pair(d_tmem, ah, bh, idesc, (kb | k) != 0);
              mma_tf32_pair(d_tmem, ah, bl, idesc, 1);
              mma_tf32_pair(d_tmem, al, bh, idesc, 1);
            } else {
              mma_tf32_one(d_tmem, ah, bh, idesc, (kb | k) != 0);
              mma_tf32_one(d_tmem, ah, bl, idesc, 1);
              mma_tf32_one(d_tmem, al, bh, idesc, 1);
            }
          }
          issued = true;
          if constexpr (kPair) mma_commit_pair_mc(empty0 + 8 * stage, 0x3);  // frees the slot in both CTAs
          else mma_commit_one(empty0 + 8 * stage);
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
        if (bad) break;
        if constexpr (kPair) mma_commit_pair_mc(accf0 + 8 * acc, 0x3);
        else mma_commit_one(accf0 + 8 * acc);
        if (++acc == 2) acc = 0, acc_phase ^= 1;
      }
      if (*abort_flag && issued) {
        if constexpr (kPair) mma_commit_pair(drain);
        else mma_commit_one(drain);
        (void)mbar_wait(drain, 0);
      }
    }
  } else if (warp >= 2 + kFEpiWarps) {
    // split warps: each takes every kFSplitWarps-th run of 32 16-byte chunks of the stage's raw part
    const int sw = warp - (2 + kFEpiWarps);
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t t = cid; t < total && !*abort_flag; t += ncl) {
      const TileCoord tc = decode<kRows>(P, t);
      const int kit = P.k_iters[tc.c];
      bool bad = false;
      for (int kb = 0; kb < kit; ++kb) {
        if (!mbar_wait(full0 + 8 * stage, phase)) { give_up(); bad = true; break; }
        float4 *raw = reinterpret_cast<float4 *>(smem + stage * RAW);
        float4 *lo = reinterpret_cast<float4 *>(smem + kFRing + stage * RAW);
#pragma unroll 4
        for (int e = sw * 32 + lane; e < RAW / 16; e += 32 * kFSplitWarps) {
          const float4 x = raw[e];
          float4 h;
          h.x = __uint_as_float(__float_as_uint(x.x) & 0xffffe000u);
          h.y = __uint_as_float(__float_as_uint(x.y) & 0xffffe000u);
          h.z = __uint_as_float(__float_as_uint(x.z) & 0xffffe000u);
          h.w = __uint_as_float(__float_as_uint(x.w) & 0xffffe000u);
          raw[e] = h;
          lo[e] = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
        }
        fence_async_smem();  // the MMAs read the stage through the async proxy
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair) mbar_arrive_cluster(split_lead0 + 8 * stage);
          else mbar_arrive(split0 + 8 * stage);
        }
        if (++stage == STAGES) stage = 0, phase ^= 1;
      }
      if (bad) break;
    }
  } else {
    // epilogue warps: TMEM lane quarter = warp % 4
    const int quarter = warp & 3;
    const uint32_t slot = smem_u32(stage_base + (warp - 2) * kFSlotBytes);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t t = cid; t < total && !*abort_flag; t += ncl) {
      const TileCoord tc = decode<kRows>(P, t);
      const int sub = P.sub0[tc.c] + tc.mat;
      const DevSub &S = A.subs[sub];
      const TcJob &J = P.job[tc.c];
      const int i0 = (kRows * tc.tm + (int)crank) * BM + quarter * 32;
      const int rows = kind_rows(J.kind, S.p, S.q), cols = kind_cols(J.kind, S.p, S.q);
      if (J.mode == kFinal) prefetch_weight_tile(S, i0, tc.tn * BN, rows, cols, lane);
      if (!mbar_wait(accf0 + 8 * acc, acc_phase)) { give_up(); break; }
      tc_fence_after();
      const float s = J.first ? A.alpha[sub] : 1.0f;
      const uint32_t trow = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      if (i0 < rows) {
        // with the per-matrix norms asked for, the weight-writing last product
        // leaves each row's sum of squares of the update direction, one
        // partial per 128 columns
        const bool stats = J.mode == kFinal && J.aux != nullptr;
        float rss[BN / 128] = {};
        const int c0 = tc.tn * BN;
        if (J.mode == kFinal && S.w_dtype == GBO_BF16) {
          final_tile_bf16(A, S, s, i0, c0, rows, cols, trow, lane, BN, stats ? rss : nullptr);
        } else {
#pragma unroll 1
          for (int ch = 0; ch < BN / 32; ++ch) {
            const int col0 = c0 + ch * 32;
            if (col0 >= cols) break;
            float v[32];
            tmem_ld32(trow + ch * 32, v);
            epilogue_block_f32(P, A, tc.c, tc.mat, S, s, i0, col0, v, slot, lane);
            if (stats) {
              float r2 = 0.f;
              const float f = S.scale * s;
#pragma unroll
              for (int k = 0; k < 32; ++k) r2 = fmaf(f * v[k], f * v[k], r2);
              rss[ch / 4] += r2;
            }
          }
        }
        if (stats && i0 + lane < rows) {
          float *part_out = static_cast<float *>(const_cast<void *>(J.aux)) + S.ss_off +
                            (int64_t)(i0 + lane) * S.ss_ntn + c0 / 128;
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            if (c0 + 128 * h < cols) part_out[h] = rss[h];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair) mbar_arrive_cluster(acce_lead0 + 8 * acc);
        else mbar_arrive(acce0 + 8 * acc);
      }
      if (++acc == 2) acc = 0, acc_phase ^= 1;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (kPair) cluster_sync();  // no copy or remote arrive may target an exited CTA
  if (warp == 1) {
    if constexpr (kPair)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                   : "memory");
  }
}

// fp32 maps: K-major loads, box 32 x 128; stores, box 32 x 32, 128-byte swizzle.
bool map_f32(CUtensorMap *map, const void *base, int64_t cols, int64_t rows, int64_t count, int64_t ld,
             uint32_t box_cols, uint32_t box_rows) {
  return encode_map(map, const_cast<void *>(base), cols, rows, count, ld, box_cols, box_rows,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4);
}

const char *xbase4(const void *region, const ShapeClass &C) {
  return static_cast<const char *>(region) + C.x_base * 4;
}
const char *xtbase4(const void *region, const ShapeClass &C) {
  return static_cast<const char *>(region) + C.xt_base * 4;
}
const char *pbase4(const void *region, const ShapeClass &C) {
  return static_cast<const char *>(region) + C.p_base * 4;
}

template <bool kPair>
int launch_mode_f32(const GemmJob *const *jobs, int32_t n_jobs, const PhaseArgs &args, int sm_count, void *stream,
                    int64_t *n_launch) {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(ns_gemm_tf32_kernel<kPair>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kFSmemBytes);
  });
  if (attr_err != cudaSuccess) return (int)attr_err;
  constexpr int kRows = FMode<kPair>::kRows;
  for (int32_t j0 = 0; j0 < n_jobs; j0 += kMaxClassesPerLaunch) {
    TcParams T;
    memset(&T, 0, sizeof T);
    T.n = std::min(kMaxClassesPerLaunch, n_jobs - j0);
    T.tile_start[0] = 0;
    for (int k = 0; k < T.n; ++k) {
      const GemmJob &J = *jobs[j0 + k];
      const ShapeClass &C = *J.cls;
      bool ok;
      int Mdim, Ndim, Kdim;
      if (J.kind == kKindGram) {  // A = X rows, B = X rows, K = q
        const char *x = xbase4(J.opA, C);
        ok = map_f32(&T.mapA[k], x, C.q, C.p, C.count, C.ld, FK, BM) &&
             map_f32(&T.mapB[k], x, C.q, C.p, C.count, C.ld, FK, BN / 2);
        Mdim = C.p, Ndim = C.p, Kdim = C.q;
      } else if (J.kind == kKindSym) {  // A = L rows, B = R rows (R symmetric), K = p
        ok = map_f32(&T.mapA[k], pbase4(J.opA, C), C.p, C.p, C.count, C.ldp, FK, BM) &&
             map_f32(&T.mapB[k], pbase4(J.opB, C), C.p, C.p, C.count, C.ldp, FK, BN / 2);
        Mdim = C.p, Ndim = C.p, Kdim = C.p;
      } else if (J.kind == kKindProdK) {  // A = L rows (K = p), B = rows of XT (q x p)
        ok = map_f32(&T.mapA[k], pbase4(J.opA, C), C.p, C.p, C.count, C.ldp, FK, BM) &&
             map_f32(&T.mapB[k], xtbase4(J.opB, C), C.p, C.q, C.count, C.ldt, FK, BN / 2);
        Mdim = C.p, Ndim = C.q, Kdim = C.p;
      } else if (J.kind == kKindProdT) {  // A = rows of XT (q x p, K = p), B = L rows
        ok = map_f32(&T.mapA[k], xtbase4(J.opA, C), C.p, C.q, C.count, C.ldt, FK, BM) &&
             map_f32(&T.mapB[k], pbase4(J.opB, C), C.p, C.p, C.count, C.ldp, FK, BN / 2);
        Mdim = C.q, Ndim = C.p, Kdim = C.p;
      } else {
        return (int)cudaErrorInvalidValue;  // MN-major kinds are not used with fp32 operands
      }
      if (J.mode == kProduct) {  // X' (p x q) and its twin X'T (q x p)
        ok = ok && map_f32(&T.mapO[k], xbase4(J.out, C), C.q, C.p, C.count, C.ld, 32, 32) &&
             map_f32(&T.mapO2[k], xtbase4(J.out2, C), C.p, C.q, C.count, C.ldt, 32, 32);
      } else if (J.mode != kFinal) {
        ok = ok && map_f32(&T.mapO[k], pbase4(J.out, C), C.p, C.p, C.count, C.ldp, 32, 32);
        if (J.mode == kGramAP) ok = ok && map_f32(&T.mapO2[k], pbase4(J.out2, C), C.p, C.p, C.count, C.ldp, 32, 32);
      }
      if (!ok) return (int)cudaErrorInvalidValue;
      TcJob &tj = T.job[k];
      tj.mode = J.mode;
      tj.kind = J.kind;
      tj.first = J.first;
      tj.a = J.a;
      tj.b = J.b;
      tj.c = J.c;
      tj.out = J.out;
      tj.out2 = J.out2;
      tj.aux = J.aux;
      T.tiles_n[k] = (Ndim + BN - 1) / BN;
      T.k_iters[k] = (Kdim + FK - 1) / FK;
      T.sub0[k] = C.sub0;
      const int items_m = ((Mdim + BM - 1) / BM + kRows - 1) / kRows;
      if (J.kind == kKindGram || J.kind == kKindSym) {
        int cnt = 0;
        for (int r = 0; r < items_m; ++r) cnt += std::max(0, T.tiles_n[k] - tri_tn_min(kRows * r));
        T.tiles_per_mat[k] = cnt;
      } else {
        T.tiles_per_mat[k] = items_m * T.tiles_n[k];
      }
      T.tile_start[k + 1] = T.tile_start[k] + (int64_t)C.count * T.tiles_per_mat[k];
    }
    const int64_t total = T.tile_start[T.n];
    if (total == 0) continue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = kFSmemBytes;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    if constexpr (kPair) {
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      static std::once_flag occ_once;
      static int max_clusters = 0;
      std::call_once(occ_once, [&] {
        cfg.gridDim = dim3(2 * std::max(1, sm_count / 2));
        if (cudaOccupancyMaxActiveClusters(&max_clusters, ns_gemm_tf32_kernel<true>, &cfg) != cudaSuccess)
          max_clusters = 0;
      });
      const int clusters =
          (int)std::min<int64_t>(total, std::max(1, max_clusters > 0 ? std::min(max_clusters, sm_count / 2)
                                                                        : sm_count / 2));
      cfg.gridDim = dim3(2 * clusters);
    } else {
      cfg.gridDim = dim3((unsigned)std::min<int64_t>(total, sm_count));
    }
    // programmatic stream serialization when enabled (this kernel waits for
    // the previous one after its prologue), and the pair's cluster
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (kPair) attrs[na++] = attr[0];
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = pdl_enabled(stream);
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    const cudaError_t lerr = cudaLaunchKernelEx(&cfg, ns_gemm_tf32_kernel<kPair>, T, args);
    if (lerr != cudaSuccess) return (int)lerr;
    count_launches(1);
    if (n_launch) ++*n_launch;
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return (int)err;
  }
  return 0;
}

}  // namespace

int launch_ns_gemm_tf32(const GemmJob *jobs, int32_t n_jobs, const PhaseArgs &globals, int sm_count, void *stream,
                        int64_t *n_launch) {
  std::vector<const GemmJob *> single, pair;
  for (int32_t j = 0; j < n_jobs; ++j) {
    if (jobs[j].cls->count == 0) continue;
    (single_job(jobs[j].cls->p, jobs[j].mode) ? single : pair).push_back(&jobs[j]);
  }
  int err = launch_mode_f32<true>(pair.data(), (int32_t)pair.size(), globals, sm_count, stream, n_launch);
  if (err) return err;
  return launch_mode_f32<false>(single.data(), (int32_t)single.size(), globals, sm_count, stream, n_launch);
}

}  // namespace gbo
