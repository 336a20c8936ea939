// Newton-Schulz GEMMs on the 5th-generation tensor cores (sm_103a):
// TMA -> shared memory (128-byte swizzle) -> tcgen05.mma (bf16 operands, fp32
// accumulators in TMEM) -> tcgen05.ld -> fused epilogue.
//
// One iteration of eq. (5) of the NorMuon paper (zskr.cn, section 2.2),
//   X <- (a I + b A + c A^2) X,  A = X X^T,
// is two (three when c != 0) launches of this kernel over every matrix of
// the step: the Gram product, the optional square, and the product back
// onto X whose last instance writes the weights.  Matrices of one oriented
// shape are stored back to back, so one 3-D tensor map (columns, rows,
// matrix) covers a whole shape class; out-of-range rows and columns of a
// tile are zero-filled by TMA loads and dropped by TMA stores.  Each shape class
// of a launch is a job with its own operands, output and epilogue, so one
// launch may run X-route and Gram-route steps (see internal.h) side by side.
//
// Persistent, warp-specialised CTA (one CTA per SM; 192 threads, 320 in
// single mode):
//   warp 0      TMA producer (one lane), STAGES-deep ring of A/B tiles
//   warp 1      TMEM owner and MMA issuer (one lane)
//   warps 2..   epilogue, one per TMEM lane quarter (two, each over half of
//               the tile's columns, in single mode): TMEM -> registers ->
//               a 64-byte-swizzled staging slot -> TMA store; in the last
//               product, full 32-row blocks of bf16 weights are loaded by
//               TMA into the staging area three 32 x 32 blocks ahead,
//               updated in place and stored by TMA, through a map of the
//               weight
// The accumulator is double-buffered in TMEM (2 x 256 columns) so the
// epilogue of one tile overlaps the MMAs of the next.  Work items are dealt
// round-robin over the resident CTA pairs; when a launch's last wave would
// occupy at most half of them, its tiles run as 256 x 128 halves instead
// (tail split, item_of below).  Every wait is
// bounded: on time-out the kernel flags GBO_STATUS_TIMEOUT, waits (bounded)
// for its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "device_common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace gbo {

namespace {

constexpr int BK = 64;   // 64 bf16 = one 128-byte swizzle row

std::atomic<int32_t> g_tail_split{1};  // see gbo_testing_set_tail_split
constexpr int A_BYTES = BM * BK * 2;             // 16 KB: this CTA's rows of A
constexpr int B_HALF = (BN / 2) * BK * 2;        // 16 KB: 128 rows of B
// Two modes share the kernel source:
//   pair   (kPair = true)  2-CTA cluster, tcgen05 cta_group::2, 256 x 256 tile;
//                          a stage holds two 64-wide K blocks, each A 16 KB +
//                          half of B 16 KB per CTA (3 stages of 64 KB: one
//                          barrier handshake per 8 MMAs; about 1% faster on
//                          the 1.23B set than 6 stages of one block, over
//                          eight interleaved runs)
//   single (kPair = false) one CTA, cta_group::1, 128 x 256 tile; a stage
//                          holds one K block, A 16 KB + all of B 32 KB (4
//                          stages); used for matrices of at most 128 rows,
//                          where a pair would spend its second CTA on padding
template <bool kPair>
struct Mode {
  static constexpr int kSub = kPair ? 2 : 1;  // BK-wide K blocks per stage
  static constexpr int kSubBytes = A_BYTES + (kPair ? B_HALF : 2 * B_HALF);
  static constexpr int kStageBytes = kSub * kSubBytes;
  // pairs: 3 x 64 KB; single CTAs: 3 x 48 KB, leaving room for deeper
  // weight loads in the epilogue staging
  static constexpr int kStages = 3;
  static constexpr int kRows = kPair ? 2 : 1;  // 128-row tiles per work item
  static constexpr int kRingBytes = kStages * kStageBytes;
};
// Epilogue warps.  Pair mode: one per TMEM lane quarter, each over the
// tile's 256 columns, with two store slots (kSlotBytes each, tc_common.cuh)
// or four weight buffers (8 KB a warp, 32 KB in all).  Single mode: two per
// lane quarter, each over 128 of the columns, with two slots or four weight
// buffers (8 KB a warp, 64 KB in all): its HBM-bound last products on small
// matrices are limited by latency, and two warps per scheduler, each with
// three weight blocks in flight, hide more of it.
template <bool kPair>
struct Epi {
  static constexpr int kWarps = kPair ? 4 : 8;
  static constexpr int kSplit = kWarps / 4;           // warps per lane quarter
  static constexpr int kSpan = BN / kSplit;           // columns a warp covers
  static constexpr int kThreads = 64 + 32 * kWarps;
  static constexpr int kWarpStage = 8 * 1024;
  static constexpr int kSlots = kWarpStage / kSlotBytes;
  static constexpr int kWBufs = kWarpStage / kWBufBytes;
  static constexpr int kStagingBytes = kWarps * kWarpStage;
  static_assert((kWBufs & (kWBufs - 1)) == 0, "weight buffers are indexed modulo a power of two");
};
// ring, then staging, then barriers; one size for both modes (the larger)
template <bool kPair>
__host__ __device__ constexpr int smem_used() { return Mode<kPair>::kRingBytes + Epi<kPair>::kStagingBytes; }
constexpr int kSmemBytes =
    1024 /*align*/ + (smem_used<true>() > smem_used<false>() ? smem_used<true>() : smem_used<false>()) +
    512 /*barriers*/;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B,
// each K-major or MN-major, N = 256, M = 128 (one CTA) or 256 (pair).
__host__ __device__ constexpr uint32_t make_idesc(int a_mn_major, int b_mn_major, int m, int n = BN) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | ((uint32_t)a_mn_major << 15) // A major-ness
         | ((uint32_t)b_mn_major << 16) // B major-ness
         | ((uint32_t)(n >> 3) << 17)   // N / 8
         | ((uint32_t)(m >> 4) << 24);  // M / 16
}

// Work item t of a launch: its tile, and which 128-column half of it when
// the item lies in the launch's split tail (half = -1: the whole tile).
// The tail split runs a launch's last partial wave of pair tiles as twice as
// many half tiles (N = 128), so it ends after half a tile's time instead of
// a whole one; each output element still sums the same products in the same
// order.
template <int kRows>
__device__ __forceinline__ TileCoord item_of(const TcParams &P, int64_t t, int &half) {
  if (t < P.split_base) {
    half = -1;
    return decode<kRows>(P, t);
  }
  const int64_t u = t - P.split_base;
  half = (int)(u & 1);
  return decode<kRows>(P, P.split_base + (u >> 1));
}

// One 128 x 256 x 16 MMA of this CTA (cta_group::1).
__device__ __forceinline__ void mma_bf16_one(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One 256 x 256 x 16 MMA over the CTA pair (issued by the even CTA): A
// rows 0-127 and B rows 0-127 come from this CTA's shared memory, the rest
// from the peer's at the same offsets; each CTA's TMEM receives its 128 rows.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Epilogue of one warp's 32 rows x 32 columns of the accumulator.  Lane r
// holds row i0 + r in v[0..31] (columns col0 .. col0 + 31); s is the
// matrix's folded pre-normalisation factor (1 unless the job folds it).
// Outputs other than the weights leave through TMA stores from the warp's
// staging slots (`stage`, `slot`).
template <int kSlots>
__device__ __forceinline__ void epilogue_block(const TcParams &P, const PhaseArgs &A, int c, int mat,
                                               const DevSub &S, float s, int i0, int col0, float (&v)[32],
                                               uint32_t stage, int &slot, int lane) {
  const TcJob &J = P.job[c];
  const int i = i0 + lane;
  if (J.mode == kProduct) {
    float o[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = s * v[k];
    tma_store_block<kSlots>(&P.mapO[c], stage, slot, o, false, col0, i0, mat, lane);
    return;
  }
  if (J.mode == kFinal) {  // fp32 weights: O = s * C, the update direction is scale * O
    const int rows = kind_rows(J.kind, S.p, S.q), cols = kind_cols(J.kind, S.p, S.q);
    if (i >= rows) return;
    float u[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) u[k] = S.scale * s * v[k];
    weight_rmw32<float>(A, S, S.r0 + i, col0, u, prefix_mask(cols - col0));
    return;
  }
  // Symmetric outputs: P = a I + b s^2 C, A = s^2 C, both (kGramAP), or
  // P = a I + b A + c C (kSquare).  Blocks are 32-aligned, so each lies on,
  // above or below the diagonal.  A block above it is stored with its
  // mirror; a block on it is stored whole; a block below it is the mirror
  // of a block above and is skipped.  Every element is written once.
  if (col0 + 32 <= i0) return;
  const bool mirror = col0 >= i0 + 32;
  const int p = S.p;
  const float s2 = s * s;
  float o[32];
  if (J.mode == kSquare) {
    float am[32];
    const bool full = i < p && col0 + 32 <= p;
    if (i < p)
      load_row32(reinterpret_cast<const __nv_bfloat16 *>(J.aux) + S.p_off + (int64_t)i * S.ldp + col0, am, full,
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
  tma_store_block<kSlots>(&P.mapO[c], stage, slot, o, mirror, col0, i0, mat, lane);
  if (J.mode == kGramAP) {  // and A = s^2 C
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = s2 * v[k];
    tma_store_block<kSlots>(&P.mapO2[c], stage, slot, o, mirror, col0, i0, mat, lane);
  }
}

// The producer's and the MMA issuer's work for one tile, specialised on the
// operand layouts (A, B K-major or MN-major), so that the single-thread
// issue loops carry no per-k-block choices.  Return false on a time-out.
template <bool kPair, bool kAmn, bool kBmn>
__device__ __forceinline__ bool produce_tile(const TcParams &P, const TileCoord &tc, int half, int tm, uint8_t *smem,
                                             uint32_t full0, uint32_t empty0, uint32_t full_lead0, bool leader,
                                             uint32_t crank, int &stage, uint32_t &phase, uint32_t *armed_parity,
                                             bool *armed, volatile int32_t *abort_flag) {
  constexpr int STAGES = Mode<kPair>::kStages;
  constexpr int STAGE_BYTES = Mode<kPair>::kStageBytes;
  const CUtensorMap *ma = &P.mapA[tc.c], *mb = &P.mapB[tc.c];
  const int kit = P.k_iters[tc.c];
  const int m0 = tm * BM;
  // this CTA's first B row (column of C): a pair's N columns are split
  // between its two CTAs, N / 2 each.  A half tile (N = 128) loads 64 rows
  // of B per CTA: a 64-row box when B is K-major, one 64-column box when it
  // is MN-major.
  const int n0 = tc.tn * BN + (half >= 0 ? half * (BN / 2) + (int)crank * (BN / 4)
                                         : (kPair ? (int)crank * (BN / 2) : 0));
  const CUtensorMap *mbh = &P.mapBh[tc.c];
  constexpr int kHalfSaved = Mode<kPair>::kSub * (B_HALF / 2);  // B bytes per CTA a half tile's stage skips
  const uint32_t stage_tx = (uint32_t)((kPair ? 2 : 1) * (STAGE_BYTES - (half >= 0 ? kHalfSaved : 0)));
  for (int kb = 0; kb < kit; ++kb) {
    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1)) return false;
    if (*abort_flag) return true;
    if (leader) {
      mbar_expect_tx(full0 + 8 * stage, stage_tx);
      armed[stage] = true;
      armed_parity[stage] = phase;
    }
#pragma unroll
    for (int sub = 0; sub < Mode<kPair>::kSub; ++sub) {
    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES + sub * Mode<kPair>::kSubBytes);
    const uint32_t sb = sa + A_BYTES;
    const int k0 = (kb * Mode<kPair>::kSub + sub) * BK;
    if constexpr (kPair) {
      const uint32_t fb = full_lead0 + 8 * stage;
      if constexpr (!kAmn) {
        tma_load_3d_pair(sa, ma, fb, k0, m0, tc.mat);
      } else {  // this CTA's 128 rows of A = columns of X, as two 64-column boxes
#pragma unroll
        for (int h = 0; h < BM / 64; ++h) tma_load_3d_pair(sa + h * 8192, ma, fb, m0 + h * 64, k0, tc.mat);
      }
      if constexpr (!kBmn) {
        tma_load_3d_pair(sb, half >= 0 ? mbh : mb, fb, k0, n0, tc.mat);
      } else {
        for (int h = 0; h < (half >= 0 ? 1 : BN / 128); ++h)
          tma_load_3d_pair(sb + h * 8192, mb, fb, n0 + h * 64, k0, tc.mat);
      }
    } else {
      const uint32_t fb = full0 + 8 * stage;
      if constexpr (!kAmn) {
        tma_load_3d(sa, ma, fb, k0, m0, tc.mat);
      } else {
#pragma unroll
        for (int h = 0; h < BM / 64; ++h) tma_load_3d(sa + h * 8192, ma, fb, m0 + h * 64, k0, tc.mat);
      }
      if constexpr (!kBmn) {
#pragma unroll
        for (int h = 0; h < 2; ++h) tma_load_3d(sb + h * B_HALF, mb, fb, k0, n0 + h * (BN / 2), tc.mat);
      } else {
#pragma unroll
        for (int h = 0; h < BN / 64; ++h) tma_load_3d(sb + h * 8192, mb, fb, n0 + h * 64, k0, tc.mat);
      }
    }
    }
    if (++stage == STAGES) stage = 0, phase ^= 1;
  }
  return true;
}

template <bool kPair, bool kAmn, bool kBmn>
__device__ __forceinline__ bool mma_tile(uint8_t *smem, uint32_t full0, uint32_t empty0, uint32_t d_tmem, int kit,
                                         bool half, int &stage, uint32_t &phase, bool &issued) {
  constexpr int STAGES = Mode<kPair>::kStages;
  constexpr int STAGE_BYTES = Mode<kPair>::kStageBytes;
  constexpr uint32_t idesc_full = make_idesc(kAmn, kBmn, Mode<kPair>::kRows * BM);
  constexpr uint32_t idesc_half = make_idesc(kAmn, kBmn, Mode<kPair>::kRows * BM, BN / 2);
  const uint32_t idesc = half ? idesc_half : idesc_full;
  // descriptors of stage 0, K step 0: a stage is STAGE_BYTES further, a K
  // step of 16 is 32 bytes (K-major) or two 8-row groups, 2048 bytes (MN-major)
  const uint64_t a0 = smem_desc(smem_u32(smem), kAmn ? 8192 : 16, 1024);
  const uint64_t b0 = smem_desc(smem_u32(smem) + A_BYTES, kBmn ? 8192 : 16, 1024);
  constexpr uint32_t astep = (kAmn ? 2048 : 32) >> 4, bstep = (kBmn ? 2048 : 32) >> 4;
  for (int kb = 0; kb < kit; ++kb) {
    if (!mbar_wait(full0 + 8 * stage, phase)) return false;
    tc_fence_after();
#pragma unroll
    for (int sub = 0; sub < Mode<kPair>::kSub; ++sub) {
      const uint32_t soff = (uint32_t)(stage * STAGE_BYTES + sub * Mode<kPair>::kSubBytes) >> 4;
#pragma unroll
      for (int k = 0; k < BK / 16; ++k) {
        const uint32_t acc = (kb | sub | k) != 0;
        if constexpr (kPair) mma_bf16_pair(d_tmem, a0 + soff + k * astep, b0 + soff + k * bstep, idesc, acc);
        else mma_bf16_one(d_tmem, a0 + soff + k * astep, b0 + soff + k * bstep, idesc, acc);
      }
    }
    issued = true;
    if constexpr (kPair) mma_commit_pair_mc(empty0 + 8 * stage, 0x3);  // frees the slot in both CTAs
    else mma_commit_one(empty0 + 8 * stage);
    if (++stage == STAGES) stage = 0, phase ^= 1;
  }
  return true;
}

template <bool kPair>
__global__ void __launch_bounds__(Epi<kPair>::kThreads, 1)
ns_gemm_tc_kernel(const __grid_constant__ TcParams P, const __grid_constant__ PhaseArgs A) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up (see device_common.cuh)
  constexpr int STAGES = Mode<kPair>::kStages;
  constexpr int kRows = Mode<kPair>::kRows;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + smem_used<kPair>());
  // bars: full[STAGES], empty[STAGES], accf[2], acce[2], drain, (TMEM
  // address, abort flag), then the weight-load barriers of the epilogue warps
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
  uint64_t *wbars = bars + 2 * STAGES + 6;
  uint8_t *stage_base = smem + Mode<kPair>::kRingBytes;  // epilogue staging, 1024-byte aligned
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t accf0 = smem_u32(bars + 2 * STAGES), acce0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t drain = smem_u32(bars + 2 * STAGES + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = kPair ? cluster_rank() : 0u;
  const bool leader = crank == 0;

  // Barrier protocol.  Single mode: everything is local to the CTA.  Pair
  // mode (the even CTA leads):
  //   full[s]   leader only: both CTAs' copies of stage s complete_tx on it;
  //             the leader's producer arms it with both CTAs' bytes
  //   empty[s]  each CTA: the leader's MMA commit (multicast) frees slot s
  //   accf[a]   each CTA: the leader's MMA commit (multicast) says
  //             accumulator a is complete in both TMEMs
  //   acce[a]   leader only: one arrival per epilogue warp of both CTAs
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf0 + 8 * a, 1);
      mbar_init(acce0 + 8 * a, (kPair ? 2 : 1) * Epi<kPair>::kWarps);
    }
    mbar_init(drain, 1);
    for (int b = 0; b < Epi<kPair>::kWarps * Epi<kPair>::kWBufs; ++b) mbar_init(smem_u32(wbars + b), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // pair mode: one warp of each CTA allocates the pair's TMEM together
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
  const int64_t total = P.n_items;
  const int64_t cid = kPair ? (blockIdx.x >> 1) : blockIdx.x;
  const int64_t ncl = kPair ? (gridDim.x >> 1) : gridDim.x;
  const uint32_t full_lead0 = kPair ? map_to_rank(full0, 0) : full0;
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
        int half;
        const TileCoord tc = item_of<kRows>(P, t, half);
        const int tm = kRows * tc.tm + (int)crank;
        const int kind = P.job[tc.c].kind;
        bool ok;
        if (kind == kKindGramT)
          ok = produce_tile<kPair, true, true>(P, tc, half, tm, smem, full0, empty0, full_lead0, leader, crank, stage,
                                               phase, armed_parity, armed, abort_flag);
        else if (kind == kKindProd)
          ok = produce_tile<kPair, false, true>(P, tc, half, tm, smem, full0, empty0, full_lead0, leader, crank,
                                                stage, phase, armed_parity, armed, abort_flag);
        else
          ok = produce_tile<kPair, false, false>(P, tc, half, tm, smem, full0, empty0, full_lead0, leader, crank,
                                                 stage, phase, armed_parity, armed, abort_flag);
        if (!ok) { give_up(); break; }
      }
      if (*abort_flag && leader) {
        // let every copy armed here land before shared memory goes away
        for (int s = 0; s < STAGES; ++s)
          if (armed[s]) (void)mbar_wait(full0 + 8 * s, armed_parity[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool issued = false;
      for (int64_t t = cid; t < total && !*abort_flag; t += ncl) {
        int half;
        const TileCoord tc = item_of<kRows>(P, t, half);
        const int kit = P.k_iters[tc.c];
        const int kind = P.job[tc.c].kind;
        const bool freed = kPair ? mbar_wait_cluster(acce0 + 8 * acc, acc_phase ^ 1)
                                 : mbar_wait(acce0 + 8 * acc, acc_phase ^ 1);
        if (!freed) { give_up(); break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        bool ok;
        const bool hf = half >= 0;
        if (kind == kKindGramT)
          ok = mma_tile<kPair, true, true>(smem, full0, empty0, d_tmem, kit, hf, stage, phase, issued);
        else if (kind == kKindProd)
          ok = mma_tile<kPair, false, true>(smem, full0, empty0, d_tmem, kit, hf, stage, phase, issued);
        else
          ok = mma_tile<kPair, false, false>(smem, full0, empty0, d_tmem, kit, hf, stage, phase, issued);
        if (!ok) { give_up(); break; }
        if constexpr (kPair) mma_commit_pair_mc(accf0 + 8 * acc, 0x3);  // accumulator ready in both TMEMs
        else mma_commit_one(accf0 + 8 * acc);
        if (++acc == 2) acc = 0, acc_phase ^= 1;
      }
      if (*abort_flag && issued) {
        // wait for the outstanding MMAs before TMEM is released
        if constexpr (kPair) mma_commit_pair(drain);
        else mma_commit_one(drain);
        (void)mbar_wait(drain, 0);
      }
    }
  } else {
    // epilogue warps: TMEM lane quarter = warp % 4; in single mode two warps
    // per quarter, each over half of the tile's columns
    using E = Epi<kPair>;
    const int quarter = warp & 3;
    const int part = (warp - 2) / 4;                  // which span of the tile's columns
    const uint32_t stage = smem_u32(stage_base + (warp - 2) * E::kWarpStage);
    const uint32_t wbar0 = smem_u32(wbars + (warp - 2) * E::kWBufs);
    uint32_t wpar = 0, winfl = 0;  // weight-load barriers: next parities, loads in flight
    int slot = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t t = cid; t < total && !*abort_flag; t += ncl) {
      int half;
      const TileCoord tc = item_of<kRows>(P, t, half);
      const int sub = P.sub0[tc.c] + tc.mat;
      const DevSub &S = A.subs[sub];
      const TcJob &J = P.job[tc.c];
      const int i0 = (kRows * tc.tm + (int)crank) * BM + quarter * 32;
      // this warp's first column and the columns it covers (a half tile's
      // accumulator is the first 128 columns of its TMEM buffer)
      const int span = half >= 0 ? BN / 2 : E::kSpan;
      const int c0 = tc.tn * BN + (half >= 0 ? half * (BN / 2) : part * E::kSpan);
      // the job's output is rows x cols (stored orientation for the weights)
      const int rows = kind_rows(J.kind, S.p, S.q), cols = kind_cols(J.kind, S.p, S.q);
      // bf16 weights in blocks of 32 whole rows with a TMA map move by TMA
      // (their first loads overlap this tile's MMAs); the rest are
      // prefetched into L2 and read by the epilogue threads
      const CUtensorMap *wmap = (J.mode == kFinal && S.w_dtype == GBO_BF16 && S.wmap >= 0)
                                    ? static_cast<const CUtensorMap *>(A.wmaps) + S.wmap
                                    : nullptr;
      const bool live = i0 < rows && c0 < cols;      // this warp's part of the tile holds outputs
      const bool wtma = live && wmap != nullptr && i0 + 32 <= rows;
      if (wtma) weight_loads_begin<E::kWBufs>(wmap, stage, wbar0, c0, cols, (int)(S.r0 + i0), lane, winfl, span);
      else if (live && J.mode == kFinal) prefetch_weight_tile(S, i0, c0, rows, cols, lane, span);
      if (!mbar_wait(accf0 + 8 * acc, acc_phase)) { give_up(); break; }
      tc_fence_after();
      const float s = J.first ? A.alpha[sub] : 1.0f;
      const uint32_t trow =
          tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + part * E::kSpan);
      // the NorMuon last product leaves each row's sum of squares of the bf16
      // values it stores, one partial per 128 columns; with the per-matrix
      // norms asked for, the weight-writing last product leaves those of the
      // update direction
      const bool stats = (J.mode == kProduct || J.mode == kFinal) && J.aux != nullptr;
      float rss[E::kSpan / 128] = {};
      if (live) {  // warps whose rows or columns are all padding have nothing to write
        if (wtma) {
          if (!final_tile_bf16_tma<E::kWBufs>(A, S, s, i0, c0, cols, trow, lane, wmap, stage, wbar0, wpar, winfl,
                                              span, stats ? rss : nullptr)) {
            give_up();
            break;
          }
        } else if (J.mode == kFinal && S.w_dtype == GBO_BF16) {
          final_tile_bf16(A, S, s, i0, c0, rows, cols, trow, lane, span, stats ? rss : nullptr);
        } else {
#pragma unroll 1
          for (int ch = 0; ch < span / 32; ++ch) {
            const int col0 = c0 + ch * 32;
            if (col0 >= cols) break;  // column chunks past the output hold nothing to write
            float v[32];
            tmem_ld32(trow + ch * 32, v);
            epilogue_block<E::kSlots>(P, A, tc.c, tc.mat, S, s, i0, col0, v, stage, slot, lane);
            if (stats) {
              float r2 = 0.f;
              const float f = J.mode == kFinal ? S.scale * s : s;
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                const float r = J.mode == kFinal ? f * v[k] : __bfloat162float(__float2bfloat16_rn(f * v[k]));
                r2 = fmaf(r, r, r2);
              }
              rss[ch / 4] += r2;
            }
          }
        }
        if (stats && i0 + lane < rows) {
          float *part_out = static_cast<float *>(const_cast<void *>(J.aux)) + S.ss_off +
                            (int64_t)(i0 + lane) * S.ss_ntn + c0 / 128;
#pragma unroll
          for (int h = 0; h < E::kSpan / 128; ++h)
            if (128 * h < span && c0 + 128 * h < cols) part_out[h] = rss[h];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // this warp is done with accumulator `acc`
        if constexpr (kPair) mbar_arrive_cluster(acce_lead0 + 8 * acc);
        else mbar_arrive(acce0 + 8 * acc);
      }
      if (++acc == 2) acc = 0, acc_phase ^= 1;
    }
    // weight loads of an abandoned tile land, and this warp's TMA stores
    // complete, before the kernel ends
    for (int b = 0; b < E::kWBufs; ++b)
      if (winfl >> b & 1u) (void)mbar_wait(wbar0 + 8 * b, (wpar >> b) & 1u);
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

}  // namespace

// Matrices of at most 128 oriented rows run in single mode; larger ones in
// pairs.
bool single_mode(int p) { return p <= BM; }

// The weight-writing last product of a class of at most 256 rows runs on
// single CTAs too: with K = p its MMAs are short, its HBM-bound weight
// traffic is what limits it, and the single-CTA kernel has twice the
// epilogue warps per SM to hide that traffic's latency.
bool single_job(int p, int32_t mode) { return p <= BM || (mode == kFinal && p <= 2 * BM); }

namespace {

// Work items of one matrix: kRows consecutive 128-row tiles (1 on single
// CTAs, 2 on pairs) x one column tile, over an output of `rows` rows; in
// pair mode an odd tile-row count runs one all-padding tile in the last
// pair.
int items_m_of(bool single, int rows) {
  const int k = single ? 1 : 2;
  return ((rows + BM - 1) / BM + k - 1) / k;
}

int64_t sym_items_of(int p) {
  const bool single = single_mode(p);
  const int rows = single ? 1 : 2;
  const int tiles_n = (p + BN - 1) / BN;
  int64_t n = 0;
  for (int r = 0; r < items_m_of(single, p); ++r) n += std::max(0, tiles_n - tri_tn_min(rows * r));
  return n;
}

double item_flops(bool single, int kdim) {  // one work item: rows x 128 x 256 outputs, K padded to a stage
  const int rows = single ? 1 : 2;
  const int kstage = rows * BK;  // pairs stage two BK-wide blocks, single CTAs one
  return 2.0 * rows * BM * BN * (double)((kdim + kstage - 1) / kstage) * kstage;
}

double item_flops(int p, int kdim) { return item_flops(single_mode(p), kdim); }

// The p x q product (wide: p x q output) or its transpose (tall: q x p);
// `final`: the weight-writing last product.
double product_flops(int p, int q, bool tall, bool final) {
  const bool single = single_job(p, final ? kFinal : kProduct);
  return tall ? (double)items_m_of(single, q) * ((p + BN - 1) / BN) * item_flops(single, p)
              : (double)items_m_of(single, p) * ((q + BN - 1) / BN) * item_flops(single, p);
}

}  // namespace

double tc_executed_flops(int p, int q, bool square, bool tall, bool final) {
  double f = sym_items_of(p) * item_flops(p, q);                  // Gram, K = q
  if (square) f += sym_items_of(p) * item_flops(p, p);            // A A
  return f + product_flops(p, q, tall, final);                    // product, K = p
}

double tc_gram_route_flops(int p, int q, int k, int squares, bool tall, bool final) {
  return sym_items_of(p) * item_flops(p, q) + (3.0 * k - 3.0 + squares) * sym_items_of(p) * item_flops(p, p) +
         product_flops(p, q, tall, final);
}

double tc_gram_chain_flops(int p, int q, int k, const float *abc, bool tall, bool fused, bool final) {
  const double gram = fused ? tc_fused_gram_flops(p, q, abc)
                            : sym_items_of(p) * item_flops(p, q) +
                                  (abc[2] != 0.f ? sym_items_of(p) * item_flops(p, p) : 0.0);
  return gram + tc_chain_flops(p, k, abc) + product_flops(p, q, tall, final);
}

namespace {

// Class base of an operand or output region: X operands live in x-space,
// everything p x p in the class's own p-space.
inline const char *xbase(const void *region, const ShapeClass &C) {
  return static_cast<const char *>(region) + C.x_base * 2;
}
inline const char *pbase(const void *region, const ShapeClass &C) {
  return static_cast<const char *>(region) + C.p_base * 2;
}

template <bool kPair>
int launch_mode(const GemmJob *const *jobs, int32_t n_jobs, const PhaseArgs &args, int sm_count, void *stream,
                int64_t *n_launch) {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(ns_gemm_tc_kernel<kPair>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBytes);
  });
  if (attr_err != cudaSuccess) return (int)attr_err;
  constexpr int kRows = Mode<kPair>::kRows;
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
      void *x = const_cast<char *>(xbase(J.kind == kKindProd ? J.opB : J.opA, C));
      if (J.kind == kKindGram) {  // X wide: A = X rows, B = X rows, K = q
        ok = encode_map(&T.mapA[k], x, C.q, C.p, C.count, C.ld, BK, BM) &&
             encode_map(&T.mapB[k], x, C.q, C.p, C.count, C.ld, BK, BN / 2) &&
             (!kPair || encode_map(&T.mapBh[k], x, C.q, C.p, C.count, C.ld, BK, BN / 4));
        Mdim = C.p, Ndim = C.p, Kdim = C.q;
      } else if (J.kind == kKindGramT) {  // X tall: A and B = columns of X (MN-major boxes), K = q
        ok = encode_map(&T.mapA[k], x, C.p, C.q, C.count, C.ld, 64, BK) &&
             encode_map(&T.mapB[k], x, C.p, C.q, C.count, C.ld, 64, BK);
        Mdim = C.p, Ndim = C.p, Kdim = C.q;
      } else if (J.kind == kKindSym) {  // A = L rows, B = R rows (R symmetric), K = p
        ok = encode_map(&T.mapA[k], const_cast<char *>(pbase(J.opA, C)), C.p, C.p, C.count, C.ldp, BK, BM) &&
             encode_map(&T.mapB[k], const_cast<char *>(pbase(J.opB, C)), C.p, C.p, C.count, C.ldp, BK, BN / 2) &&
             (!kPair ||
              encode_map(&T.mapBh[k], const_cast<char *>(pbase(J.opB, C)), C.p, C.p, C.count, C.ldp, BK, BN / 4));
        Mdim = C.p, Ndim = C.p, Kdim = C.p;
      } else if (J.kind == kKindProd) {  // X wide: A = L rows (K = p), B = X with rows as K, columns as N
        ok = encode_map(&T.mapA[k], const_cast<char *>(pbase(J.opA, C)), C.p, C.p, C.count, C.ldp, BK, BM) &&
             encode_map(&T.mapB[k], x, C.q, C.p, C.count, C.ld, 64, BK);
        Mdim = C.p, Ndim = C.q, Kdim = C.p;
      } else {  // kKindProdT, X tall: A = X rows (K = p), B = L rows (L symmetric)
        ok = encode_map(&T.mapA[k], x, C.p, C.q, C.count, C.ld, BK, BM) &&
             encode_map(&T.mapB[k], const_cast<char *>(pbase(J.opB, C)), C.p, C.p, C.count, C.ldp, BK, BN / 2) &&
             (!kPair ||
              encode_map(&T.mapBh[k], const_cast<char *>(pbase(J.opB, C)), C.p, C.p, C.count, C.ldp, BK, BN / 4));
        Mdim = C.q, Ndim = C.p, Kdim = C.p;
      }
      // outputs stored by TMA: a p x p matrix in the class's p-space, or X'
      if (J.mode == kProduct) {
        char *xo = static_cast<char *>(J.out) + C.x_base * 2;
        ok = ok && (J.kind == kKindProdT
                        ? encode_map(&T.mapO[k], xo, C.p, C.q, C.count, C.ld, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)
                        : encode_map(&T.mapO[k], xo, C.q, C.p, C.count, C.ld, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B));
      } else if (J.mode != kFinal) {
        ok = ok && encode_map(&T.mapO[k], static_cast<char *>(J.out) + C.p_base * 2, C.p, C.p, C.count, C.ldp, 32,
                              32, CU_TENSOR_MAP_SWIZZLE_64B);
        if (J.mode == kGramAP)
          ok = ok && encode_map(&T.mapO2[k], static_cast<char *>(J.out2) + C.p_base * 2, C.p, C.p, C.count, C.ldp,
                                32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
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
      constexpr int kStageK = Mode<kPair>::kSub * BK;
      T.k_iters[k] = (Kdim + kStageK - 1) / kStageK;
      T.sub0[k] = C.sub0;
      const int items_m = ((Mdim + BM - 1) / BM + kRows - 1) / kRows;
      if (!is_product_kind(J.kind)) {
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
    cfg.blockDim = dim3(Epi<kPair>::kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    if constexpr (kPair) {
      // persistent grid: as many CTA pairs as can be resident at once
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
        if (cudaOccupancyMaxActiveClusters(&max_clusters, ns_gemm_tc_kernel<true>, &cfg) != cudaSuccess)
          max_clusters = 0;
      });
      // every pair the device holds, within the SMs this launch may use
      const int64_t resident = std::max(1, max_clusters > 0 ? std::min(max_clusters, sm_count / 2) : sm_count / 2);
      // tail split: a last partial wave of at most half the resident pairs
      // runs as half tiles, one per pair
      const int64_t rem = total % resident;
      const int64_t n_split = (g_tail_split.load() != 0 && rem > 0 && 2 * rem <= resident) ? rem : 0;
      T.split_base = total - n_split;
      T.n_items = total + n_split;
      const int clusters = (int)std::min<int64_t>(T.n_items, resident);
      cfg.gridDim = dim3(2 * clusters);
    } else {
      T.split_base = T.n_items = total;
      cfg.gridDim = dim3((unsigned)std::min<int64_t>(total, sm_count));  // one CTA per SM
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
    const cudaError_t lerr = cudaLaunchKernelEx(&cfg, ns_gemm_tc_kernel<kPair>, T, args);
    if (lerr != cudaSuccess) return (int)lerr;
    count_launches(1);
    if (n_launch) ++*n_launch;
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return (int)err;
  }
  return 0;
}

}  // namespace

namespace {

// The bounded wait of the Newton-Schulz kernel, on an mbarrier that nothing
// arrives on: it must give up after `limit_ns`, flag the time-out and
// return, leaving the context usable.
__global__ void wait_timeout_kernel(int32_t *status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (!mbar_wait_ns(b, 0, limit_ns)) flag_status(status, GBO_STATUS_TIMEOUT);
}

}  // namespace

int32_t set_tail_split(int32_t enable) { return g_tail_split.exchange(enable != 0 ? 1 : 0); }

int32_t pair_residency() {
  if (cudaFuncSetAttribute(ns_gemm_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
      cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(Epi<true>::kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  int dev = 0, sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  cfg.gridDim = dim3(2 * std::max(1, sm / 2));
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, ns_gemm_tc_kernel<true>, &cfg) == cudaSuccess ? n : -1;
}

int launch_wait_timeout(int32_t *status, uint64_t limit_ns, void *stream) {
  wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status, limit_ns);
  count_launches(1);
  return (int)cudaGetLastError();
}

int build_weight_maps(const gbo_muon_desc *descs, int32_t n, void **out) {
  *out = nullptr;
  if (n <= 0) return 0;
  std::vector<CUtensorMap> maps((size_t)n);
  memset(maps.data(), 0, maps.size() * sizeof(CUtensorMap));
  for (int32_t t = 0; t < n; ++t) {
    const gbo_muon_desc &d = descs[t];
    if (d.w_dtype != GBO_BF16 || (d.cols * 2) % 16 != 0 || (reinterpret_cast<uintptr_t>(d.w) & 15) != 0) continue;
    if (!encode_map(&maps[t], d.w, d.cols, d.rows, 1, d.cols, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return (int)cudaErrorInvalidValue;
  }
  void *dev = nullptr;
  cudaError_t e = cudaMalloc(&dev, maps.size() * sizeof(CUtensorMap));
  if (e != cudaSuccess) return (int)e;
  e = cudaMemcpy(dev, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(dev);
    return (int)e;
  }
  *out = dev;
  return 0;
}

int launch_ns_gemm_tc(const GemmJob *jobs, int32_t n_jobs, const PhaseArgs &globals, int sm_count, void *stream,
                      int64_t *n_launch) {
  std::vector<const GemmJob *> single, pair, chain;
  for (int32_t j = 0; j < n_jobs; ++j) {
    if (jobs[j].cls->count == 0) continue;
    if (jobs[j].mode == kChain) chain.push_back(&jobs[j]);
    else (single_job(jobs[j].cls->p, jobs[j].mode) ? single : pair).push_back(&jobs[j]);
  }
  int err = launch_mode<true>(pair.data(), (int32_t)pair.size(), globals, sm_count, stream, n_launch);
  if (err) return err;
  err = launch_mode<false>(single.data(), (int32_t)single.size(), globals, sm_count, stream, n_launch);
  if (err) return err;
  return launch_ns_chain_tc(chain.data(), (int32_t)chain.size(), globals, sm_count, stream, n_launch);
}

}  // namespace gbo
