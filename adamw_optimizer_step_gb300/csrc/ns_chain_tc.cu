// The Gram route's p x p iterations for matrices of at most 192 rows, on
// chip (bf16 mode).  With A_0 = X_0 X_0^T and P_0 from the Gram launch, the
// iterations of eq. (5) of the NorMuon paper (zskr.cn, section 2.2) become
// products of commuting symmetric p x p matrices,
//   T = P_j A_j,  Q_{j+1} = P_j Q_j (Q_1 = P_0),  A_{j+1} = P_j T,
//   P_{j+1} = a I + b A_{j+1} (+ c A_{j+1}^2),
// and only Q_k is needed for X_k = Q_k X_0.  For a small matrix every one of
// these products is one or two 128-row tiles, so instead of one launch per
// product, with each p x p result making a round trip through HBM, one CTA
// keeps the matrix's P, A (or T) and Q in shared memory as bf16 MMA operands
// and runs the whole chain: loads A_0 and P_0 by TMA, runs each product on
// the tensor cores (tcgen05.mma, fp32 accumulators in TMEM), turns the
// accumulator back into the next bf16 operand in shared memory, and stores
// Q_k by TMA.  The left operand is read K-major (rows of L) and the right
// one MN-major (rows of R as K), so no product relies on its operands being
// exactly symmetric: intermediate results are written whole, row by row,
// each element rounded to bf16 once.  Q_k leaves mirrored from its upper
// triangle, as the tile kernel's epilogue stores symmetric results, because
// the product of a tall X_0 with Q_k takes Q_k's rows as its columns.
//
// For a matrix with p <= 128 the Gram itself runs here too (kFuse): X_0
// streams in by TMA, 64 columns at a time (64 rows of an X_0 held tall, q x
// p, whose Gram X_0^T X_0 reads both operands MN-major), through a ring of
// six 16 KB stages laid over the slot's own P, A and Q (free until the
// Gram's epilogue writes them), the MMAs accumulate the Gram in the slot's
// TMEM columns, and the epilogue folds in the pre-normalisation factor and
// writes A_0, P_0 and Q_1 = P_0 (with c != 0, A_0 and then P_0 from an
// on-chip square).  Each slot then has an MMA issuer of its own, and the
// epilogue warps poll both slots instead of taking them in turn, so one
// slot's X_0 stream (bound by HBM) runs under the other slot's chain (bound
// by latency) and neither slot's ops queue behind the other's issue.
//
// The momentum pass can run here too (kMom, with kFuse, for wide matrices
// with bf16 gradients on 16-byte rows): instead of X_0, G and B stream in
// by TMA through per-weight maps, 64 columns of the matrix's rows at a
// time, in two 48 KB stages per slot laid over the slot's P, A and Q.  The
// epilogue warps, between their chain epilogues, turn each landed stage
// into B <- mu B + G and D = G + mu B (NorMuon paper, section 2.2, eq. (1);
// OMN page, Muon path), write B and X_0 = bf16(D) to HBM and bf16(D) in
// place over G as the Gram's K-major operand, and keep per-thread running
// statistics (max |D| and the sum of (D / max)^2, rescaled when the max
// grows, so nothing can overflow).  After a matrix's last stage every warp
// publishes its statistics; the Gram epilogue combines them in a fixed
// order into the pre-normalisation factor (OMN page: max-abs rescale, then
// the Frobenius norm, each with its 1e-7), which it folds into A_0 and also
// writes out for the last product.  X_0 is then never read back for the
// Gram, and the memory-bound momentum pass of these matrices runs under the
// latency-bound chain of the other slot.
//
// Two geometries (template parameter kH, 128-row halves of a matrix):
//   kH = 1  p <= 128: 128 x 128 matrices (32 KB each), two matrices in
//           flight per CTA so the epilogue of one slot's product overlaps
//           the other slot's MMAs; T and Q_{j+1} are one N = 256 product
//           over [A | Q] (two 128-column accumulators side by side)
//   kH = 2  128 < p <= 192: 192 x 192 matrices (72 KB each), one matrix per
//           CTA; each product is two M = 128 row halves with N = 192, and
//           T and Q_{j+1} are separate products (their accumulators would
//           not fit TMEM together)
// Persistent CTA (320 threads, 352 with kFuse; one per SM):
//   warp 0      TMA loads (one lane): A_0, P_0 (into P and Q) of the next
//               matrix of each slot, or its X_0 blocks (kFuse)
//   warp 1      TMEM owner and MMA issuer (one lane): alternating slots, or
//               (kFuse) slot 0 only
//   warps 2..9  epilogue, two per TMEM lane quarter, each taking half of
//               the column blocks of the quarter's rows
//   warp 10     (kFuse) MMA issuer of slot 1, so that neither slot's chain
//               ops queue behind the other slot's bursts of Gram MMAs
// Every wait is bounded: on time-out the kernel flags GBO_STATUS_TIMEOUT,
// lets its own copies and MMAs land (bounded), frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
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

constexpr int CK = 64;                        // 64 bf16: one 128-byte swizzle row
constexpr int kCEpiWarps = 8;
constexpr int kCThreads = 64 + 32 * kCEpiWarps;
constexpr int kMaxOps = 4 * GBO_MAX_NS_STEPS + 1;
constexpr int kCTmemCols = 512;
constexpr int kRing = 6;                 // X_0 blocks in flight per slot (kFuse)
constexpr int kRingBytes = 128 * CK * 2; // one 128-row, 64-column bf16 block of X_0
constexpr int kMRing = 2;                // kMom: G and B blocks in flight per slot
constexpr int kMGBytes = 128 * CK * 2;   // kMom: a stage's G block (p x 64 bf16, then X_0's operand in place)
constexpr int kMStage = kMGBytes + 128 * CK * 4;  // ... followed by its B block (p x 64 fp32): 48 KB
// loaded, mmad, epid, qdone, freed (2 each), drain, full/empty rings, drain2,
// then (kMom) the rings' computed barriers and the statistics barriers
constexpr int kNBars = 12 + 4 * kRing + 2 * kRing + 2;
constexpr int kNClocks = 20;             // idle-stretch starts: one per warp
// kFuse: a second MMA issuer warp (slot 1) after the epilogue warps; with
// 11 warps a scheduler still holds at most three, so the register budget
// per thread is that of 10
constexpr int kIssuer2 = kCThreads / 32;
// kMom: five warpgroups.  Warp 0 loads, warps 1 and 2 issue slot 0's and
// slot 1's MMAs, warp 3 idles; warps 4..11 are the chain's epilogue warps;
// warps 12..19 run the momentum pass.  setmaxnreg moves registers from the
// first and last groups to the epilogue warps; the shares must not exceed
// the launch's 640 threads x registers per thread (checked before launch).
constexpr int kMomWarps = 8;
constexpr int kMomWarp0 = 12;
constexpr int kRegsCtl = 48, kRegsEpi = 152, kRegsMom = 56;
constexpr int kMomRegShares = 128 * kRegsCtl + 256 * kRegsEpi + 256 * kRegsMom;
template <bool kFuse, bool kMom = false>
constexpr int chain_threads() { return kMom ? 32 * (kMomWarp0 + kMomWarps) : kCThreads + (kFuse ? 32 : 0); }
// first epilogue warp
template <bool kMom>
constexpr int epi_warp0() { return kMom ? 4 : 2; }

// Shared-memory geometry of one slot matrix (K-major rows of 128 bytes in
// 64-column blocks, 128-byte swizzle, as TMA writes it).
template <int kH>
struct Geo {
  static constexpr int R = kH == 1 ? 128 : 192;  // rows (= columns) of a slot matrix
  static constexpr int KB = R / CK;              // 64-column blocks
  static constexpr int Blk = R * 128;            // bytes of one 64-column block
  static constexpr int Mat = KB * Blk;           // 32 KB or 72 KB
  static constexpr int Slots = kH == 1 ? 2 : 1;
  static constexpr int SlotSize = 3 * Mat;       // P, A (or T), Q
  static constexpr int Smem = 1024 /*align*/ + Slots * SlotSize + 1024 /*barriers, statistics*/;
  static constexpr int WarpBlocks = R / 64;      // 32-column blocks per epilogue warp and row block
  // kind::f16: fp32 accumulator, bf16 A and B, A K-major, B MN-major, M = 128, N = R
  static constexpr uint32_t Idesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                    ((uint32_t)(R >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  // the Gram: A and B K-major (rows of a wide X_0) or both MN-major (an
  // X_0 held tall)
  static constexpr uint32_t IdescK = Idesc & ~(1u << 16);
  static constexpr uint32_t IdescMN = Idesc | (1u << 15);
  // N = 256 (kH = 1): T and Q_{j+1} in one product, B = [A | Q], the two
  // matrices side by side in shared memory
  static constexpr uint32_t IdescN2 = (Idesc & ~(0x3Fu << 17)) | ((uint32_t)(2 * R >> 3) << 17);
};
static_assert(Geo<1>::Smem <= 232448 && Geo<2>::Smem <= 232448, "shared memory per CTA");
static_assert(kRing * kRingBytes <= Geo<1>::SlotSize, "the X_0 ring lies within one slot");
static_assert(Geo<1>::Mat == 2 * Geo<1>::Blk, "kH = 1: Q's two 64-column blocks follow A's, one N = 256 operand");
static_assert(kMRing * kMStage <= Geo<1>::SlotSize, "the G and B ring lies within one slot");
static_assert((kNBars + 1 + kNClocks) * 8 + 2 * 2 * kMomWarps * 4 <= 1024,
              "barriers, TMEM address, abort flag, idle clocks and the momentum statistics");

// Products of slot matrices (L R: L read K-major, R MN-major) and
// epilogues of one op of the chain.
enum ChainMma : int32_t {
  kMmaPA = 0,   // acc0 = P A
  kMmaPAQ = 1,  // acc0 = P A, acc1 = P Q (kH = 1)
  kMmaAA = 2,   // acc0 = A A
  kMmaPQ = 3,   // acc0 = P Q
  kMmaGram = 4, // acc0 = X_0 X_0^T, streamed (kFuse)
};
enum ChainEpi : int32_t {
  kEpiT = 0,    // A <- acc0 (T)
  kEpiTQ = 1,   // A <- acc0 (T), Q <- acc1 (kH = 1)
  kEpiAP = 2,   // A <- acc0, P <- a I + b acc0
  kEpiA = 3,    // A <- acc0
  kEpiP = 4,    // P <- a I + b acc0
  kEpiSq = 5,   // P <- a I + b A + c acc0 (acc0 = A A)
  kEpiOut = 6,  // Q <- acc0, then Q is stored to HBM
  kEpiQ = 7,    // Q <- acc0 (kH = 2)
  kEpiGram = 8, // A <- s^2 acc0, P and Q <- a I + b s^2 acc0 (kFuse, c == 0)
  kEpiGramA = 9,// A <- s^2 acc0 (kFuse, c != 0)
  kEpiSqQ = 10, // P and Q <- a I + b A + c acc0 (acc0 = A A; kFuse, c != 0)
};

struct ChainOp {
  int32_t mma, epi;
  float a, b, c;
};

struct ChainParams {
  CUtensorMap mapP[kMaxClassesPerLaunch];  // P_0 (loads: 64-column boxes of R rows, 128-byte swizzle)
  CUtensorMap mapA[kMaxClassesPerLaunch];  // A_0
  CUtensorMap mapQ[kMaxClassesPerLaunch];  // Q_k (stores, same boxes)
  CUtensorMap mapX[kMaxClassesPerLaunch];  // X_0 (kFuse): p x q in 64-column boxes of 128 rows, or q x p
                                           // (tall) in 64 x 64 boxes
  int64_t mat_start[kMaxClassesPerLaunch + 1];
  int32_t p[kMaxClassesPerLaunch];
  int32_t q[kMaxClassesPerLaunch];         // kFuse: the Gram's K (columns of X_0, rows when tall)
  int32_t tall[kMaxClassesPerLaunch];      // kFuse: X_0 held q x p
  int32_t sub0[kMaxClassesPerLaunch];      // kFuse: the class's first matrix in the pre-normalisation factors
  void *x0;                                // kMom: the X_0 region (each matrix at its DevSub x_off)
  int32_t n;
  int32_t n_ops;
  ChainOp ops[kMaxOps];
};

template <int kH>
__device__ __forceinline__ void chain_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate,
                                          uint32_t idesc = Geo<kH>::Idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Row half h of D = L R over kit 64-wide K blocks, in 16-wide K steps; L and
// R are slot matrices at shared-memory addresses l and r (with the N = 256
// descriptor, R and the matrix after it).  L is K-major: its
// rows 128 h .. start 16 KB into each block, a K step of 16 is 32 bytes
// along its rows, a K block the next 64-column block.  R is MN-major: its
// rows are K, a K step is two 8-row groups (2048 bytes), a K block 64 rows
// (8192 bytes), and its N columns continue in the next 64-column block
// (leading byte offset Blk).  Rows 192 .. 255 of an L with kH = 2 lie in the
// buffer after it (A after P, Q after A): they feed only accumulator rows
// that are never written back.
template <int kH>
__device__ __forceinline__ void chain_product(uint32_t d_tmem, uint32_t l, uint32_t r, int kit, int h,
                                              uint32_t idesc = Geo<kH>::Idesc) {
  const uint64_t ld = smem_desc(l + (uint32_t)h * 16384u, 16, 1024), rd = smem_desc(r, Geo<kH>::Blk, 1024);
  for (int kb = 0; kb < kit; ++kb)
#pragma unroll
    for (int k = 0; k < CK / 16; ++k)
      chain_mma<kH>(d_tmem, ld + ((uint32_t)(kb * Geo<kH>::Blk + k * 32) >> 4),
                    rd + ((uint32_t)(kb * 8192 + k * 2048) >> 4), (kb | k) != 0, idesc);
}

// Byte offset of 16-byte chunk q (columns 8q .. 8q + 7) of row r of a slot
// matrix: the chunk index within a 128-byte row XOR the row index mod 8.
template <int kH>
__device__ __forceinline__ uint32_t sw128(int r, int q) {
  return (uint32_t)((q >> 3) * Geo<kH>::Blk + r * 128 + (((q & 7) ^ (r & 7)) << 4));
}

// Lane r writes row i, columns col0 .. col0 + 31 (col0 a multiple of 32),
// as bf16.
template <int kH>
__device__ __forceinline__ void put_row(uint32_t m, int i, int col0, const float (&o)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(m + sw128<kH>(i, col0 / 8 + q)),
                 "r"(pack_bf16(o[8 * q], o[8 * q + 1])), "r"(pack_bf16(o[8 * q + 2], o[8 * q + 3])),
                 "r"(pack_bf16(o[8 * q + 4], o[8 * q + 5])), "r"(pack_bf16(o[8 * q + 6], o[8 * q + 7]))
                 : "memory");
}

// The transpose: element (i, col0 + k) goes to (col0 + k, i).
template <int kH>
__device__ __forceinline__ void put_col(uint32_t m, int i, int col0, const float (&o)[32]) {
  const uint32_t byte = (uint32_t)((i & 7) * 2);
#pragma unroll
  for (int k = 0; k < 32; ++k)
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(m + sw128<kH>(col0 + k, i >> 3) + byte),
                 "h"(__bfloat16_as_ushort(__float2bfloat16_rn(o[k])))
                 : "memory");
}

template <int kH>
__device__ __forceinline__ void get_row(uint32_t m, int i, int col0, float (&o)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(m + sw128<kH>(i, col0 / 8 + q))
                 : "memory");
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[h]);
      o[8 * q + 2 * h] = __low2float(b);
      o[8 * q + 2 * h + 1] = __high2float(b);
    }
  }
}

// Rows and columns at or past p hold zeros (the padding the next products
// multiply by).
__device__ __forceinline__ void mask_pad(int i, int col0, int p, float (&o)[32]) {
  if (i >= p) {
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = 0.f;
  } else if (col0 + 32 > p) {
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (col0 + k >= p) o[k] = 0.f;
  }
}

// Q_k leaves the accumulator as the tile kernel stores a symmetric result:
// of the 32 x 32 blocks, one on the diagonal is written whole, one above it
// is written with its mirror, one below it is skipped.
template <int kH>
__device__ __forceinline__ void put_sym(uint32_t m, int i, int i0, int col0, int p, float (&o)[32]) {
  mask_pad(i, col0, p, o);
  put_row<kH>(m, i, col0, o);
  if (col0 >= i0 + 32) put_col<kH>(m, i, col0, o);
}

template <int kH>
__device__ __forceinline__ void put_full(uint32_t m, int i, int col0, int p, float (&o)[32]) {
  mask_pad(i, col0, p, o);
  put_row<kH>(m, i, col0, o);
}

__device__ __forceinline__ int chain_class(const ChainParams &P, int64_t t) {
  int c = 0;
  while (c + 1 < P.n && P.mat_start[c + 1] <= t) ++c;
  return c;
}

// One op's epilogue for the rows of one TMEM lane quarter and column blocks
// cb0 .. cb1 - 1 of a slot's matrices at mP, mA, mQ; acc0 is the quarter's
// first accumulator column of the slot, s2 the square of the matrix's
// pre-normalisation factor (the Gram ops).
template <int kH, bool kFuse>
__device__ __forceinline__ void chain_epilogue(const ChainOp &o, uint32_t acc_row, int quarter, int lane, int cb0,
                                               int cb1, int p, float s2, uint32_t mP, uint32_t mA, uint32_t mQ) {
  using G = Geo<kH>;
  for (int h = 0; h < kH; ++h) {
    const int i0 = h * 128 + quarter * 32, i = i0 + lane;
    if (i0 >= G::R) continue;  // kH = 2: rows 192 .. 255 are padding
    const uint32_t acc0 = acc_row + (uint32_t)(h * 256);
    const uint32_t acc1 = acc0 + 128;
    // whole rows for the next products; Q_k: blocks on or above the
    // diagonal, mirrored
    for (int cb = o.epi == kEpiOut ? max(i0 / 32, cb0) : cb0; cb < cb1; ++cb) {
      const int col0 = cb * 32;
      float v[32];
      tmem_ld32(acc0 + col0, v);
      float w[32];
      switch (o.epi) {
        case kEpiT:
        case kEpiA:
          put_full<kH>(mA, i, col0, p, v);
          break;
        case kEpiQ:
          put_full<kH>(mQ, i, col0, p, v);
          break;
        case kEpiOut:
          put_sym<kH>(mQ, i, i0, col0, p, v);
          break;
        case kEpiTQ:
          put_full<kH>(mA, i, col0, p, v);
          tmem_ld32(acc1 + col0, w);
          put_full<kH>(mQ, i, col0, p, w);
          break;
        case kEpiAP:
        case kEpiP:
#pragma unroll
          for (int k = 0; k < 32; ++k) w[k] = o.b * v[k] + (i == col0 + k ? o.a : 0.f);
          if (o.epi == kEpiAP) put_full<kH>(mA, i, col0, p, v);
          put_full<kH>(mP, i, col0, p, w);
          break;
        case kEpiGram:  // A first, then P and Q from a second read of the accumulator
          if constexpr (kFuse) {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] *= s2;
            put_full<kH>(mA, i, col0, p, v);
            tmem_ld32(acc0 + col0, v);
            const float bs2 = o.b * s2;
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = bs2 * v[k] + (i == col0 + k ? o.a : 0.f);
            put_full<kH>(mP, i, col0, p, v);
            put_full<kH>(mQ, i, col0, p, v);
          }
          break;
        case kEpiGramA:
          if constexpr (kFuse) {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] *= s2;
            put_full<kH>(mA, i, col0, p, v);
          }
          break;
        default: {  // kEpiSq, kEpiSqQ
          float am[32];
          get_row<kH>(mA, i, col0, am);
#pragma unroll
          for (int k = 0; k < 32; ++k) w[k] = o.c * v[k] + o.b * am[k] + (i == col0 + k ? o.a : 0.f);
          put_full<kH>(mP, i, col0, p, w);
          if (kFuse && o.epi == kEpiSqQ) put_full<kH>(mQ, i, col0, p, w);
          break;
        }
      }
    }
  }
}

// Warp-uniform test of an mbarrier phase (lane 0 polls, the warp follows);
// non-blocking, since the caller polls other barriers when this one is not
// ready.
__device__ __forceinline__ bool warp_try(uint32_t bar, uint32_t parity, int lane) {
  int ok = 0;
  if (lane == 0) ok = mbar_test(bar, parity) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// A polling loop's bound: true once nothing has moved for kWaitNs.  The
// start of the idle stretch is kept in shared memory (at t0), not in a
// register across the loop.
struct IdleClock {
  volatile uint64_t *t0;
  uint32_t spin = 0;
  __device__ __forceinline__ explicit IdleClock(uint64_t *at) : t0(at) {}
  __device__ __forceinline__ bool expired(bool moved) {
    if (moved) {
      spin = 0;
      return false;
    }
    if (spin++ == 0) *t0 = global_ns();
    return (spin & 255u) == 0 && global_ns() - *t0 > kWaitNs;
  }
};

// kMom: a thread's running statistics of the direction D over its elements:
// m = max |D|, ss = sum of (D / m)^2 (rescaled whenever m grows), inv = 1 / m.
struct MomStats {
  float m, ss, inv;
};

__device__ __forceinline__ void mom_accumulate(MomStats &st, const float (&d)[4]) {
  const float gm = fmaxf(fmaxf(fabsf(d[0]), fabsf(d[1])), fmaxf(fabsf(d[2]), fabsf(d[3])));
  if (gm > st.m) {
    const float inv = 1.0f / gm;
    const float r = st.m * inv;
    st.ss *= r * r;
    st.m = gm;
    st.inv = inv;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float y = d[k] * st.inv;
    st.ss = fmaf(y, y, st.ss);
  }
}

// kMom: the momentum pass over one landed stage (columns 64 kb .. + 63 of
// matrix S) for the rows of epilogue warp ew: rows 2 ew + 16 j + (lane >> 4),
// columns 4 (lane & 15) .. + 3 of the block.  B <- mu B + G and X_0 =
// bf16(D) go to HBM (columns past the matrix are not stored); bf16(D)
// replaces G in the stage as the Gram's K-major operand (128-byte swizzle),
// for every column of the block (TMA filled the ones past the matrix with
// zeros, so D is zero there).  Rows at or past the matrix's are left alone:
// they feed only accumulator entries the Gram epilogue discards.
__device__ __forceinline__ void mom_stage(uint32_t stage, const DevSub &S, __nv_bfloat16 *x0, int kb, int ew,
                                          int lane, float mu, int nesterov, MomStats &st) {
  // the matrix's fields in registers: the stores below could alias the
  // table as far as the compiler knows, and would force a reload of each
  // field after every store
  const int m = S.m;
  const int64_t cols = S.cols, ld = S.ld;
  const int c4 = lane & 15;
  const int col = kb * CK + 4 * c4;
  const bool colok = col < S.n;
  float *__restrict__ bg = S.mom + S.r0 * cols + col;
  __nv_bfloat16 *__restrict__ xg = x0 + S.x_off + col;
  for (int j = 0; j < 128 / 16; j += 2) {
    uint32_t gv[2][2] = {}, bv[2][4] = {};
    int rr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      rr[h] = (j + h) * 16 + 2 * ew + (lane >> 4);
      if (rr[h] < m) {
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                     : "=r"(gv[h][0]), "=r"(gv[h][1])
                     : "r"(stage + (uint32_t)(rr[h] * 128 + c4 * 8))
                     : "memory");
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(bv[h][0]), "=r"(bv[h][1]), "=r"(bv[h][2]), "=r"(bv[h][3])
                     : "r"(stage + (uint32_t)(kMGBytes + rr[h] * 256 + c4 * 16))
                     : "memory");
      }
    }
    __syncwarp();  // every lane has read its G before the rows are overwritten in place
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rr[h];
      if (r >= m) continue;
      float g[4], nb[4], d[4];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162 *>(&gv[h][k]);
        g[2 * k] = __low2float(b2);
        g[2 * k + 1] = __high2float(b2);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        nb[k] = fmaf(mu, __uint_as_float(bv[h][k]), g[k]);
        d[k] = nesterov ? fmaf(mu, nb[k], g[k]) : nb[k];
      }
      const uint32_t p01 = pack_bf16(d[0], d[1]), p23 = pack_bf16(d[2], d[3]);
      if (colok) {
        *reinterpret_cast<float4 *>(bg + (int64_t)r * cols) = make_float4(nb[0], nb[1], nb[2], nb[3]);
        *reinterpret_cast<uint2 *>(xg + (int64_t)r * ld) = make_uint2(p01, p23);
      }
      asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(stage + (uint32_t)(r * 128 + ((((c4 >> 1) ^ (r & 7))) << 4) +
                                                                          (c4 & 1) * 8)),
                   "r"(p01), "r"(p23)
                   : "memory");
      mom_accumulate(st, d);
    }
  }
}

template <int kH, bool kFuse, bool kMom>
__global__ void __launch_bounds__(chain_threads<kFuse, kMom>(), 1)
ns_chain_kernel(const __grid_constant__ ChainParams P, const __grid_constant__ PhaseArgs A) {
  pdl_launch();  // the next kernel may be scheduled as SMs free up (see device_common.cuh)
  using G = Geo<kH>;
  static_assert(!kFuse || kH == 1, "the Gram runs on chip for p <= 128 only");
  static_assert(!kMom || kFuse, "the momentum pass runs on chip only with the Gram");
  constexpr int kStages = kMom ? kMRing : kRing;         // ring stages per slot
  constexpr int kStageBytes = kMom ? kMStage : kRingBytes;
  constexpr int S = G::Slots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * G::SlotSize);
  // bars: loaded[2], mmad[2], epid[2], qdone[2], freed[2], drain, full[2][kRing],
  // empty[2][kRing], drain2, then the TMEM address and the abort flag, then
  // one idle clock per warp
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNBars);
  uint64_t *clocks = bars + kNBars + 1;
  // kMom: per slot and epilogue warp, (max |D|, sum of (D / max)^2)
  volatile float *mpart = reinterpret_cast<volatile float *>(clocks + kNClocks);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
  const uint32_t loaded0 = smem_u32(bars), mmad0 = smem_u32(bars + 2), epid0 = smem_u32(bars + 4);
  const uint32_t qdone0 = smem_u32(bars + 6), freed0 = smem_u32(bars + 8), drain = smem_u32(bars + 10);
  const uint32_t full0 = smem_u32(bars + 11), empty0 = smem_u32(bars + 11 + 2 * kRing);
  const uint32_t drain2 = smem_u32(bars + 11 + 4 * kRing);
  const uint32_t cfull0 = smem_u32(bars + 12 + 4 * kRing), momdone0 = smem_u32(bars + 12 + 6 * kRing);
  auto full_bar = [&](int s, int st) { return full0 + (uint32_t)(8 * (s * kRing + st)); };
  auto empty_bar = [&](int s, int st) { return empty0 + (uint32_t)(8 * (s * kRing + st)); };
  // kMom: a stage's momentum pass is done (all epilogue warps) and its
  // operand may be read; a slot's matrix has its statistics published
  auto cfull_bar = [&](int s, int st) { return cfull0 + (uint32_t)(8 * (s * kRing + st)); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(loaded0 + 8 * s, 1);
      mbar_init(mmad0 + 8 * s, 1);
      mbar_init(epid0 + 8 * s, kCEpiWarps);
      mbar_init(qdone0 + 8 * s, kCEpiWarps);
      mbar_init(freed0 + 8 * s, 1);
      if (kFuse)
        for (int st = 0; st < kStages; ++st) {
          mbar_init(full_bar(s, st), 1);
          mbar_init(empty_bar(s, st), 1);
          if (kMom) mbar_init(cfull_bar(s, st), kMomWarps);
        }
      if (kMom) mbar_init(momdone0 + 8 * s, kMomWarps);
    }
    mbar_init(drain, 1);
    mbar_init(drain2, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kCTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int64_t total = P.mat_start[P.n];
  const uint32_t slots = smem_u32(smem);
  // matrix g of this CTA is blockIdx.x + g * gridDim.x, in slot g % S; a
  // slot's matrices run P.n_ops ops each, counted by u (barrier phases)
  auto mat_of = [&](int64_t g) { return (int64_t)blockIdx.x + g * (int64_t)gridDim.x; };
  auto give_up = [&]() {
    *abort_flag = 1;
    flag_status(A.status, GBO_STATUS_TIMEOUT);
  };
  constexpr int kE0 = epi_warp0<kMom>();
  const int issuer1 = kMom ? 2 : kIssuer2;
  // kMom: each role branch first sets its warpgroup's register share (all
  // four warps of a warpgroup take the same one), so that the compiler
  // allocates the branch's code within it

  if (warp == 0) {
    if constexpr (kMom) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (lane == 0) {
      int64_t armed[S], ring_n[S];  // the loads of the slot's last matrix; X_0 blocks loaded
      for (int s = 0; s < S; ++s) armed[s] = -1, ring_n[s] = 0;
      bool stop = false;
      if constexpr (kMom) {
        // Both slots stream at once: polling the two, each slot's next block
        // is issued as soon as its ring has a free stage (and, for the
        // slot's next matrix, once the previous one has left the slot), so
        // one slot's loads keep going while the other slot's chain runs and
        // the bytes in flight are not capped by one slot's ring.  (The
        // X_0-streaming variant loads matrix by matrix: there the chain, not
        // the stream, bounds the time, and streaming both slots at once
        // delays both chains; measured slower.)
        int64_t cur[S];  // the slot's current matrix
        int kbn[S];      // its next block
        bool open[S];    // the slot's previous matrix has left it
        for (int s = 0; s < S; ++s) cur[s] = s, kbn[s] = 0, open[s] = false;
        IdleClock idle(clocks + warp);
        for (bool any = true; any && !stop && !*abort_flag;) {
          any = false;
          bool moved = false;
          for (int s = 0; s < S; ++s) {
            const int64_t t = mat_of(cur[s]);
            if (t >= total) continue;
            any = true;
            const int64_t gs = cur[s] / S;  // the slot's matrix count so far
            if (!open[s]) {
              if (gs >= 1 && !mbar_test(freed0 + 8 * s, (uint32_t)((gs - 1) & 1))) continue;
              open[s] = true;
            }
            const int64_t n = ring_n[s];
            const int st = (int)(n % kStages);
            // a stage is reloaded once the MMAs that read it have completed
            if (n >= kStages && !mbar_test(empty_bar(s, st), (uint32_t)((n / kStages - 1) & 1))) continue;
            const int c = chain_class(P, t);
            const int mat = (int)(t - P.mat_start[c]);
            const int nk = (P.q[c] + CK - 1) / CK;
            const int kb = kbn[s];
            const uint32_t dst = slots + s * G::SlotSize + st * kStageBytes;
            // G and B: 64 columns of the matrix's rows, through its weight's maps
            const DevSub &Sd = A.subs[P.sub0[c] + mat];
            const CUtensorMap *gmap = static_cast<const CUtensorMap *>(A.gbmaps) + 2 * Sd.gbmap;
            mbar_expect_tx(full_bar(s, st), (uint32_t)P.p[c] * (CK * 2 + CK * 4));
            tma_load_3d(dst, gmap, full_bar(s, st), kb * CK, (int)Sd.r0, 0);
            tma_load_3d(dst + kMGBytes, gmap + 1, full_bar(s, st), kb * CK, (int)Sd.r0, 0);
            ring_n[s] = n + 1;
            moved = true;
            if (++kbn[s] == nk) kbn[s] = 0, cur[s] += S, open[s] = false;
          }
          if (any && idle.expired(moved)) {
            give_up();
            stop = true;
          }
          if (!moved) __nanosleep(64);  // a pass with nothing to issue: leave the issue slots to others
        }
      } else {
        for (int64_t g = 0; mat_of(g) < total && !stop && !*abort_flag; ++g) {
          const int s = (int)(g % S);
          const int64_t gs = g / S;  // the slot's matrix count so far
          if (gs >= 1 && !mbar_wait(freed0 + 8 * s, (uint32_t)((gs - 1) & 1))) {
            give_up();
            break;
          }
          const int64_t t = mat_of(g);
          const int c = chain_class(P, t);
          const int mat = (int)(t - P.mat_start[c]);
          const uint32_t base = slots + s * G::SlotSize;
          if constexpr (kFuse) {
            // X_0 in blocks of 64 along K (a tall X_0's 64-row block as two
            // 64 x 64 boxes, the second holding columns 64 .. 127); a stage is
            // reloaded once the MMAs that read it have completed
            const int nk = (P.q[c] + CK - 1) / CK;
            for (int kb = 0; kb < nk; ++kb) {
              const int64_t n = ring_n[s];
              const int st = (int)(n % kRing);
              if (n >= kRing && !mbar_wait(empty_bar(s, st), (uint32_t)((n / kRing - 1) & 1))) {
                give_up();
                stop = true;
                break;
              }
              const uint32_t dst = base + st * kRingBytes;
              mbar_expect_tx(full_bar(s, st), kRingBytes);
              if (P.tall[c]) {
                tma_load_3d(dst, &P.mapX[c], full_bar(s, st), 0, kb * CK, mat);
                tma_load_3d(dst + kRingBytes / 2, &P.mapX[c], full_bar(s, st), CK, kb * CK, mat);
              } else {
                tma_load_3d(dst, &P.mapX[c], full_bar(s, st), kb * CK, 0, mat);
              }
              ring_n[s] = n + 1;
            }
          } else {
            const uint32_t bar = loaded0 + 8 * s;
            mbar_expect_tx(bar, 3 * G::Mat);
            armed[s] = gs;
            for (int kb = 0; kb < G::KB; ++kb) {
              tma_load_3d(base + kb * G::Blk, &P.mapP[c], bar, kb * CK, 0, mat);               // P <- P_0
              tma_load_3d(base + G::Mat + kb * G::Blk, &P.mapA[c], bar, kb * CK, 0, mat);      // A <- A_0
              tma_load_3d(base + 2 * G::Mat + kb * G::Blk, &P.mapP[c], bar, kb * CK, 0, mat);  // Q <- Q_1 = P_0
            }
          }
        }
      }
      if (*abort_flag)  // let the copies armed here land before shared memory goes away
        for (int s = 0; s < S; ++s) {
          if (armed[s] >= 0) (void)mbar_wait(loaded0 + 8 * s, (uint32_t)(armed[s] & 1));
          for (int64_t n = ring_n[s] > kStages ? ring_n[s] - kStages : 0; n < ring_n[s]; ++n)
            (void)mbar_wait(full_bar(s, (int)(n % kStages)), (uint32_t)((n / kStages) & 1));
        }
    }
  } else if (warp == 1 || (kFuse && warp == issuer1)) {
    if constexpr (kMom) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (lane == 0) {
      if constexpr (kFuse) {
        // one MMA issuer per slot: warp 1 takes slot 0, warp issuer1 slot 1
        const int s = warp == 1 ? 0 : 1;
        const uint32_t base = slots + s * G::SlotSize;
        const uint32_t acc = tmem_base + (uint32_t)(s * 256);
        const uint32_t mP = base, mA = base + G::Mat, mQ = base + 2 * G::Mat;
        int64_t ring_c = 0;  // X_0 blocks consumed in this slot
        uint32_t u = 0;      // ops issued in this slot (barrier phases)
        bool issued = false, ok = true;
        for (int64_t g = s; ok && mat_of(g) < total && !*abort_flag; g += S) {
          const int c = chain_class(P, mat_of(g));
          const int kit = (P.p[c] + CK - 1) / CK;
          for (int op = 0; op < P.n_ops && !*abort_flag; ++op) {
            // the slot's previous epilogue has read the accumulators and
            // written the operands
            if (u > 0 && !mbar_wait(epid0 + 8 * s, (u - 1) & 1)) {
              give_up();
              ok = false;
              break;
            }
            tc_fence_after();
            if (op == 0) {
              // the Gram, block by block as X_0 lands.  Wide: K-major rows,
              // a K step 32 bytes along them; tall: K is the stage's rows
              // (16 rows = 2048 bytes a step), its two 64-column halves 8 KB
              // apart
              const int nk = (P.q[c] + CK - 1) / CK;
              const bool tall = P.tall[c] != 0;
              const uint32_t lbo = tall ? kRingBytes / 2 : 16, kstep = tall ? 2048 >> 4 : 32 >> 4;
              const uint32_t idesc = tall ? G::IdescMN : G::IdescK;
              for (int kb = 0; kb < nk; ++kb, ++ring_c) {
                const int st = (int)(ring_c % kStages);
                // the landed block, or (kMom) the operand the momentum pass made of it
                const uint32_t ready = kMom ? cfull_bar(s, st) : full_bar(s, st);
                if (!mbar_wait(ready, (uint32_t)((ring_c / kStages) & 1))) {
                  give_up();
                  ok = false;
                  break;
                }
                tc_fence_after();
                const uint64_t d = smem_desc(base + (uint32_t)(st * kStageBytes), lbo, 1024);
#pragma unroll
                for (int k = 0; k < CK / 16; ++k)
                  chain_mma<kH>(acc, d + k * kstep, d + k * kstep, (kb | k) != 0, idesc);
                mma_commit_one(empty_bar(s, st));
                issued = true;
              }
              if (!ok) break;
            } else {
              const int mma = P.ops[op].mma;
              if (mma == kMmaPA) chain_product<kH>(acc, mP, mA, kit, 0);
              else if (mma == kMmaAA) chain_product<kH>(acc, mA, mA, kit, 0);
              else if (mma == kMmaPQ) chain_product<kH>(acc, mP, mQ, kit, 0);
              else  // kMmaPAQ: acc0 = P A, acc1 = P Q from one N = 256 product over [A | Q]
                chain_product<kH>(acc, mP, mA, kit, 0, G::IdescN2);
            }
            issued = true;
            mma_commit_one(mmad0 + 8 * s);
            ++u;
          }
        }
        if (*abort_flag && issued) {  // the outstanding MMAs complete before TMEM is released
          const uint32_t dr = s == 0 ? drain : drain2;
          mma_commit_one(dr);
          (void)mbar_wait(dr, 0);
        }
      } else {
        int64_t g[S];
        int op[S];
        uint32_t u[S];
        for (int s = 0; s < S; ++s) g[s] = s, op[s] = 0, u[s] = 0;
        bool issued = false;
        for (bool any = true; any && !*abort_flag;) {
          any = false;
          for (int s = 0; s < S && !*abort_flag; ++s) {
            const int64_t t = mat_of(g[s]);
            if (t >= total) continue;
            any = true;
            // the slot's previous epilogue has read its accumulators and
            // written the operands; a new matrix's loads have landed
            if (u[s] > 0 && !mbar_wait(epid0 + 8 * s, (u[s] - 1) & 1)) { give_up(); break; }
            if (op[s] == 0 && !mbar_wait(loaded0 + 8 * s, (uint32_t)((g[s] / S) & 1))) { give_up(); break; }
            tc_fence_after();
            const int kit = (P.p[chain_class(P, t)] + CK - 1) / CK;
            const uint32_t base = slots + s * G::SlotSize;
            const uint32_t mP = base, mA = base + G::Mat, mQ = base + 2 * G::Mat;
            const uint32_t acc = tmem_base + (uint32_t)(s * 256);
            const int mma = P.ops[op[s]].mma;
            for (int h = 0; h < kH; ++h) {
              const uint32_t d = acc + (uint32_t)(h * 256);
              if (mma == kMmaPA) chain_product<kH>(d, mP, mA, kit, h);
              else if (mma == kMmaAA) chain_product<kH>(d, mA, mA, kit, h);
              else if (mma == kMmaPQ) chain_product<kH>(d, mP, mQ, kit, h);
              else  // kMmaPAQ (kH = 1): acc0 = P A, acc1 = P Q from one N = 256 product over [A | Q]
                chain_product<kH>(d, mP, mA, kit, h, G::IdescN2);
            }
            issued = true;
            mma_commit_one(mmad0 + 8 * s);
            ++u[s];
            if (++op[s] == P.n_ops) op[s] = 0, g[s] += S;
          }
        }
        if (*abort_flag && issued) {  // the outstanding MMAs complete before TMEM is released
          mma_commit_one(drain);
          (void)mbar_wait(drain, 0);
        }
      }
    }
  } else if (warp >= kE0 && warp < kE0 + kCEpiWarps) {
    if constexpr (kMom) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    const int quarter = warp & 3;      // TMEM lane quarter of this warp
    const int wh = (warp - kE0) >> 2;  // its column blocks: wh * WarpBlocks ..
    const int cb0 = wh * G::WarpBlocks, cb1 = cb0 + G::WarpBlocks;
    int64_t g[S];
    int op[S];
    uint32_t u[S];
    for (int s = 0; s < S; ++s) g[s] = s, op[s] = 0, u[s] = 0;
    bool stop = false;
    IdleClock idle(clocks + warp);
    for (bool any = true; any && !stop && !*abort_flag;) {
      any = false;
      bool moved = false;
      for (int s = 0; s < S && !stop && !*abort_flag; ++s) {
        const int64_t t = mat_of(g[s]);
        if (t >= total) continue;
        any = true;
        if (kFuse) {
          if (!warp_try(mmad0 + 8 * s, u[s] & 1, lane)) continue;
          // every lane's own acquire of the completed phase (it cannot move
          // on before this warp's arrival, so the wait returns at once)
          (void)mbar_wait(mmad0 + 8 * s, u[s] & 1);
        } else if (!mbar_wait(mmad0 + 8 * s, u[s] & 1)) {
          give_up();
          stop = true;
          break;
        }
        tc_fence_after();
        const int c = chain_class(P, t);
        const ChainOp o = P.ops[op[s]];
        const uint32_t base = slots + s * G::SlotSize;
        const uint32_t mP = base, mA = base + G::Mat, mQ = base + 2 * G::Mat;
        float s2 = 1.f;
        if (kFuse && (o.epi == kEpiGram || o.epi == kEpiGramA)) {
          const int64_t si = P.sub0[c] + (t - P.mat_start[c]);
          float al;
          if constexpr (kMom) {
            // the pre-normalisation factor from the eight warps' statistics,
            // combined in a fixed order (as the momentum kernel's partials
            // are): s = max(max |D|, 1e-7), alpha = 1 / (s (||D / s||_F + 1e-7))
            if (!mbar_wait(momdone0 + 8 * s, (uint32_t)((g[s] / S) & 1))) {
              give_up();
              stop = true;
              break;
            }
            float M = 0.f;
            for (int w = 0; w < kMomWarps; ++w) M = fmaxf(M, mpart[(s * kMomWarps + w) * 2]);
            float ss = 0.f;
            if (M > 0.f) {
              const float inv = 1.0f / M;
              for (int w = 0; w < kMomWarps; ++w) {
                const float r = mpart[(s * kMomWarps + w) * 2] * inv;
                ss = fmaf(mpart[(s * kMomWarps + w) * 2 + 1], r * r, ss);
              }
            }
            const float sc = fmaxf(M, 1e-7f);
            const float norm_y = (M / sc) * sqrtf(ss);
            al = 1.0f / (sc * (norm_y + 1e-7f));
            const bool bad = !isfinite(M) || !isfinite(ss) || !isfinite(al);
            if (bad) al = __int_as_float(0x7fc00000);
            if (warp == kE0 && lane == 0) {
              A.alpha_out[si] = al;
              if (bad) flag_status(A.status, GBO_STATUS_NONFINITE);
              if (A.stats) A.stats[2 * A.subs[si].mat_idx] = M > 0.f ? M * sqrtf(ss) : (isfinite(M) ? 0.f : M);
            }
          } else {
            al = A.alpha[si];
          }
          s2 = al * al;
        }
        chain_epilogue<kH, kFuse>(o, tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(s * 256), quarter, lane,
                           cb0, cb1, P.p[c], s2, mP, mA, mQ);
        // the writes reach the tensor cores' and TMA's proxy; the
        // accumulators have been read
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (o.epi == kEpiOut) {
          // Q_k to HBM once all epilogue warps have written it; the slot is
          // free for its next matrix when the store has read it
          if (lane == 0) mbar_arrive(qdone0 + 8 * s);
          if (warp == kE0) {
            const uint32_t qpar = (uint32_t)((g[s] / S) & 1);
            if (!mbar_wait(qdone0 + 8 * s, qpar)) {
              give_up();
              stop = true;
              break;
            }
            if (lane == 0) {
              const int mat = (int)(t - P.mat_start[c]);
              for (int kb = 0; kb * CK < P.p[c]; ++kb) tma_store_3d(&P.mapQ[c], mQ + kb * G::Blk, kb * CK, 0, mat);
              bulk_commit();
              bulk_wait_read<0>();
              mbar_arrive(freed0 + 8 * s);
            }
            __syncwarp();
          }
        }
        if (lane == 0) mbar_arrive(epid0 + 8 * s);
        moved = true;
        ++u[s];
        if (++op[s] == P.n_ops) op[s] = 0, g[s] += S;
      }
      if (kFuse && any && !stop) {
        int late = 0;
        if (lane == 0) late = idle.expired(moved) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, late, 0)) {
          if (lane == 0) give_up();
          stop = true;
        }
        if (!moved) __nanosleep(32);
      }
    }
    if (lane == 0) bulk_wait_all();  // this warp's stores complete before the kernel ends
    __syncwarp();
  } else if (kMom && warp >= kMomWarp0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsMom));
    // The momentum pass: each landed stage of either slot, in the slot's
    // order, by all eight warps (each its rows); after a matrix's last
    // stage each warp publishes its statistics, before releasing that stage
    // to the MMA issuer, so they are in place by the time the Gram's MMAs
    // (and so its epilogue) complete.
    const int mw = warp - kMomWarp0;
    int64_t g[S];     // the slot's current matrix
    int64_t mrc[S];   // G and B stages consumed in the slot
    int mkb[S];       // stages of the slot's current matrix done
    MomStats mst[S];  // this thread's statistics of the slot's current matrix
    for (int s = 0; s < S; ++s) g[s] = s, mrc[s] = 0, mkb[s] = 0, mst[s] = MomStats{0.f, 0.f, 0.f};
    bool stop = false;
    IdleClock idle(clocks + warp);
    for (bool any = true; any && !stop && !*abort_flag;) {
      any = false;
      bool moved = false;
      // the slot holding the older matrix first, so that it finishes its
      // stream (and starts its chain) while the other slot still streams,
      // rather than the two slots streaming and then chaining in lockstep
      const int first = (S > 1 && g[1] < g[0]) ? 1 : 0;
      for (int k = 0; k < S && !*abort_flag; ++k) {
        const int s = k == 0 ? first : 1 - first;
        const int64_t t = mat_of(g[s]);
        if (t >= total) continue;
        any = true;
        const int cm = chain_class(P, t);
        const int nk = (P.q[cm] + CK - 1) / CK;
        const int64_t n = mrc[s];
        const int st = (int)(n % kStages);
        const uint32_t par = (uint32_t)((n / kStages) & 1);
        if (!warp_try(full_bar(s, st), par, lane)) continue;
        (void)mbar_wait(full_bar(s, st), par);  // every lane's own acquire (completes at once)
        const DevSub &Sd = A.subs[P.sub0[cm] + (t - P.mat_start[cm])];
        MomStats stt = mst[s];
        mom_stage(slots + s * G::SlotSize + st * kStageBytes, Sd, static_cast<__nv_bfloat16 *>(P.x0), mkb[s], mw,
                  lane, A.mu, A.nesterov, stt);
        const bool last = mkb[s] + 1 == nk;
        if (last) {
          const float mx = warp_max(stt.m);
          float sw = 0.f;
          if (mx > 0.f) {
            const float r = stt.m / mx;
            sw = stt.ss * r * r;
          }
          sw = warp_sum(sw);
          if (lane == 0) {
            mpart[(s * kMomWarps + mw) * 2] = mx;
            mpart[(s * kMomWarps + mw) * 2 + 1] = sw;
            mbar_arrive(momdone0 + 8 * s);
          }
          stt = MomStats{0.f, 0.f, 0.f};
        }
        mst[s] = stt;
        fence_async_smem();  // the operand written in place reaches the tensor cores' proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(cfull_bar(s, st));
        mrc[s] = n + 1;
        if (last) mkb[s] = 0, g[s] += S;
        else ++mkb[s];
        moved = true;
        break;  // poll again from the older slot
      }
      if (any) {
        int late = 0;
        if (lane == 0) late = idle.expired(moved) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, late, 0)) {
          if (lane == 0) give_up();
          stop = true;
        }
        if (!moved) __nanosleep(32);
      }
    }
  } else if (kMom) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));  // warp 3: no role
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kCTmemCols)
                 : "memory");
}

// The ops of one matrix's chain for k iterations with coefficients abc
// (3 per iteration): iteration j < k - 1 forms T = P_j A_j (with
// Q_{j+1} = P_j Q_j from j = 1: together when kH = 1, as a second product
// when kH = 2), then A_{j+1} = P_j T and P_{j+1} (through a square of
// A_{j+1} when its c != 0); Q_k = P_{k-1} Q_{k-1} closes the chain.
int chain_ops(int kh, int k, const float *abc, ChainOp *ops) {
  int n = 0;
  for (int j = 0; j + 1 < k; ++j) {
    if (j == 0) {
      ops[n++] = ChainOp{kMmaPA, kEpiT, 0.f, 0.f, 0.f};
    } else if (kh == 1) {
      ops[n++] = ChainOp{kMmaPAQ, kEpiTQ, 0.f, 0.f, 0.f};
    } else {
      ops[n++] = ChainOp{kMmaPA, kEpiT, 0.f, 0.f, 0.f};
      ops[n++] = ChainOp{kMmaPQ, kEpiQ, 0.f, 0.f, 0.f};
    }
    const float *t = abc + 3 * (j + 1);
    if (t[2] != 0.f) {
      ops[n++] = ChainOp{kMmaPA, kEpiA, 0.f, 0.f, 0.f};
      ops[n++] = ChainOp{kMmaAA, kEpiSq, t[0], t[1], t[2]};
    } else {
      ops[n++] = ChainOp{kMmaPA, j + 2 < k ? kEpiAP : kEpiP, t[0], t[1], 0.f};
    }
  }
  ops[n++] = ChainOp{kMmaPQ, kEpiOut, 0.f, 0.f, 0.f};
  return n;
}

// The ops of a chain that starts from X_0 (kFuse): the Gram, with c != 0 the
// square of A_0 that gives P_0, then the chain's own ops.
int fused_ops(int k, const float *abc, ChainOp *ops) {
  int n = 0;
  if (abc[2] != 0.f) {
    ops[n++] = ChainOp{kMmaGram, kEpiGramA, abc[0], abc[1], abc[2]};
    ops[n++] = ChainOp{kMmaAA, kEpiSqQ, abc[0], abc[1], abc[2]};
  } else {
    ops[n++] = ChainOp{kMmaGram, kEpiGram, abc[0], abc[1], 0.f};
  }
  return n + chain_ops(1, k, abc, ops + n);
}

int chain_halves(int p) { return p <= 128 ? 1 : 2; }

template <int kH, bool kFuse, bool kMom>
int launch_geometry(const GemmJob *const *jobs, int32_t n_jobs, const PhaseArgs &args, int sm_count, void *stream,
                    int64_t *n_launch) {
  using G = Geo<kH>;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err =
        cudaFuncSetAttribute(ns_chain_kernel<kH, kFuse, kMom>, cudaFuncAttributeMaxDynamicSharedMemorySize, G::Smem);
    if (kMom && attr_err == cudaSuccess) {
      // setmaxnreg.inc waits until the registers it asks for are free: the
      // warpgroups' shares must fit in what the block is launched with
      cudaFuncAttributes fa;
      attr_err = cudaFuncGetAttributes(&fa, ns_chain_kernel<kH, kFuse, kMom>);
      if (attr_err == cudaSuccess && (int64_t)fa.numRegs * chain_threads<kFuse, kMom>() < kMomRegShares)
        attr_err = cudaErrorInvalidConfiguration;
    }
  });
  if (attr_err != cudaSuccess) return (int)attr_err;
  for (int32_t j0 = 0; j0 < n_jobs; j0 += kMaxClassesPerLaunch) {
    ChainParams T;
    memset(&T, 0, sizeof T);
    T.n = std::min(kMaxClassesPerLaunch, n_jobs - j0);
    const GemmJob &J0 = *jobs[j0];
    if (J0.steps < 2 || J0.steps > GBO_MAX_NS_STEPS || !J0.abc) return (int)cudaErrorInvalidValue;
    T.n_ops = kFuse ? fused_ops(J0.steps, J0.abc, T.ops) : chain_ops(kH, J0.steps, J0.abc, T.ops);
    for (int k = 0; k < T.n; ++k) {
      const GemmJob &J = *jobs[j0 + k];
      const ShapeClass &C = *J.cls;
      const bool gram = J.kind == kKindGram || J.kind == kKindGramT;
      if (chain_halves(C.p) != kH || C.p > G::R || J.steps != J0.steps || J.abc != J0.abc || gram != kFuse ||
          (kFuse && (J.kind == kKindGramT) != (C.x_tall != 0)) || (C.mom_fused != 0) != kMom ||
          (kMom && (C.x_tall || J.opA != J0.opA || !args.gbmaps || !args.alpha_out)))
        return (int)cudaErrorInvalidValue;
      auto at = [&](const void *region) { return static_cast<char *>(const_cast<void *>(region)) + C.p_base * 2; };
      bool ok = encode_map(&T.mapQ[k], at(J.out), C.p, C.p, C.count, C.ldp, CK, G::R);
      if (kMom) {  // X_0 is written, not read: its region base
        T.x0 = const_cast<void *>(J.opA);
      } else if (kFuse) {  // X_0 in x-space: count matrices of p rows (q when tall), row stride ld
        char *x = static_cast<char *>(const_cast<void *>(J.opA)) + C.x_base * 2;
        ok = ok && (C.x_tall ? encode_map(&T.mapX[k], x, C.p, C.q, C.count, C.ld, CK, CK)
                             : encode_map(&T.mapX[k], x, C.q, C.p, C.count, C.ld, CK, 128));
      } else {
        ok = ok && encode_map(&T.mapP[k], at(J.opA), C.p, C.p, C.count, C.ldp, CK, G::R) &&
             encode_map(&T.mapA[k], at(J.opB), C.p, C.p, C.count, C.ldp, CK, G::R);
      }
      if (!ok) return (int)cudaErrorInvalidValue;
      T.p[k] = C.p;
      T.q[k] = C.q;
      T.tall[k] = C.x_tall;
      T.sub0[k] = C.sub0;
      T.mat_start[k + 1] = T.mat_start[k] + C.count;
    }
    const int64_t total = T.mat_start[T.n];
    if (total == 0) continue;
    const unsigned grid = (unsigned)std::min<int64_t>(total, sm_count);  // one CTA per SM
    const cudaError_t err = launch_kernel(ns_chain_kernel<kH, kFuse, kMom>, dim3(grid), dim3(chain_threads<kFuse, kMom>()),
                                          G::Smem, reinterpret_cast<cudaStream_t>(stream), 1, T, args);
    count_launches(1);
    if (n_launch) ++*n_launch;
    if (err != cudaSuccess) return (int)err;
  }
  return 0;
}

}  // namespace

double tc_chain_flops(int p, int k, const float *abc) {
  const int kh = chain_halves(p);
  const int n_cols = kh == 1 ? 128 : 192;
  std::vector<ChainOp> ops(kMaxOps);
  const int n = chain_ops(kh, k, abc, ops.data());
  const double kdim = (double)((p + CK - 1) / CK) * CK;
  double f = 0;
  for (int j = 0; j < n; ++j) f += kh * 2.0 * 128 * (ops[j].mma == kMmaPAQ ? 2 * n_cols : n_cols) * kdim;
  return f;
}

double tc_fused_gram_flops(int p, int q, const float *abc) {
  const double tile = 2.0 * 128 * 128;
  return tile * (double)((q + CK - 1) / CK) * CK + (abc[2] != 0.f ? tile * (double)((p + CK - 1) / CK) * CK : 0.0);
}

static_assert(sizeof(CUtensorMap) == 128, "tensor map size assumed by the plan's G and B map table");

bool encode_gb_maps(void *maps2, const void *g, const float *mom, int64_t rows, int64_t cols, int box_rows) {
  CUtensorMap *m = static_cast<CUtensorMap *>(maps2);
  return encode_map(&m[0], const_cast<void *>(g), cols, rows, 1, cols, CK, (uint32_t)box_rows,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2) &&
         encode_map(&m[1], const_cast<float *>(mom), cols, rows, 1, cols, CK, (uint32_t)box_rows,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4);
}

int chain_geometry(const GemmJob &J) {
  if (J.kind == kKindGram || J.kind == kKindGramT) return J.cls->mom_fused ? kChainFusedMom : kChainFused;
  return chain_halves(J.cls->p) == 1 ? kChainOne : kChainTwo;
}

int launch_ns_chain_tc(const GemmJob *const *jobs, int32_t n_jobs, const PhaseArgs &args, int sm_count,
                       void *stream, int64_t *n_launch) {
  std::vector<const GemmJob *> by[kChainGeometries];
  for (int32_t j = 0; j < n_jobs; ++j) {
    if (jobs[j]->cls->p > kChainMaxP) return (int)cudaErrorInvalidValue;
    by[chain_geometry(*jobs[j])].push_back(jobs[j]);
  }
  // the momentum pass first: it writes the X_0 and factors other launches read
  int err = launch_geometry<1, true, true>(by[kChainFusedMom].data(), (int32_t)by[kChainFusedMom].size(), args,
                                           sm_count, stream, n_launch);
  if (err) return err;
  err = launch_geometry<1, true, false>(by[kChainFused].data(), (int32_t)by[kChainFused].size(), args, sm_count,
                                        stream, n_launch);
  if (err) return err;
  err = launch_geometry<1, false, false>(by[kChainOne].data(), (int32_t)by[kChainOne].size(), args, sm_count,
                                         stream, n_launch);
  if (err) return err;
  return launch_geometry<2, false, false>(by[kChainTwo].data(), (int32_t)by[kChainTwo].size(), args, sm_count,
                                          stream, n_launch);
}

}  // namespace gbo
