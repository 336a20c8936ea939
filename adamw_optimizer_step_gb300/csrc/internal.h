// Internal declarations shared by the host plan code and the CUDA kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include "gbo.h"

namespace gbo {

constexpr int kMomTile = 64;        // momentum tiles: 64 x 64 elements of a matrix, or
constexpr int kMomFlat = kMomTile * kMomTile;  // 4096 consecutive elements of a matrix
constexpr int kRowBlock = 64;       // NorMuon: stored rows per block
constexpr int kMaxClassesPerLaunch = 8;
constexpr int kMaxFreeSms = 64;  // gbo_muon_plan_set_free_sms

// One independent matrix (a view block or split range of a stored weight),
// as the kernels see it.  Orientation: the stored matrix is m x n; the
// Newton-Schulz side is p x q with p = min(m, n); `transposed` is set when
// m > n, in which case X holds D^T.
struct DevSub {
  void *w;
  const void *g;
  float *mom;
  float *row_v;
  int64_t r0;       // first stored row of this matrix in its weight
  int64_t cols;     // row stride of the weight (== n)
  int64_t x_off;    // element offset of this matrix in each X buffer
  int64_t xt_off;   // element offset of this matrix in each XT buffer (fp32 mode: X transposed)
  int64_t p_off;    // element offset of this matrix in the P (and A) buffer
  int64_t dbg_off;  // element offset of the weight's first element in dbg_update
  int64_t tile0;    // first momentum tile of this matrix (global tile index)
  int64_t rb0;      // first NorMuon row block of this matrix
  int64_t ss_off;   // NorMuon (bf16 mode): first of this matrix's m x ss_ntn row-statistics partials
  int32_t m, n;     // stored rows, cols
  int32_t p, q;     // oriented rows, cols
  int32_t ld;       // X row stride (elements)
  int32_t ldt;      // XT row stride (elements), fp32 mode
  int32_t has_xt;   // the momentum pass also writes X0 transposed (fp32 mode)
  int32_t ldp;      // P row stride (elements)
  int32_t tiles_c;  // momentum tiles along n (2-D tiles), or 0 for flat tiles
  int32_t ntiles;   // momentum tiles of this matrix
  int32_t transposed;  // X holds D^T (fp32 mode: tall matrices)
  int32_t w_dtype, g_dtype;
  int32_t vec_ok;   // g and mom rows start on 16-byte boundaries (n % 8 == 0)
  int32_t cls;
  float scale;      // sqrt(max(1, m / n))
  float lr_mult;
  float wd;
  int32_t w_vec;    // weight rows start on 16-byte boundaries (vector read-modify-write)
  int32_t x_sel;    // X buffer (0 or 1) that holds the last iterate (NorMuon rows read it)
  int32_t wmap;     // index of the weight's TMA map (bf16 weights with 16-byte rows), or -1
  int32_t ss_ntn;   // NorMuon (bf16 mode): partials per stored row, one per 128 output columns
  int32_t mom_fused; // the momentum pass of this matrix runs inside the chain kernel (no momentum tiles)
  int32_t gbmap;     // with mom_fused: index of its pair of G and B TMA maps (2 * gbmap, 2 * gbmap + 1)
  int32_t desc;      // the descriptor (stored weight) this matrix belongs to
  int32_t mat_idx;   // its place among the plan's matrices in table order (per-matrix statistics)
};

// Matrices of one oriented shape (p, q), stored back to back in the
// workspace so one 3-D TMA map covers all of them.
//
// Two routes to the same k-step result (bf16 mode):
//   kRouteX     every iteration forms A = X X^T and X <- P X on the p x q
//               iterate;
//   kRouteGram  the iteration runs on p x p matrices only.  Every iterate is
//               X_j = Q_j X_0 with Q_j a polynomial in A_0 = X_0 X_0^T, so
//               A_{j+1} = P_j A_j P_j and Q_{j+1} = P_j Q_j are products of
//               commuting symmetric matrices (upper triangle only), and the
//               p x q product runs once, X_k = Q_k X_0.  Cheaper whenever
//               q > p.  With c != 0, P_j = a I + b A_j + c A_j^2 takes one
//               more symmetric product, the square of A_j.
struct ShapeClass {
  int32_t p, q, ld, ldp;
  int32_t count;  // matrices in the class
  int32_t sub0;   // index of the first matrix in the DevSub table
  int32_t route;  // kRouteX | kRouteGram
  int32_t tall;   // the stored matrix has more rows than columns (m > n)
  int32_t x_tall; // bf16 mode: X holds a tall matrix in stored orientation, q x p
  int32_t ldt;    // fp32 mode: row stride of XT, X's transposed twin (q x p)
  int32_t mom_fused; // the chain kernel streams G and B and runs the momentum pass of these matrices
  int64_t xt_base; // element offset of the class in each XT buffer
  int64_t x_base; // element offset of the class in each X buffer
  int64_t p_base; // element offset of the class in its p x p buffers (its route's space)
};

enum NsRoute : int32_t { kRouteX = 0, kRouteGram = 1 };

// Epilogue selector of the Newton-Schulz GEMMs.
enum GemmMode : int32_t {
  kGram = 0,      // C = X X^T;  write P = a I + b s^2 C          (c == 0)
  kGramA = 1,     // C = X X^T;  write A = s^2 C                   (c != 0)
  kSquare = 2,    // C = A A;    write P = a I + b A + c C
  kProduct = 3,   // C = P X;    write X' = s C
  kFinal = 4,     // C = P X;    O = s C; update the weight (+ dbg)
  kGramAP = 5,    // C symmetric; write A = s^2 C and P = a I + b A
  kChain = 6,     // the Gram route's p x p chain on chip (p <= kChainMaxP): A_0, P_0 -> Q_k
};

// Operand shapes of one tensor-core GEMM job.  X is p x q ("wide") or, for
// a matrix stored with more rows than columns, q x p in stored orientation
// ("tall"); the tall kinds are the transposes of the wide ones, so no
// matrix is ever transposed in memory on the tensor-core path.
enum GemmKind : int32_t {
  kKindGram = 0,   // C = X X^T, X wide: A and B operands are rows of X (K = q); symmetric output
  kKindSym = 1,    // C = L R, L and R symmetric p x p and commuting: symmetric output
  kKindProd = 2,   // C = L X, X wide: B = X with K along its rows (MN-major); p x q output
  kKindGramT = 3,  // C = X^T X, X tall: A and B are columns of X (both MN-major, K = q); symmetric output
  kKindProdT = 4,  // C = X L, X tall: A = rows of X (K = p), B = rows of L; q x p output
  kKindProdK = 5,  // C = L X, X wide, from its transposed twin XT (q x p): B = rows of XT; p x q output
};

// Products have full outputs; the other kinds a symmetric p x p output.
__host__ __device__ inline bool is_product_kind(int kind) {
  return kind == kKindProd || kind == kKindProdT || kind == kKindProdK;
}

// Rows and columns of a job's output for matrix S.
__host__ __device__ inline int kind_rows(int kind, int p, int q) { return kind == kKindProdT ? q : p; }
__host__ __device__ inline int kind_cols(int kind, int p, int q) {
  return (kind == kKindProd || kind == kKindProdK) ? q : p;
}

// One shape class of a tensor-core launch and what it computes.  Operand
// and output pointers are region bases; the launcher adds the class base
// (x-space for X operands, the class's p x p space otherwise) and the
// epilogue adds each matrix's offset.
struct GemmJob {
  const ShapeClass *cls;
  int32_t mode;   // GemmMode of the epilogue
  int32_t kind;   // GemmKind
  int32_t first;  // fold the pre-normalisation factor (s = alpha)
  float a, b, c;
  const void *opA, *opB;
  void *out, *out2;  // out: P, A, T, Q or X'; out2: A of kGramAP
  const void *aux;   // kSquare: the A matrix read by the epilogue; kProduct: NorMuon
                     // row-statistics partials (fp32) when this is the last product
  int32_t steps;     // kChain: iterations k and their coefficients (3 per iteration)
  const float *abc;
};

// Per-step arguments every Newton-Schulz launch shares (the per-class work
// is in its GemmJob).
struct PhaseArgs {
  float lr;
  const void *wmaps;  // device array of the weights' TMA maps (CUtensorMap), see build_weight_maps
  const DevSub *subs;
  const float *alpha; // per matrix pre-normalisation factor
  float *dbg;         // dbg_update or nullptr
  int32_t *status;
  const void *gbmaps; // device array of G and B TMA maps (CUtensorMap) of the matrices with mom_fused
  float *alpha_out;   // the same factors, written by the chain kernel for its matrices with mom_fused
  float mu;           // momentum coefficient and Nesterov flag, for the chain kernel's momentum pass
  int32_t nesterov;
  float *stats;       // per-matrix norms (||D||_F, ||U||_F) at 2 * mat_idx, or nullptr
};

// Launchers (implemented in the .cu files).  Each returns a cudaError_t as
// int and adds its launches to the library's counter.
// x0t: X0's transposed twin (fp32 mode), or nullptr.
// stream_g: 0, or (every matrix with flat tiles, bf16 X) the element size of
// G when all G are bf16 (2) or else 4: the tiles then stream through shared
// memory by bulk copies (momentum_stream_kernel), with bitwise the same
// results.  status: where a timed-out wait is flagged.
int launch_momentum(const DevSub *subs, int32_t n_subs, int64_t n_tiles, float mu, int32_t nesterov,
                    void *x0, void *x0t, int32_t x_dtype, float *partials, int32_t stream_g, int32_t *status,
                    int sm_count, void *stream);
// Whether momentum_stream_kernel may run where the table allows it (on by
// default); returns the previous setting (gbo_testing_set_momentum_stream).
int32_t set_momentum_stream(int32_t enable);
// stats: nullptr, or where each matrix's ||D||_F goes (2 * mat_idx)
int launch_prenorm_finalize(const DevSub *subs, int32_t n_subs, const float *partials,
                            float *alpha, int32_t *status, float *stats, int sm_count, void *stream);
// Per-matrix ||U||_F into stats[2 * mat_idx + 1]: from the last product's
// per-(row, 128 columns) sums of U^2 (rowss), or with NorMuon from the rows
// kernels' per-row-block sums of (1 / (sqrt(v) + eps))^2 ||X_i||^2 (rowpart).
int launch_stats_finalize(const DevSub *subs, int32_t n_subs, int32_t normuon, float rms_target,
                          const float *rowss, const float *rowpart, float *stats, void *stream);
// NorMuon rows; with rms_target > 0 a statistics pass, the per-matrix
// RMS-keeping scale and a write pass (rowf: n_row_blocks * kRowBlock floats,
// rowpart: n_row_blocks, mscale: n_subs), else one fused pass.
// rowss: the last product's per-(row, 128 columns) sums of squares of
// X_k (bf16 mode), or nullptr to take the statistics from X_k itself.
// streamed: every matrix has bf16 X and bf16 weight rows on 16-byte
// boundaries, so the write pass streams rows through shared memory.
// stats: the single pass also leaves per-row-block sums of
// (1 / (sqrt(v) + eps))^2 ||X_i||^2 in rowpart (the two-pass modes do anyway).
int launch_normuon_rows(const DevSub *subs, int32_t n_subs, int64_t n_row_blocks, const void *x0,
                        const void *x1, int32_t x_dtype, float beta2, float eps, float lr, float *dbg,
                        int32_t *status, float rms_target, float *rowf, float *rowpart, float *mscale,
                        const float *rowss, bool streamed, bool stats, int sm_count, void *stream);
int launch_normuon_rownorm_plain(const float *O, int64_t rows, int64_t cols, float *row_v, void *w,
                                 int32_t w_dtype, float beta2, float eps, float scale, float lr,
                                 float wd, float *dbg, void *stream);
int launch_clip_norm(const gbo_tensor *grads, int32_t n, float max_norm, float *total, float *coef,
                     int32_t *status, float *partials, int sm_count, void *stream);
int launch_adamw(const gbo_adamw_desc *descs, int32_t n, const gbo_adamw_opts *opts,
                 const float *coef, int32_t *status, int sm_count, void *stream);

// tcgen05 path: one Newton-Schulz step over a set of jobs (any mix of
// classes and kinds).  `globals` supplies subs, alpha, lr, dbg and status.
// Adds the number of kernel launches made to *n_launch.  The bf16 kernel,
// and the fp32 one (three TF32 products, K-major operands only: the Gram,
// symmetric and ProdK / ProdT kinds).
int launch_ns_gemm_tc(const GemmJob *jobs, int32_t n_jobs, const PhaseArgs &globals, int sm_count,
                      void *stream, int64_t *n_launch);
int launch_ns_gemm_tf32(const GemmJob *jobs, int32_t n_jobs, const PhaseArgs &globals, int sm_count,
                        void *stream, int64_t *n_launch);
// kChain jobs (bf16, p <= kChainMaxP): opA = P_0, opB = A_0, out = Q_k
// regions; or, for a wide class of p <= 128 (kind kKindGram), opA = X_0:
// the Gram runs on chip too; and when the class has mom_fused, the kernel
// streams G and B instead, runs the momentum pass, writes X_0 to opA and
// the pre-normalisation factors to globals.alpha_out.  Every job of one
// call has the same steps and abc.
constexpr int kChainMaxP = 192;
int launch_ns_chain_tc(const GemmJob *const *jobs, int32_t n_jobs, const PhaseArgs &globals, int sm_count,
                       void *stream, int64_t *n_launch);
// The chain kernel's launch groups: the Gram on chip (p <= 128, wide),
// p <= 128, 128 < p <= kChainMaxP, the momentum pass and the Gram on chip
// (p <= 128, wide, bf16 G).
enum ChainGeometry : int32_t { kChainFused = 0, kChainOne = 1, kChainTwo = 2, kChainFusedMom = 3 };
constexpr int kChainGeometries = 4;
// G and B TMA maps of one weight for matrices of `rows` rows: 2-D over the
// weight's rows x cols, boxes of 64 columns x rows (bf16 G, fp32 B), no
// swizzle.  Returns false if the driver refuses them.
bool encode_gb_maps(void *maps2, const void *g, const float *mom, int64_t rows, int64_t cols, int box_rows);
int chain_geometry(const GemmJob &J);
// FLOPs of the on-chip Gram of one p x q matrix: a 128 x 128 tile, K = q
// padded to 64, and with c_0 != 0 the square of A_0 (K = p padded to 64).
double tc_fused_gram_flops(int p, int q, const float *abc);
// FLOPs the chain kernel executes for one p x p matrix (p <= kChainMaxP)
// over k iterations with coefficients abc: 128 x 128 (or x 256) tiles for
// p <= 128, two 128 x 192 row halves for larger p, K padded to 64.
double tc_chain_flops(int p, int k, const float *abc);
// FLOPs the tensor-core kernel executes for one p x q matrix and one
// iteration (Gram over the upper block-triangle of tiles, square when c != 0,
// product), counting the zero padding of partial tiles; `tall`: X is held
// q x p and the product runs transposed; `final`: the product is the
// weight-writing last one (see single_job).
double tc_executed_flops(int p, int q, bool square, bool tall, bool final);
// FLOPs executed for one p x q matrix over k iterations on the Gram route:
// the Gram, 3k - 3 symmetric p x p products plus one square of A for each
// of `squares` iterations with c != 0, the product with X_0.
double tc_gram_route_flops(int p, int q, int k, int squares, bool tall, bool final);
// The same when the p x p chain runs on chip: the Gram (and the square of
// A_0 when c_0 != 0) on the tile kernel or, `fused`, on chip, the chain,
// the product with X_0.
double tc_gram_chain_flops(int p, int q, int k, const float *abc, bool tall, bool fused, bool final);
// Whether the tensor-core kernel runs a shape class of p oriented rows on
// single CTAs (p <= 128) rather than on CTA pairs.
bool single_mode(int p);
// Whether a job of that class in epilogue mode `mode` runs on single CTAs:
// single_mode(p), or the weight-writing last product (kFinal) of a class of
// at most 256 rows.
bool single_job(int p, int32_t mode);
// The bf16 pair kernel's tail split on (1, the default) or off; returns the
// previous setting (gbo_testing_set_tail_split).
int32_t set_tail_split(int32_t enable);
// How many CTA pairs of the bf16 Newton-Schulz kernel fit on the current
// device at once (gbo_testing_pair_residency); -1 on a CUDA error.
int32_t pair_residency();
// One 3-D TMA map (columns, rows, 1) per descriptor for the last product's
// weight stores: 32 x 32 boxes, 64-byte swizzle, for bf16 weights whose rows
// start on 16-byte boundaries (others zero, and their matrices carry wmap =
// -1).  *out receives a device array the caller frees with cudaFree.
int build_weight_maps(const gbo_muon_desc *descs, int32_t n, void **out);
// Testing: the GEMM's bounded mbarrier wait on a barrier nothing arrives on.
int launch_wait_timeout(int32_t *status, uint64_t limit_ns, void *stream);

void count_launches(uint64_t n);
// Whether a launch on `stream` carries the programmatic-dependent-launch
// attribute (gbo_testing_set_pdl; by default only while the stream is being
// captured into a CUDA graph).
int32_t pdl_enabled(void *stream);

// Error and device helpers of the host code, for entry points that live in
// other files: record a message for gbo_last_error, clear it, and check
// that the current device is an sm_103 part (returns its SM count).
int report_error(int code, const char *msg);
int report_ok();
int require_device(int *dev, int *sm_count);

constexpr int kClipBlocks = 1024;  // partial sums of the clip norm

}  // namespace gbo
