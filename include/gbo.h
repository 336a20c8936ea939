/*
 * gbo.h -- C ABI of the GB300 hybrid-optimizer library (libgbo.so).
 *
 * One optimizer step of the hybrid Muon + AdamW recipe on one GPU:
 *   - the Muon path on 2-D projection weights, each stored weight split into
 *     independent matrices by a view ("build_parameter_groups", kimi-k3 docs,
 *     section "Recording independent matrix geometry");
 *   - the elementwise AdamW path with a global-norm clip on the AdamW
 *     gradients only ("Dual-Manifold Optimization in OMN", AdamW paragraph).
 *
 * Conventions for every entry point
 *   - Device pointers point to memory the caller allocated (PyTorch, or
 *     cudaMalloc); the library never frees them.  Host pointers are read
 *     during the call only unless stated otherwise.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and is asynchronous: no entry point synchronises the
 *     host with the device, except gbo_muon_plan_phase_times.
 *   - Return value: GBO_OK (0) or a negative GBO_ERR_* code.  On error
 *     nothing is enqueued and gbo_last_error() returns a message (per host
 *     thread).
 *   - Conditions found on the device (a non-finite norm, a wait that ran out
 *     of time) are OR-ed into an int32 status word in device memory
 *     (`dev_status`, may be NULL).  The library never clears it; the caller
 *     zeroes it when it wants a fresh reading.  Kernels never trap.
 *   - All matrices are row-major.  A stored weight is rows x cols in
 *     PyTorch's out-by-in orientation.
 *   - Every reduction runs in a fixed order: results are bitwise
 *     reproducible run to run on the same device and inputs.
 */
#ifndef GBO_H
#define GBO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GBO_ABI_VERSION 5

/* ---- status codes (return values) ------------------------------------ */
#define GBO_OK 0
#define GBO_ERR_INVALID_ARG (-1) /* NULL or out-of-range argument, misaligned pointer */
#define GBO_ERR_SHAPE (-2)       /* view product / split-sum / size rules broken       */
#define GBO_ERR_CONFLICT (-3)    /* one weight listed twice in a descriptor table      */
#define GBO_ERR_EMPTY (-4)       /* empty descriptor table                             */
#define GBO_ERR_DTYPE (-5)       /* unsupported dtype                                  */
#define GBO_ERR_WORKSPACE (-6)   /* workspace missing, too small or misaligned         */
#define GBO_ERR_CUDA (-7)        /* a CUDA runtime or driver call failed               */
#define GBO_ERR_UNSUPPORTED (-8) /* device or option this build does not handle        */

/* ---- device status bits (OR-ed into *dev_status) ---------------------- */
#define GBO_STATUS_NONFINITE 1 /* a norm or a scale came out NaN or Inf             */
#define GBO_STATUS_TIMEOUT 2   /* a bounded device-side wait gave up; outputs invalid */

/* ---- element types ------------------------------------------------------ */
#define GBO_F32 0
#define GBO_BF16 1

/* ---- Newton-Schulz arithmetic ------------------------------------------ */
#define GBO_NS_BF16 0 /* bf16 operands, fp32 accumulation (tcgen05 tensor cores) */
#define GBO_NS_F32 1  /* fp32 operands (three TF32 products), fp32 accumulation    */

#define GBO_MAX_VIEW_DIMS 6
#define GBO_MAX_NS_STEPS 64

/* cudaStream_t-compatible handle, so this header needs no CUDA header. */
typedef struct CUstream_st *gbo_stream_t;

/* Opaque plan: validated descriptor table, the expansion of every view into
 * independent matrices, their batching by shape, and the device tables. */
typedef struct gbo_plan gbo_plan;

/*
 * One Muon weight.  The view and split rules follow "build_parameter_groups"
 * (kimi-k3 docs), section "Recording independent matrix geometry": every
 * view entry is a positive integer; the product of all view entries but the
 * last equals `rows` and the last equals `cols`.  The view's second-to-last
 * axis `r` is the row count of one block; split sizes (optional) cut each
 * block's rows into consecutive ranges and must sum to `r`.  Each range is
 * one independent matrix (worked shapes on that page: (32,8) viewed
 * (2,16,8) is two 16x8 matrices; (20,8) viewed (2,10,8) split (4,6) is
 * 4x8, 6x8, 4x8, 6x8).
 */
typedef struct {
  void *w;        /* device: weight, rows x cols, w_dtype; updated in place            */
  const void *g;  /* device: gradient, rows x cols, g_dtype; read only.  NULL skips the
                     weight (inactive expert): w, mom, row_v are left untouched       */
  float *mom;     /* device: fp32 momentum buffer rows x cols, updated in place; start it
                     at zero                                                           */
  float *row_v;   /* device: NorMuon row second moment, `rows` fp32 (start at zero), or
                     NULL when NorMuon is off                                          */
  int64_t rows;   /* stored rows (out features), >= 1                                 */
  int64_t cols;   /* stored cols (in features), >= 1                                  */
  int64_t view[GBO_MAX_VIEW_DIMS]; /* first view_ndim entries used                    */
  int32_t w_dtype;   /* GBO_F32 | GBO_BF16                                             */
  int32_t g_dtype;   /* GBO_F32 | GBO_BF16                                             */
  int32_t view_ndim; /* 0: plain rows x cols matrix; else 2..GBO_MAX_VIEW_DIMS         */
  int32_t n_split;   /* 0: no split; else the count of split sizes in the shared pool  */
  int32_t split_off; /* index of this weight's first split size in split_pool          */
  float lr_mult;     /* per-weight learning-rate multiplier (1.0 for the plain recipe) */
  float wd;          /* decoupled weight decay (0.0 in the OMN recipe)                 */
  int32_t reserved;  /* set to 0                                                       */
} gbo_muon_desc;

/*
 * Muon options.  Momentum and Nesterov direction: NorMuon paper (zskr.cn),
 * section 2.2, eq. (1); OMN page, Muon path (coefficient 0.95).  Iterations:
 * eq. (5) of the same section,
 *   X <- a X + b (X X^T) X + c (X X^T)^2 X,
 * whose (a, b, c) = (1.5, -0.5, 0) case is the cubic of the "MuonClip
 * Optimizer" page.  NorMuon rows: NorMuon paper, section 3.1; its
 * RMS-keeping learning-rate scale is read as: with rms_target > 0, each
 * matrix's row-normalised update U becomes rms_target sqrt(m n) U / ||U||_F
 * (no rectangular scale on top; an all-zero U stays zero).
 */
typedef struct {
  const float *abc;      /* host: (a,b,c) triples, 1 triple or ns_steps triples; copied */
  float mu;              /* momentum coefficient, e.g. 0.95                            */
  float beta2;           /* NorMuon second-moment decay (e.g. 0.95)                     */
  float eps;             /* NorMuon epsilon, added outside the square root (1e-8)      */
  int32_t nesterov;      /* 1: D = G + mu*B (after B = mu*B + G); 0: D = B              */
  int32_t ns_steps;      /* number of iterations k, 1..GBO_MAX_NS_STEPS (5)             */
  int32_t abc_per_step;  /* 0: one shared triple; 1: one triple per iteration           */
  int32_t precision;     /* GBO_NS_BF16 | GBO_NS_F32                                    */
  int32_t normuon;       /* 1: NorMuon row normalisation; every desc needs row_v        */
  int32_t route;         /* GBO_ROUTE_AUTO (0) | GBO_ROUTE_X | GBO_ROUTE_GRAM          */
  float rms_target;      /* NorMuon only: > 0 scales each matrix's update to this RMS  */
  int32_t reserved;      /* set to 0                                                    */
  int64_t workspace_cap; /* 0: one schedule over every matrix; > 0: see below           */
} gbo_muon_opts;

/*
 * Workspace cap.  The step's scratch (each matrix's Newton-Schulz iterates and
 * polynomial matrices) grows with the model.  With workspace_cap > 0 the plan
 * splits its descriptor table into groups of consecutive descriptors, each as
 * large as fits the cap, and the step runs the groups one after another on the
 * same workspace: gbo_muon_workspace_bytes is then at most the cap.  Every
 * matrix is computed exactly as without the cap (its reductions and products
 * never involve other matrices), so the results are bitwise the same; the cost
 * is more, smaller launches.  gbo_muon_plan_create fails with
 * GBO_ERR_WORKSPACE when a single descriptor needs more than the cap.
 */

/*
 * Route of the k iterations of one shape class (bf16 mode).  Both give the
 * k-step result of eq. (5); they differ in rounding order and cost.
 *   X     every iteration forms A = X X^T (p x p) and X <- P X (p x q).
 *   GRAM  every iterate is X_j = Q_j X_0 with Q_j a polynomial in
 *         A_0 = X_0 X_0^T, so the iteration runs on p x p matrices only
 *         (A_{j+1} = P_j A_j P_j, Q_{j+1} = P_j Q_j) and the p x q product
 *         runs once: X_k = Q_k X_0.  Executes p^2 q + (3k - 3) p^3 + 2 p^2 q
 *         instead of about k (p^2 q + 2 p^2 q) FLOPs (plus one p x p square
 *         of A per iteration with c != 0, on both routes); needs k >= 2.
 *   AUTO  GRAM where it is allowed and executes at least 10% fewer FLOPs
 *         (q > p), else X.  In bf16 mode the p x p iterations of a matrix of
 *         at most 192 rows run in one on-chip launch, counted as such: those
 *         matrices take GRAM even when square.
 * Both precisions run on the tensor cores: bf16 operands, or in the fp32
 * mode fp32 operands as three TF32 products (hi hi + hi lo + lo hi).
 */
#define GBO_ROUTE_AUTO 0
#define GBO_ROUTE_X 1
#define GBO_ROUTE_GRAM 2

/*
 * Validate a Muon descriptor table and build a plan (host memory only; the
 * device tables are uploaded by the first gbo_muon_step on a device, which
 * should therefore come before any stream capture).
 *   descs[n]            host array; pointers inside are remembered by the plan
 *   split_pool[pool_len] host array of split sizes, indexed by split_off
 *   opts                host; abc is copied
 *   out                 receives the plan; destroy it with gbo_muon_plan_destroy
 * Errors: INVALID_ARG (NULL table/out, missing mom, row_v missing with
 * normuon, bad ns_steps/precision/mu, misaligned pointers), SHAPE (a view
 * or split rule broken, or a matrix side above 2^31-1), CONFLICT (the same w
 * twice), EMPTY (n == 0), DTYPE.
 */
int gbo_muon_plan_create(const gbo_muon_desc *descs, int32_t n, const int64_t *split_pool,
                         int32_t pool_len, const gbo_muon_opts *opts, gbo_plan **out);

/* Release a plan and its device tables.  NULL is accepted. */
void gbo_muon_plan_destroy(gbo_plan *plan);

/* Bytes of device workspace gbo_muon_step needs for this plan (>= 0). */
size_t gbo_muon_workspace_bytes(const gbo_plan *plan);

/*
 * 64-bit FNV-1a hash of what the plan computes: shapes, views, splits,
 * dtypes and options, not pointers.  A checkpoint stores it and a resume
 * with a different layout is refused by comparing it ("build_parameter_groups":
 * names and shapes take part in checkpoint compatibility).  0 for NULL.
 */
uint64_t gbo_desc_hash(const gbo_plan *plan);

/*
 * One Muon step for every weight of the plan whose g is not NULL
 * (OMN page, Muon path order):
 *   B <- mu B + G;  D = G + mu B;
 *   per matrix: X0 = Y / (||Y||_F + 1e-7), Y = D / max(max|D|, 1e-7);
 *               transpose if rows > cols; k iterations of eq. (5); restore;
 *               O scaled by sqrt(max(1, rows/cols)) of that matrix;
 *               (NorMuon) v_i <- beta2 v_i + (1-beta2) mean_j O_ij^2,
 *                         O_ij <- O_ij / (sqrt(v_i) + eps), before the scale;
 *   W <- W - lr*lr_mult*(wd*W + scale*O), rounded once to w_dtype.
 *   lr          the step's learning rate (host scalar)
 *   workspace   device, >= gbo_muon_workspace_bytes(plan) bytes, 256-byte
 *               aligned; contents need no initialisation and are scratch
 *               after the call
 *   dbg_update  device fp32, NULL or sum(rows*cols) over the plan's weights in
 *               table order: receives scale*O (the update before lr) for
 *               every updated weight; untouched for skipped ones
 *   dev_status  device int32 or NULL (GBO_STATUS_* bits OR-ed in)
 * Asynchronous on `stream`.  The first call of a plan sets up its device
 * tables (it allocates and copies, synchronously); later calls only launch
 * kernels, so a later call may be captured into a CUDA graph and replayed.
 * While the stream is being captured, the launches carry the
 * programmatic-dependent-launch attribute (each kernel's prologue overlaps
 * the previous kernel's tail; see gbo_testing_set_pdl).
 * Errors: INVALID_ARG, WORKSPACE, UNSUPPORTED (device is not sm_103),
 * CUDA.
 */
int gbo_muon_step(gbo_plan *plan, float lr, void *workspace, size_t ws_bytes, float *dbg_update,
                  int32_t *dev_status, gbo_stream_t stream);

/*
 * NorMuon row normalisation and weight write for one matrix (NorMuon paper,
 * section 3.1), callable on its own.  O is the unscaled orthogonalised
 * update, fp32 rows x cols row-major (device, read only).  For every row i:
 *   v_i <- beta2 v_i + (1-beta2) * mean_j O_ij^2
 *   U_ij = scale * O_ij / (sqrt(v_i) + eps)
 *   W_ij <- W_ij - lr * (wd * W_ij + U_ij)      (rounded once to w_dtype)
 * row_v: device fp32[rows], updated in place.  dbg_update: NULL or device
 * fp32 rows x cols receiving U.  Errors: INVALID_ARG, DTYPE, CUDA.
 */
int gbo_normuon_rownorm(const float *O, int64_t rows, int64_t cols, float *row_v, void *w,
                        int32_t w_dtype, float beta2, float eps, float scale, float lr, float wd,
                        float *dbg_update, gbo_stream_t stream);

/* ---- AdamW path ---------------------------------------------------------- */

/* One gradient tensor for the clip norm. */
typedef struct {
  const void *ptr; /* device, numel elements of dtype, contiguous */
  int64_t numel;   /* >= 0                                        */
  int32_t dtype;   /* GBO_F32 | GBO_BF16                          */
  int32_t reserved;
} gbo_tensor;

/* Bytes of device scratch gbo_clip_norm needs (a constant of this build). */
size_t gbo_clip_norm_workspace_bytes(void);

/*
 * Global gradient norm over the given (AdamW) gradients and the clip
 * coefficient (OMN page: clipping at 1.0 on AdamW parameters only; the
 * Muon path is never clipped).
 *   N = sqrt(sum of g^2 over all tensors);  coef = N > max_norm ? max_norm/N : 1
 *   dev_total_norm, dev_coef   device fp32 scalars, written (either may be NULL)
 *   workspace                  device scratch, >= gbo_clip_norm_workspace_bytes()
 *                              bytes, 16-byte aligned
 * A non-finite N gives coef = NaN and sets GBO_STATUS_NONFINITE.
 * The gradients are not modified: gbo_adamw_step applies coef.
 * Errors: INVALID_ARG, DTYPE, WORKSPACE, CUDA.  n == 0 writes N = 0, coef = 1.
 */
int gbo_clip_norm(const gbo_tensor *grads, int32_t n, float max_norm, float *dev_total_norm,
                  float *dev_coef, int32_t *dev_status, void *workspace, size_t ws_bytes,
                  gbo_stream_t stream);

/*
 * gbo_clip_norm_noalloc -- the same norm and coefficient as gbo_clip_norm,
 * for callers that cannot allocate device memory.  The source pages have no
 * counterpart: this is an interface for callers, not part of the method.
 *
 * Some callers cannot provide scratch memory: all of the device's memory
 * already belongs to another allocator (a training framework's caching pool
 * that reserved HBM at start-up), or they run where a cudaMalloc, which can
 * synchronise the device, is not allowed.  This entry point allocates
 * nothing: its scratch (1024 fp32 partial sums, 4 KB) is a fixed array in
 * the library's device memory, held by every GPU that loads the library
 * until the process exits.
 *   grads, n, max_norm, dev_total_norm, dev_coef, dev_status: as gbo_clip_norm
 *   n           at most GBO_CLIP_NOALLOC_MAX_TENSORS tensors (any sizes);
 *               more is refused with GBO_ERR_INVALID_ARG
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it for the device's current CUDA context; the
 * first call in a new context (after a device reset, for instance) looks it
 * up again.  Make the first call before any stream capture.  Every
 * call shares the one array, so calls whose work overlaps on the GPU race
 * (use one stream, or order them); it keeps the last call's contents, and no
 * slot needs clearing because each call writes every slot it reads.
 * Errors: INVALID_ARG, DTYPE, UNSUPPORTED, CUDA.
 */
#define GBO_CLIP_NOALLOC_MAX_TENSORS 65536
int gbo_clip_norm_noalloc(const gbo_tensor *grads, int32_t n, float max_norm, float *dev_total_norm,
                          float *dev_coef, int32_t *dev_status, gbo_stream_t stream);

/* One AdamW parameter with its state; all fp32 except g (fp32 or bf16). */
typedef struct {
  float *p;       /* device, numel, updated in place */
  const void *g;  /* device, numel, read only        */
  float *m;       /* device, numel, first moment     */
  float *v;       /* device, numel, second moment    */
  int64_t numel;  /* >= 0                            */
  int32_t g_dtype; /* GBO_F32 | GBO_BF16             */
  int32_t reserved;
} gbo_adamw_desc;

/* AdamW hyper-parameters (OMN page: betas (0.9, 0.95), eps 1e-8, zero decay). */
typedef struct {
  float lr;
  float beta1;
  float beta2;
  float eps;
  float weight_decay;
  int32_t step; /* t >= 1: the step being taken, for bias correction */
  /* NULL, or a device int32 holding t >= 1, read when the kernel runs (then
   * `step` is ignored): a launch captured in a CUDA graph then replays with
   * the current count, which the caller advances on the device. */
  const int32_t *dev_step;
} gbo_adamw_opts;

/*
 * Bias-corrected AdamW with decoupled decay (Qwen3.8 optimizer notes: Adam
 * moments with bias correction, AdamW's decay on the weight), elementwise:
 *   g' = coef * g;  m <- b1 m + (1-b1) g';  v <- b2 v + (1-b2) g'^2
 *   p <- p - lr*wd*p - lr * (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps)
 *   dev_coef  device fp32 scalar (e.g. gbo_clip_norm's output) or NULL for 1
 * descs is a host array read during the call.  Errors: INVALID_ARG, DTYPE,
 * CUDA.
 */
int gbo_adamw_step(const gbo_adamw_desc *descs, int32_t n, const gbo_adamw_opts *opts,
                   const float *dev_coef, int32_t *dev_status, gbo_stream_t stream);

/* ---- host-to-device transfer -------------------------------------------- */

/*
 * gbo_h2d_copy -- copy nbytes from page-locked host memory to device memory
 * with a kernel whose threads load the host memory over the chip-to-chip
 * link, instead of a copy engine.  The source pages have no counterpart:
 * this moves a step's inputs (the gradients) onto the device.
 *
 * On a GB300 host both routes move ~200 GB/s, but copy-engine uploads of a
 * few GB stall now and then for tens to hundreds of milliseconds; this
 * kernel's did not.  It runs `blocks` blocks of 1024 threads (0: one per
 * SM), each holding a whole SM to itself: a block reserves more than half
 * of an SM's shared memory, so no SM runs two of them or one beside a
 * Newton-Schulz CTA.  To overlap the copy with a step, leave that many SMs
 * free in the step's plan (gbo_muon_plan_set_free_sms).  Measured on a
 * GB300: a block moves ~50 GB/s alone (four: ~200 GB/s, the link's rate),
 * ~27 GB/s beside a step's GEMMs.
 *   dst     device memory, 16-byte aligned, nbytes writable
 *   src     page-locked host memory mapped for the device (cudaHostRegister,
 *           cudaMallocHost, or pinned tensors), 16-byte aligned; the
 *           first and last byte are checked
 *   nbytes  >= 0; any size (the last nbytes % 16 are copied bytewise)
 *   blocks  >= 0
 * Asynchronous on `stream`, like cudaMemcpyAsync: src must stay valid and
 * unchanged, and dst unread, until the stream reaches the copy.  The caller
 * owns both buffers.  Errors: INVALID_ARG (NULL, misaligned, negative size
 * or blocks, src not page-locked and mapped, dst not device memory), CUDA.
 */
int gbo_h2d_copy(void *dst, const void *src, int64_t nbytes, int32_t blocks, gbo_stream_t stream);

/* ---- diagnostics ---------------------------------------------------------- */

/* Message for the last non-zero return on this host thread ("" if none). */
const char *gbo_last_error(void);

/* GBO_ABI_VERSION of the built library. */
int32_t gbo_abi_version(void);

/* sizeof of an ABI struct, for binding checks: 0 gbo_muon_desc,
 * 1 gbo_muon_opts, 2 gbo_tensor, 3 gbo_adamw_desc, 4 gbo_adamw_opts,
 * 5 gbo_plan_info; 0 for other values. */
size_t gbo_struct_size(int32_t which);

/* Number of kernels this library has launched in this process. */
uint64_t gbo_launch_count(void);

/* What a plan holds, for reporting. */
typedef struct {
  int64_t n_weights;       /* descriptors in the table                          */
  int64_t n_active;        /* descriptors with a gradient                       */
  int64_t n_matrices;      /* independent matrices of the active weights        */
  int64_t n_shape_classes; /* distinct oriented (p, q) shapes                   */
  int64_t muon_params;     /* elements of the active weights                    */
  double ns_flops;         /* dense-count Newton-Schulz FLOPs per step          */
  double ns_flops_executed;/* FLOPs the kernels execute (same unless symmetric) */
  int64_t launches_per_step; /* kernels one gbo_muon_step launches              */
  int64_t n_gram_route;    /* matrices whose iterations take the Gram route     */
  int64_t n_mom_fused;     /* matrices whose momentum pass runs inside the
                              Newton-Schulz chain launch (wide, at most 128
                              rows, bf16 G on 16-byte rows)                     */
} gbo_plan_info;

int gbo_muon_plan_info(const gbo_plan *plan, gbo_plan_info *out);

/*
 * Executed Newton-Schulz FLOPs per step of every descriptor of the plan (the
 * sum over its matrices; 0 for a descriptor whose g is NULL), in table
 * order: the cost a static partition of whole matrices over devices
 * balances (Qwen3.8-Flash-Next optimizer notes, distributed Muon: the
 * partitioner assigns complete matrices by estimated NS FLOPs; NorMuon
 * paper, section 3.2: each parameter has one owner that orthogonalises
 * it).  flops: host array of n doubles, n = the plan's descriptor count.
 * Errors: INVALID_ARG.
 */
int gbo_muon_plan_desc_flops(const gbo_plan *plan, double *flops, int32_t n);

/*
 * Phase timing.  When enabled, gbo_muon_step records CUDA events around its
 * phases on its stream.  gbo_muon_plan_phase_times synchronises on the last
 * recorded event, adds the elapsed milliseconds of every step since the last
 * reset into ms[phase] and the number of kernel launches into
 * launches[phase], then resets.  Phases: 0 momentum (+ the norm reduction;
 * the momentum pass of n_mom_fused matrices runs in the chain launch, timed
 * under phase 2), 1 Newton-Schulz Gram products, 2 Newton-Schulz products back onto X
 * except the one that writes the weights, 3 Gram squares (c != 0), 4 NorMuon
 * rows and weight write, 5 the last product with the weight write (no
 * NorMuon).  n_phases is the array length (<= GBO_N_PHASES).
 */
#define GBO_N_PHASES 6

/*
 * Per-matrix norms, for monitoring a run (the OMN page's matched comparison
 * tracks gradient and update norms).  After the call, every later
 * gbo_muon_step writes two floats per matrix of the plan's active weights,
 * in table order (a weight's matrices in view order): stats[2 j] = ||D_j||_F,
 * the Frobenius norm of the momentum direction the matrix is orthogonalised
 * from (before the pre-normalisation), and stats[2 j + 1] = ||U_j||_F, the
 * norm of the update direction the weight moves along (scale * O, row-
 * normalised with NorMuon; the weight moves by lr * lr_mult * U).  The
 * sums are taken in a fixed order from the reductions the step already
 * runs: the pre-normalisation's, and per-row partial sums of squares the
 * last product (or the NorMuon rows pass) leaves in the workspace; a
 * non-finite norm is written as such.  dev_stats: device fp32, 2 *
 * gbo_plan_info.n_matrices values; NULL stops.  Errors: INVALID_ARG.
 */
int gbo_muon_plan_set_stats(gbo_plan *plan, float *dev_stats);

/*
 * Record `event` (a cudaEvent_t, created by the caller) on the step's stream
 * right after phase `phase` of every later gbo_muon_step, or stop doing so
 * when `event` is NULL.  Phase numbers as above; the phase-0 event is
 * recorded once the momentum buffers are updated and the gradients are no
 * longer read (after the chain launch that runs the momentum pass of the
 * n_mom_fused matrices, when there are any), so work on
 * another stream that waits on the event (the AdamW path, the next
 * gradients) overlaps the Newton-Schulz GEMMs.  Errors: INVALID_ARG.
 */
int gbo_muon_plan_set_event(gbo_plan *plan, int32_t phase, void *event);
/*
 * Leave n SMs free of the persistent Newton-Schulz kernels in every later
 * gbo_muon_step: the CTA-pair kernel then runs at most (SMs - n) / 2 pairs,
 * the single-CTA and chain kernels at most SMs - n CTAs, so that work on
 * another stream that needs whole SMs (gbo_h2d_copy with n blocks) runs
 * beside the step.  The results do not change (each output element sums
 * the same products in the same order); the GEMMs lose about n / SMs of
 * their rate.  0 <= n <= 64; default 0.  Errors: INVALID_ARG.
 */
int gbo_muon_plan_set_free_sms(gbo_plan *plan, int32_t n);
int gbo_muon_plan_set_timing(gbo_plan *plan, int32_t enable);
int gbo_muon_plan_phase_times(gbo_plan *plan, float *ms, int64_t *launches, int32_t n_phases);

#ifdef __cplusplus
}
#endif

#endif /* GBO_H */
