// Host side of the library: descriptor validation, expansion of views into
// independent matrices, batching by oriented shape, workspace layout, the
// device tables, and the extern "C" entry points declared in gbo.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <cstdlib>
#include <tuple>
#include <mutex>
#include <string>
#include <utility>
#include <vector>
#include <atomic>

#include "gbo.h"
#include "gbo_testing.h"
#include "internal.h"

namespace gbo {

static std::atomic<uint64_t> g_launches{0};
static std::atomic<int32_t> g_small_chain{1};  // see gbo_testing_set_small_chain
static std::atomic<int32_t> g_fused_gram{1};   // see gbo_testing_set_fused_gram
static std::atomic<int32_t> g_fused_mom{0};    // see gbo_testing_set_fused_momentum (off: measured slower)
void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
// see gbo_testing_set_pdl: 2 (the default) in CUDA graph capture only
static std::atomic<int32_t> g_pdl{2};
int32_t pdl_enabled(void *stream) {
  const int32_t mode = g_pdl.load(std::memory_order_relaxed);
  if (mode != 2) return mode;
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &st) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return st == cudaStreamCaptureStatusActive ? 1 : 0;
}

namespace {

thread_local std::string t_last_error;

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

int ok() {
  t_last_error.clear();
  return GBO_OK;
}

int cuda_fail(int err, const char *what) {
  return fail(GBO_ERR_CUDA, "%s: %s", what, cudaGetErrorString((cudaError_t)err));
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t dtype_size(int32_t dt) { return dt == GBO_BF16 ? 2 : 4; }

bool valid_dtype(int32_t dt) { return dt == GBO_F32 || dt == GBO_BF16; }

// FNV-1a, 64 bit.
struct Fnv {
  uint64_t h = 1469598103934665603ull;
  void bytes(const void *p, size_t n) {
    const unsigned char *c = static_cast<const unsigned char *>(p);
    for (size_t i = 0; i < n; ++i) {
      h ^= c[i];
      h *= 1099511628211ull;
    }
  }
  template <typename T>
  void put(T v) { bytes(&v, sizeof v); }
};

// Per-device facts, looked up once.
struct DeviceInfo {
  int sm_count = 0;
  int major = 0, minor = 0;
  bool known = false;
};
std::mutex g_dev_mu;
std::map<int, DeviceInfo> g_devs;

int current_device(int *dev, DeviceInfo *info) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo &d = g_devs[*dev];
  if (!d.known) {
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, *dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, *dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, *dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.known = true;
  }
  *info = d;
  if (!(d.major == 10 && d.minor == 3))
    return fail(GBO_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only",
                *dev, d.major, d.minor);
  return GBO_OK;
}

constexpr int kPhaseMomentum = 0, kPhaseGram = 1, kPhaseProduct = 2, kPhaseSquare = 3,
              kPhaseRows = 4, kPhaseFinal = 5;

}  // namespace

int report_error(int code, const char *msg) { return fail(code, "%s", msg); }

int report_ok() { return ok(); }

int require_device(int *dev, int *sm_count) {
  DeviceInfo di;
  const int rc = current_device(dev, &di);
  if (rc == GBO_OK) *sm_count = di.sm_count;
  return rc;
}

}  // namespace gbo

using namespace gbo;

struct gbo_plan {
  std::vector<gbo_muon_desc> descs;
  std::vector<int64_t> pool;
  gbo_muon_opts opts{};
  std::vector<float> abc;  // 3 * ns_steps
  bool any_c = false;
  bool any_gram = false;     // some class takes the Gram route
  bool small_chain = true;   // Gram-route classes with p <= kChainMaxP run the on-chip chain (bf16)
  bool fused_gram = true;    // ... and those of p <= 128 held wide start it from X_0
  bool fused_mom = false;    // ... and those with bf16 G on 16-byte rows run their momentum pass there too
  bool any_mom_fused = false;
  int64_t n_unfused = 0;     // matrices whose momentum pass is the momentum kernel's
  // (descriptor, rows) of every G and B TMA map pair the fused momentum pass uses
  std::vector<std::pair<int32_t, int32_t>> gb_pairs;
  std::vector<DevSub> subs;  // sorted by shape class
  std::vector<ShapeClass> classes;
  int64_t n_tiles = 0, n_row_blocks = 0;
  // the momentum tiles stream through shared memory (every matrix with flat
  // tiles, bf16 X): G's element size, 2 when all G are bf16, else 4; or 0
  int32_t mom_stream_g = 0;
  int32_t x_dtype = GBO_BF16;
  size_t off_x[2] = {0, 0}, off_p = 0, off_a = 0, off_alpha = 0, off_part = 0, ws_bytes = 0;
  size_t off_xt[2] = {0, 0};  // fp32 mode: the X buffers' transposed twins
  // Gram-route p x p buffers: A, T, P (two), Q (two)
  size_t off_g[6] = {0, 0, 0, 0, 0, 0};
  // NorMuon RMS-keeping scale: per-row factors, row-block partials, per-matrix scales
  size_t off_rowf = 0, off_rowpart = 0, off_mscale = 0;
  // NorMuon, bf16 mode: the last product's row-statistics partials, and
  // whether every matrix's weight rows allow the streamed write pass
  size_t off_rowss = 0;
  bool rows_streamed = false;
  uint64_t hash = 0;
  gbo_plan_info info{};
  std::vector<double> class_flops;  // executed Newton-Schulz FLOPs of one matrix of each class
  // device state, set by the first step
  int device = -1;
  int sm_count = 0;
  DevSub *d_subs = nullptr;
  void *d_wmaps = nullptr;  // the weights' TMA maps (bf16 mode)
  void *d_gbmaps = nullptr; // the G and B TMA maps of the fused momentum pass
  // phase timing
  bool timing = false;
  struct Interval {
    cudaEvent_t a, b;
    int phase;
    int64_t launches;
  };
  std::vector<Interval> pending;
  std::vector<cudaEvent_t> event_pool;
  cudaEvent_t after_phase[8] = {};  // caller events recorded after a phase
  // workspace cap: plans of consecutive descriptor groups, stepped in turn on
  // one workspace (this plan keeps the whole table's layout for its info,
  // hash and per-descriptor FLOPs, but runs nothing itself)
  std::vector<gbo_plan *> kids;
  int64_t dbg_base = 0;  // a group's first element in the whole table's dbg_update
  int64_t mat_base = 0;  // a group's first matrix among the whole table's
  float *stats = nullptr;  // per-matrix norms (gbo_muon_plan_set_stats), or nullptr
  int32_t free_sms = 0;     // SMs the Newton-Schulz kernels leave free (gbo_muon_plan_set_free_sms)
};

namespace {

// Iterations whose polynomial has c != 0 (each costs a square of A).
int squares(const gbo_plan *P) {
  int n = 0;
  for (int it = 0; it < P->opts.ns_steps; ++it) n += P->abc[3 * it + 2] != 0.f;
  return n;
}

// Gram-route classes of at most kChainMaxP rows run their p x p iterations
// in the on-chip chain kernel (bf16 mode).
bool uses_chain(const gbo_plan *P, const ShapeClass &C) {
  return P->small_chain && P->x_dtype == GBO_BF16 && C.route == kRouteGram && C.p <= kChainMaxP &&
         P->opts.ns_steps >= 2;
}

// Of those, the classes of at most 128 rows run their Gram in the chain
// kernel too, streaming X_0 through the shared memory of the matrix.
bool fuses_gram(const gbo_plan *P, int p) { return P->fused_gram && p <= 128; }
bool fuses_gram(const gbo_plan *P, const ShapeClass &C) { return uses_chain(P, C) && fuses_gram(P, C.p); }

// Route of a p x q class: the Gram route needs k >= 2; AUTO takes it when it
// executes at least 10% fewer FLOPs, counting the on-chip chain where the
// class would run it (in practice: whenever q is clearly above p, and for
// every matrix of at most kChainMaxP rows in bf16 mode, where the chain also
// replaces 2k launches by three).
int32_t choose_route(const gbo_plan *P, int p, int q, bool tall) {
  const int k = P->opts.ns_steps;
  if (k < 2 || P->opts.route == GBO_ROUTE_X) return kRouteX;
  if (P->opts.route == GBO_ROUTE_GRAM) return kRouteGram;
  const bool x_tall = P->x_dtype == GBO_BF16 && tall;
  const bool fin = !P->opts.normuon;  // the last product writes the weights (NorMuon: X, for the rows pass)
  double fx = 0;
  for (int it = 0; it < k; ++it) fx += tc_executed_flops(p, q, P->abc[3 * it + 2] != 0.f, x_tall, fin && it == k - 1);
  const bool chain = P->small_chain && P->x_dtype == GBO_BF16 && p <= kChainMaxP;
  const double fg = chain ? tc_gram_chain_flops(p, q, k, P->abc.data(), x_tall, fuses_gram(P, p), fin)
                          : tc_gram_route_flops(p, q, k, squares(P), x_tall, fin);
  return fg < 0.9 * fx ? kRouteGram : kRouteX;
}

int validate_and_expand(gbo_plan *P) {
  const gbo_muon_opts &o = P->opts;
  const int32_t n = (int32_t)P->descs.size();
  std::map<const void *, int32_t> seen;
  struct Pending {
    DevSub s;
    int32_t order;
  };
  std::vector<DevSub> subs;
  // classes: (p, q, tall), tall = more rows than columns.  The bf16 path keeps
  // a tall matrix's X in stored orientation (q x p); the fp32 path holds X =
  // D^T (p x q) and a transposed twin XT (q x p) of every X
  using ClassKey = std::tuple<int32_t, int32_t, int32_t>;
  std::map<ClassKey, int32_t> class_of;
  std::vector<ClassKey> class_shapes;
  const bool tc_path = P->x_dtype == GBO_BF16;
  int64_t dbg_off = 0;
  for (int32_t t = 0; t < n; ++t) {
    const gbo_muon_desc &d = P->descs[t];
    if (!d.w) return fail(GBO_ERR_INVALID_ARG, "desc %d: w is NULL", t);
    if (!valid_dtype(d.w_dtype) || !valid_dtype(d.g_dtype))
      return fail(GBO_ERR_DTYPE, "desc %d: dtype must be GBO_F32 or GBO_BF16", t);
    if (d.rows <= 0 || d.cols <= 0)
      return fail(GBO_ERR_SHAPE, "desc %d: stored shape %lld x %lld must be positive", t,
                  (long long)d.rows, (long long)d.cols);
    if (d.rows > INT32_MAX || d.cols > INT32_MAX)
      return fail(GBO_ERR_SHAPE, "desc %d: a side above 2^31-1", t);
    if (!aligned(d.w, dtype_size(d.w_dtype)) || (d.g && !aligned(d.g, dtype_size(d.g_dtype))) ||
        (d.mom && !aligned(d.mom, 4)) || (d.row_v && !aligned(d.row_v, 4)))
      return fail(GBO_ERR_INVALID_ARG, "desc %d: pointer not aligned to its element size", t);
    if (seen.count(d.w))
      return fail(GBO_ERR_CONFLICT, "desc %d: weight %p already listed as desc %d", t, d.w, seen[d.w]);
    seen[d.w] = t;
    // view rules
    int64_t view[GBO_MAX_VIEW_DIMS];
    int nd = d.view_ndim;
    if (nd == 0) {
      nd = 2;
      view[0] = d.rows;
      view[1] = d.cols;
    } else {
      if (nd < 2 || nd > GBO_MAX_VIEW_DIMS)
        return fail(GBO_ERR_SHAPE, "desc %d: view_ndim %d outside 2..%d", t, nd, GBO_MAX_VIEW_DIMS);
      int64_t lead = 1;
      for (int k = 0; k < nd; ++k) {
        view[k] = d.view[k];
        if (view[k] <= 0) return fail(GBO_ERR_SHAPE, "desc %d: view entry %d is not positive", t, k);
        if (k < nd - 1) {
          if (lead > d.rows / view[k] + 1) return fail(GBO_ERR_SHAPE, "desc %d: view product overflows", t);
          lead *= view[k];
        }
      }
      if (lead != d.rows || view[nd - 1] != d.cols)
        return fail(GBO_ERR_SHAPE,
                    "desc %d: flattened view leading axes give %lld x %lld, stored %lld x %lld", t,
                    (long long)lead, (long long)view[nd - 1], (long long)d.rows, (long long)d.cols);
    }
    const int64_t r = view[nd - 2];
    std::vector<int64_t> split;
    if (d.n_split < 0) return fail(GBO_ERR_SHAPE, "desc %d: negative n_split", t);
    if (d.n_split > 0) {
      if (!P->pool.size() || d.split_off < 0 || (int64_t)d.split_off + d.n_split > (int64_t)P->pool.size())
        return fail(GBO_ERR_INVALID_ARG, "desc %d: split sizes outside the split pool", t);
      int64_t sum = 0;
      for (int k = 0; k < d.n_split; ++k) {
        const int64_t s = P->pool[d.split_off + k];
        if (s <= 0) return fail(GBO_ERR_SHAPE, "desc %d: split size %d is not positive", t, k);
        sum += s;
        split.push_back(s);
      }
      if (sum != r)
        return fail(GBO_ERR_SHAPE, "desc %d: split sizes sum to %lld, view row axis is %lld", t,
                    (long long)sum, (long long)r);
    } else {
      split.push_back(r);
    }
    const int64_t this_dbg = dbg_off;
    dbg_off += d.rows * d.cols;
    if (!d.g) continue;  // skipped this step: inactive
    if (!d.mom) return fail(GBO_ERR_INVALID_ARG, "desc %d: mom is NULL", t);
    if (o.normuon && !d.row_v) return fail(GBO_ERR_INVALID_ARG, "desc %d: NorMuon needs row_v", t);
    // momentum kernel: eight elements per 16-byte (bf16) or 2 x 16-byte (fp32) access
    const bool vec_rows = (d.cols % 8 == 0) && aligned(d.g, 16) && aligned(d.mom, 16);
    const int64_t blocks = d.rows / r;
    for (int64_t b = 0; b < blocks; ++b) {
      int64_t start = b * r;
      for (int64_t s : split) {
        DevSub S{};
        S.w = d.w;
        S.g = d.g;
        S.mom = d.mom;
        S.row_v = d.row_v;
        S.r0 = start;
        S.cols = d.cols;
        S.m = (int32_t)s;
        S.n = (int32_t)d.cols;
        S.transposed = !tc_path && S.m > S.n;
        S.has_xt = !tc_path;
        S.p = std::min(S.m, S.n);
        S.q = std::max(S.m, S.n);
        S.w_dtype = d.w_dtype;
        S.g_dtype = d.g_dtype;
        S.vec_ok = vec_rows;
        S.w_vec = ((d.cols * (int64_t)dtype_size(d.w_dtype)) % 16 == 0) && aligned(d.w, 16);
        // the last product stores bf16 weights through a TMA map of the weight
        S.wmap = (P->x_dtype == GBO_BF16 && d.w_dtype == GBO_BF16 && S.w_vec) ? t : -1;
        S.scale = (float)std::sqrt(std::max(1.0, (double)S.m / (double)S.n));
        S.lr_mult = d.lr_mult;
        S.wd = d.wd;
        S.dbg_off = this_dbg;
        S.gbmap = t;  // the descriptor, until the fused momentum pass's maps are numbered
        S.desc = t;
        S.mat_idx = (int32_t)subs.size();  // table order: the matrices are pushed in it
        const ClassKey key(S.p, S.q, S.m > S.n ? 1 : 0);
        auto it = class_of.find(key);
        if (it == class_of.end()) {
          it = class_of.emplace(key, (int32_t)class_shapes.size()).first;
          class_shapes.push_back(key);
        }
        S.cls = it->second;
        subs.push_back(S);
        start += s;
      }
    }
  }
  // Route of each class; X-route classes first, so the second X buffer only
  // spans them when nothing else needs it.
  std::vector<int32_t> route(class_shapes.size());
  for (size_t c = 0; c < class_shapes.size(); ++c)
    route[c] = choose_route(P, std::get<0>(class_shapes[c]), std::get<1>(class_shapes[c]),
                            std::get<2>(class_shapes[c]) != 0);
  std::vector<int32_t> order;
  for (int r : {(int)kRouteX, (int)kRouteGram})
    for (size_t c = 0; c < class_shapes.size(); ++c)
      if (route[c] == r) order.push_back((int32_t)c);
  std::vector<int32_t> new_index(class_shapes.size());
  for (size_t k = 0; k < order.size(); ++k) new_index[order[k]] = (int32_t)k;
  for (DevSub &S : subs) S.cls = new_index[S.cls];
  // order by class (stable: table order within a class)
  std::stable_sort(subs.begin(), subs.end(), [](const DevSub &a, const DevSub &b) { return a.cls < b.cls; });
  const size_t es = P->x_dtype == GBO_BF16 ? 2 : 4;
  // classes whose every matrix can stream G and B through the chain kernel:
  // bf16 G, and G and B rows on 16-byte boundaries (the TMA maps' strides)
  std::vector<char> mom_ok(class_shapes.size(), 1);
  for (const DevSub &S : subs)
    if (S.g_dtype != GBO_BF16 || !S.vec_ok) mom_ok[S.cls] = 0;
  P->classes.clear();
  P->any_gram = false;
  P->any_mom_fused = false;
  P->gb_pairs.clear();
  std::map<std::pair<int32_t, int32_t>, int32_t> gb_index;
  int64_t xoff = 0, xtoff = 0, poff = 0, goff = 0, x_route_end = 0;
  for (size_t c = 0; c < order.size(); ++c) {
    ShapeClass C{};
    C.p = std::get<0>(class_shapes[order[c]]);
    C.q = std::get<1>(class_shapes[order[c]]);
    C.tall = std::get<2>(class_shapes[order[c]]);
    C.x_tall = tc_path && C.tall;
    C.route = route[order[c]];
    const int32_t xrows = C.x_tall ? C.q : C.p;  // X is p x q, or q x p when held tall
    C.ld = (int32_t)round_up(C.x_tall ? C.p : C.q, 16);
    C.ldt = tc_path ? 0 : (int32_t)round_up(C.p, 16);  // XT: q x p
    C.ldp = (int32_t)round_up(C.p, 16);
    C.count = 0;
    C.sub0 = -1;
    C.x_base = xoff;
    C.xt_base = xtoff;
    // p x p buffers: the X route's P (and A) space, or the Gram route's own space
    int64_t &pspace = C.route == kRouteGram ? goff : poff;
    C.p_base = pspace;
    // the momentum pass in the chain kernel: wide classes whose Gram runs on chip
    C.mom_fused = (P->fused_mom && tc_path && !C.x_tall && fuses_gram(P, C) && mom_ok[c]) ? 1 : 0;
    P->any_mom_fused = P->any_mom_fused || C.mom_fused;
    for (size_t k = 0; k < subs.size(); ++k)
      if (subs[k].cls == (int32_t)c) {
        if (C.sub0 < 0) C.sub0 = (int32_t)k;
        DevSub &S = subs[k];
        S.ld = C.ld;
        S.ldt = C.ldt;
        S.ldp = C.ldp;
        S.x_off = xoff + (int64_t)C.count * xrows * C.ld;
        S.xt_off = xtoff + (int64_t)C.count * C.q * C.ldt;
        S.p_off = pspace + (int64_t)C.count * C.p * C.ldp;
        // the last iterate: X_k of the X route alternates buffers from X0;
        // the Gram route writes X_k = Q_k X_0 into the second buffer
        S.x_sel = C.route == kRouteGram ? 1 : (o.ns_steps & 1);
        S.mom_fused = C.mom_fused;
        if (C.mom_fused) {  // one G and B map pair per (descriptor, rows)
          const std::pair<int32_t, int32_t> key(S.gbmap, S.m);
          auto it = gb_index.find(key);
          if (it == gb_index.end()) {
            it = gb_index.emplace(key, (int32_t)P->gb_pairs.size()).first;
            P->gb_pairs.push_back(key);
          }
          S.gbmap = it->second;
        } else {
          S.gbmap = -1;
        }
        C.count++;
      }
    xoff = round_up(xoff + (int64_t)C.count * xrows * C.ld, 128);
    xtoff = round_up(xtoff + (int64_t)C.count * C.q * C.ldt, 128);
    pspace = round_up(pspace + (int64_t)C.count * C.p * C.ldp, 128);
    if (C.route == kRouteX) x_route_end = xoff;
    else P->any_gram = true;
    P->classes.push_back(C);
  }
  // momentum tiles and NorMuon row blocks, in table order of subs
  int64_t tiles = 0, rbs = 0;
  P->n_unfused = 0;
  for (DevSub &S : subs) {
    if (S.mom_fused) {  // no momentum tiles: the chain kernel runs its momentum pass
      S.tiles_c = 0;
      S.ntiles = 0;
      S.tile0 = tiles;
      S.rb0 = rbs;
      rbs += (S.m + kRowBlock - 1) / kRowBlock;
      continue;
    }
    P->n_unfused++;
    // A matrix that is not transposed is one contiguous block of its weight
    // (views split rows only), and so is its X when ld == n: its momentum
    // tiles are flat runs of 4096 elements.  Tall matrices use 64 x 64 tiles
    // transposed through shared memory.
    const bool flat = !S.transposed && !S.has_xt && S.vec_ok && S.ld == S.n;
    S.tiles_c = flat ? 0 : (S.n + kMomTile - 1) / kMomTile;
    S.ntiles = flat ? (int32_t)(((int64_t)S.m * S.n + kMomFlat - 1) / kMomFlat)
                    : ((S.m + kMomTile - 1) / kMomTile) * S.tiles_c;
    S.tile0 = tiles;
    tiles += S.ntiles;
    S.rb0 = rbs;
    rbs += (S.m + kRowBlock - 1) / kRowBlock;
  }
  P->n_tiles = tiles;
  P->n_row_blocks = rbs;
  bool all_flat = P->x_dtype == GBO_BF16, all_g16 = true;
  for (const DevSub &S : subs)
    if (!S.mom_fused) {
      all_flat = all_flat && S.tiles_c == 0;
      all_g16 = all_g16 && S.g_dtype == GBO_BF16;
    }
  P->mom_stream_g = all_flat ? (all_g16 ? 2 : 4) : 0;
  // NorMuon row statistics from the last product (bf16 mode): per stored row
  // of each matrix, one partial per 128 columns of its output
  // and, for the per-matrix norms, the last product's sums of squares of
  // the update in any mode (one float per stored row and 128 columns)
  int64_t rowss = 0;
  P->rows_streamed = o.normuon && tc_path;
  for (DevSub &S : subs) {
    P->rows_streamed = P->rows_streamed && S.w_dtype == GBO_BF16 && S.w_vec && !S.transposed && S.n % 8 == 0;
    S.ss_ntn = (S.n + 127) / 128;
    S.ss_off = rowss;
    rowss += (int64_t)S.m * S.ss_ntn;
  }
  P->subs = std::move(subs);
  // workspace layout
  size_t off = 0;
  auto region = [&](size_t bytes) {
    const size_t at = off;
    off = (size_t)round_up((int64_t)(off + bytes), 256);
    return at;
  };
  P->off_x[0] = region((size_t)xoff * es);
  // the Gram route writes its last iterate into the second buffer only for NorMuon
  P->off_x[1] = region((size_t)(o.normuon ? xoff : x_route_end) * es);
  // fp32 mode: XT twins of both X buffers (the second one for the X route's
  // products and the NorMuon last iterate)
  P->off_xt[0] = region((size_t)xtoff * es);
  P->off_xt[1] = region((size_t)xtoff * es);
  P->off_p = region((size_t)poff * es);
  P->off_a = region(P->any_c ? (size_t)poff * es : 0);
  for (int b = 0; b < 6; ++b) P->off_g[b] = region((size_t)goff * es);
  P->off_alpha = region(P->subs.size() * sizeof(float));
  P->off_part = region((size_t)tiles * 8 * 2 * sizeof(float));  // (max, sum of squares) per warp of a tile
  const bool rms = o.normuon && o.rms_target > 0.f;
  // per-row factors: the RMS scale's statistics pass, or the streamed write
  // pass's statistics pass
  const bool rowf = rms || P->rows_streamed;
  P->off_rowf = region(rowf ? (size_t)rbs * kRowBlock * sizeof(float) : 0);
  P->off_rowpart = region(o.normuon ? (size_t)rbs * sizeof(float) : 0);
  P->off_mscale = region(rms ? P->subs.size() * sizeof(float) : 0);
  P->off_rowss = region((size_t)rowss * sizeof(float));
  P->ws_bytes = off;
  // info
  gbo_plan_info &I = P->info;
  I.n_weights = n;
  I.n_active = 0;
  for (const auto &d : P->descs)
    if (d.g) I.n_active++, I.muon_params += d.rows * d.cols;
  I.n_matrices = (int64_t)P->subs.size();
  I.n_shape_classes = (int64_t)P->classes.size();
  double fl = 0;
  for (const DevSub &S : P->subs) {
    const double p = S.p, q = S.q;
    for (int it = 0; it < o.ns_steps; ++it)
      fl += 4.0 * p * p * q + (P->abc[3 * it + 2] != 0.f ? 2.0 * p * p * p : 0.0);
  }
  I.ns_flops = fl;
  I.n_gram_route = 0;
  I.n_mom_fused = 0;
  for (const DevSub &S : P->subs) I.n_mom_fused += S.mom_fused;
  {
    // the tile FLOPs of one pass (the fp32 kernel runs each as three TF32 products)
    double ex = 0;
    P->class_flops.assign(P->classes.size(), 0.0);
    for (size_t k = 0; k < P->classes.size(); ++k) {
      const ShapeClass &C = P->classes[k];
      double per = 0;  // one matrix of the class
      const bool fin = !o.normuon;  // the last product writes the weights
      if (C.route == kRouteGram) {
        per = uses_chain(P, C) ? tc_gram_chain_flops(C.p, C.q, o.ns_steps, P->abc.data(), C.x_tall != 0,
                                                     fuses_gram(P, C), fin)
                               : tc_gram_route_flops(C.p, C.q, o.ns_steps, squares(P), C.x_tall != 0, fin);
        I.n_gram_route += C.count;
      } else {
        for (int it = 0; it < o.ns_steps; ++it)
          per += tc_executed_flops(C.p, C.q, P->abc[3 * it + 2] != 0.f, C.x_tall != 0, fin && it == o.ns_steps - 1);
      }
      P->class_flops[k] = per;
      ex += C.count * per;
    }
    I.ns_flops_executed = ex;
  }
  return GBO_OK;
}

uint64_t layout_hash(const gbo_plan *P) {
  Fnv f;
  f.put<int32_t>((int32_t)P->descs.size());
  for (const auto &d : P->descs) {
    f.put(d.rows);
    f.put(d.cols);
    f.put(d.w_dtype);
    f.put(d.view_ndim);
    for (int k = 0; k < d.view_ndim; ++k) f.put(d.view[k]);
    f.put(d.n_split);
    for (int k = 0; k < d.n_split; ++k) f.put(P->pool[d.split_off + k]);
  }
  f.put(P->opts.normuon);
  return f.h;
}

// One tensor-core step of the schedule: the jobs of every class that has
// work at this point, and the phase it is timed under.
struct TcStep {
  std::vector<GemmJob> jobs;
  int phase = kPhaseGram;
};

// The tensor-core schedule of one Muon step (bf16 mode).  The X route takes
// 2k steps (3 per iteration when c != 0), the Gram route 2k + 1, or with the
// on-chip chain three: the Gram (and the square of A_0 when c_0 != 0), the
// chain, the last product.  A chain that runs its own Gram takes the chain's
// step, so every class's last product shares a step.  Step i of the step
// runs step i of both routes, whose classes and buffers are disjoint; steps
// left empty are dropped.  With ws == nullptr the pointers are offsets (for
// counting).
std::vector<TcStep> build_schedule(const gbo_plan *P, char *ws) {
  const int k = P->opts.ns_steps;
  const bool normuon = P->opts.normuon != 0;
  auto R = [ws](size_t off) { return reinterpret_cast<void *>(reinterpret_cast<uintptr_t>(ws) + off); };
  void *x[2] = {R(P->off_x[0]), R(P->off_x[1])};
  void *pb = R(P->off_p), *ab = R(P->off_a);
  void *gA = R(P->off_g[0]), *gT = R(P->off_g[1]);
  void *gP[2] = {R(P->off_g[2]), R(P->off_g[3])};
  void *gQ[2] = {R(P->off_g[4]), R(P->off_g[5])};
  void *xt[2] = {R(P->off_xt[0]), R(P->off_xt[1])};
  const bool f32 = P->x_dtype == GBO_F32;
  // the NorMuon last product's row-statistics partials (bf16 mode), and the
  // weight-writing last product's sums of squares of the update when the
  // per-matrix norms are asked for
  void *rowss = (normuon && !f32) ? R(P->off_rowss) : nullptr;
  void *uss = P->stats ? R(P->off_rowss) : nullptr;
  auto last_product = [&](GemmJob J) {
    if (J.mode == kProduct) J.aux = rowss;
    else if (J.mode == kFinal) J.aux = uss;
    return J;
  };
  auto job = [](const ShapeClass *C, int mode, int kind, int first, const float *abc, const void *opA,
                const void *opB, void *out, void *out2 = nullptr, const void *aux = nullptr) {
    GemmJob J{};
    J.cls = C;
    J.mode = mode;
    J.kind = kind;
    J.first = first;
    J.a = abc ? abc[0] : 0.f;
    J.b = abc ? abc[1] : 0.f;
    J.c = abc ? abc[2] : 0.f;
    J.opA = opA;
    J.opB = opB;
    J.out = out;
    J.out2 = out2;
    J.aux = aux;
    return J;
  };
  std::vector<TcStep> xs, gs;
  auto at = [](std::vector<TcStep> &v, size_t i, int phase) -> TcStep & {
    if (v.size() <= i) v.resize(i + 1);
    v[i].phase = phase;
    return v[i];
  };
  for (const ShapeClass &C : P->classes) {
    if (C.count == 0) continue;
    const int kGramK = C.x_tall ? kKindGramT : kKindGram;  // X X^T, or X^T X of an X held tall
    // the product with X = x[cur] into x[cur ^ 1]:
    //   bf16   L X, or X L of an X held tall (then weights in stored orientation)
    //   fp32   L X with B from X's twin XT, writing X' and X'T; the weight write
    //          of a tall matrix takes XT L, which is in stored orientation
    auto product = [&](int mode, int first, const float *abc, const void *L, int cur) {
      if (!f32)
        return C.x_tall ? job(&C, mode, kKindProdT, first, abc, x[cur], L, x[cur ^ 1])
                        : job(&C, mode, kKindProd, first, abc, L, x[cur], x[cur ^ 1]);
      if (mode == kFinal && C.tall) return job(&C, mode, kKindProdT, first, abc, xt[cur], L, nullptr);
      return job(&C, mode, kKindProdK, first, abc, L, xt[cur], x[cur ^ 1], xt[cur ^ 1]);
    };
    if (C.route == kRouteX) {
      size_t i = 0;
      int cur = 0;
      for (int it = 0; it < k; ++it) {
        const float *abc = &P->abc[3 * it];
        const int first = it == 0;
        if (abc[2] != 0.f) {
          at(xs, i++, kPhaseGram).jobs.push_back(job(&C, kGramA, kGramK, first, abc, x[cur], x[cur], ab));
          at(xs, i++, kPhaseSquare).jobs.push_back(job(&C, kSquare, kKindSym, 0, abc, ab, ab, pb, nullptr, ab));
        } else {
          at(xs, i++, kPhaseGram).jobs.push_back(job(&C, kGram, kGramK, first, abc, x[cur], x[cur], pb));
        }
        const bool last = it == k - 1;
        const int mode = (last && !normuon) ? kFinal : kProduct;
        const GemmJob pj = product(mode, first, abc, pb, cur);
        at(xs, i++, mode == kFinal ? kPhaseFinal : kPhaseProduct).jobs.push_back(last ? last_product(pj) : pj);
        cur ^= 1;
      }
    } else {
      // A_0 = alpha^2 X_0 X_0^T and P_0;  Q_1 = P_0.  An iteration with c != 0
      // writes A only and takes P = a I + b A + c A^2 from a square of A.
      size_t i = 0;
      if (fuses_gram(P, C)) {
        // the Gram, the square of A_0 and every p x p product in one
        // on-chip launch, in the step where the other classes' chains run
        // (so that all last products share one step)
        GemmJob J = job(&C, kChain, kGramK, 1, &P->abc[0], x[0], x[0], gQ[k & 1]);
        J.steps = k;
        J.abc = P->abc.data();
        i = P->abc[2] != 0.f ? 2 : 1;
        at(gs, i++, kPhaseProduct).jobs.push_back(J);
        const int mode = normuon ? kProduct : kFinal;
        at(gs, i++, mode == kFinal ? kPhaseFinal : kPhaseProduct)
            .jobs.push_back(last_product(product(mode, 1, nullptr, gQ[k & 1], 0)));
        continue;
      }
      if (P->abc[2] == 0.f) {
        at(gs, i++, kPhaseGram).jobs.push_back(job(&C, kGramAP, kGramK, 1, &P->abc[0], x[0], x[0], gP[0], gA));
      } else {
        at(gs, i++, kPhaseGram).jobs.push_back(job(&C, kGramA, kGramK, 1, &P->abc[0], x[0], x[0], gA));
        at(gs, i++, kPhaseSquare).jobs.push_back(job(&C, kSquare, kKindSym, 0, &P->abc[0], gA, gA, gP[0], nullptr, gA));
      }
      if (uses_chain(P, C)) {  // every p x p product of the iterations in one on-chip launch
        GemmJob J = job(&C, kChain, kKindSym, 0, nullptr, gP[0], gA, gQ[k & 1]);
        J.steps = k;
        J.abc = P->abc.data();
        at(gs, i++, kPhaseProduct).jobs.push_back(J);
        const int mode = normuon ? kProduct : kFinal;
        at(gs, i++, mode == kFinal ? kPhaseFinal : kPhaseProduct)
            .jobs.push_back(last_product(product(mode, 1, nullptr, gQ[k & 1], 0)));
        continue;
      }
      for (int j = 0; j + 1 < k; ++j) {
        void *Pj = gP[j & 1];
        // T = P_j A_j and, from j = 1, Q_{j+1} = P_j Q_j
        TcStep &la = at(gs, i++, kPhaseProduct);
        la.jobs.push_back(job(&C, kGramA, kKindSym, 0, nullptr, Pj, gA, gT));
        if (j >= 1) la.jobs.push_back(job(&C, kGramA, kKindSym, 0, nullptr, Pj, j == 1 ? gP[0] : gQ[j & 1], gQ[(j + 1) & 1]));
        // A_{j+1} = P_j T and P_{j+1} (with c == 0, A_{k-1} itself is not needed)
        const float *abc = &P->abc[3 * (j + 1)];
        void *Pn = gP[(j + 1) & 1];
        if (abc[2] != 0.f) {
          at(gs, i++, kPhaseGram).jobs.push_back(job(&C, kGramA, kKindSym, 0, abc, Pj, gT, gA));
          at(gs, i++, kPhaseSquare).jobs.push_back(job(&C, kSquare, kKindSym, 0, abc, gA, gA, Pn, nullptr, gA));
        } else if (j + 2 < k) {
          at(gs, i++, kPhaseGram).jobs.push_back(job(&C, kGramAP, kKindSym, 0, abc, Pj, gT, Pn, gA));
        } else {
          at(gs, i++, kPhaseGram).jobs.push_back(job(&C, kGram, kKindSym, 0, abc, Pj, gT, Pn));
        }
      }
      // Q_k = P_{k-1} Q_{k-1}, then X_k = Q_k X_0 (alpha folded in)
      at(gs, i++, kPhaseProduct)
          .jobs.push_back(job(&C, kGramA, kKindSym, 0, nullptr, gP[(k - 1) & 1], k == 2 ? gP[0] : gQ[(k - 1) & 1],
                              gQ[k & 1]));
      const int mode = normuon ? kProduct : kFinal;
      at(gs, i++, mode == kFinal ? kPhaseFinal : kPhaseProduct)
          .jobs.push_back(last_product(product(mode, 1, nullptr, gQ[k & 1], 0)));
    }
  }
  std::vector<TcStep> steps;
  for (size_t i = 0; i < std::max(xs.size(), gs.size()); ++i) {
    TcStep st;
    if (i < gs.size()) {
      st.phase = gs[i].phase;
      st.jobs = gs[i].jobs;
    }
    if (i < xs.size()) {  // label by the X route where it has a step
      st.phase = xs[i].phase;
      st.jobs.insert(st.jobs.end(), xs[i].jobs.begin(), xs[i].jobs.end());
    }
    if (!st.jobs.empty()) steps.push_back(st);  // steps the on-chip Gram left empty
  }
  return steps;
}

// Kernel launches of one step of the schedule (classes go 8 to a launch,
// pairs and single CTAs separately).
int64_t tc_step_launches(const TcStep &st) {
  int64_t single = 0, pair = 0, chain[kChainGeometries] = {};
  for (const GemmJob &J : st.jobs) {
    if (J.mode == kChain) ++chain[chain_geometry(J)];
    else (single_job(J.cls->p, J.mode) ? single : pair)++;
  }
  auto groups = [](int64_t n) { return (n + kMaxClassesPerLaunch - 1) / kMaxClassesPerLaunch; };
  int64_t n = groups(single) + groups(pair);
  for (int g = 0; g < kChainGeometries; ++g) n += groups(chain[g]);
  return n;
}

cudaEvent_t take_event(gbo_plan *P) {
  if (!P->event_pool.empty()) {
    cudaEvent_t e = P->event_pool.back();
    P->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

}  // namespace

extern "C" {

const char *gbo_last_error(void) { return t_last_error.c_str(); }

int32_t gbo_abi_version(void) { return GBO_ABI_VERSION; }

size_t gbo_struct_size(int32_t which) {
  switch (which) {
    case 0: return sizeof(gbo_muon_desc);
    case 1: return sizeof(gbo_muon_opts);
    case 2: return sizeof(gbo_tensor);
    case 3: return sizeof(gbo_adamw_desc);
    case 4: return sizeof(gbo_adamw_opts);
    case 5: return sizeof(gbo_plan_info);
    default: return 0;
  }
}

uint64_t gbo_launch_count(void) { return g_launches.load(); }

}  // extern "C"

namespace {

int make_plan(const gbo_muon_desc *descs, int32_t n, const int64_t *split_pool, int32_t pool_len,
              const gbo_muon_opts *opts, gbo_plan **out) {
  if (!out) return fail(GBO_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!opts) return fail(GBO_ERR_INVALID_ARG, "opts is NULL");
  if (n < 0) return fail(GBO_ERR_INVALID_ARG, "negative descriptor count");
  if (n == 0) return fail(GBO_ERR_EMPTY, "empty descriptor table: nothing to optimise");
  if (!descs) return fail(GBO_ERR_INVALID_ARG, "descs is NULL");
  if (pool_len < 0 || (pool_len > 0 && !split_pool)) return fail(GBO_ERR_INVALID_ARG, "bad split pool");
  if (opts->ns_steps < 1 || opts->ns_steps > GBO_MAX_NS_STEPS)
    return fail(GBO_ERR_INVALID_ARG, "ns_steps %d outside 1..%d", opts->ns_steps, GBO_MAX_NS_STEPS);
  if (!opts->abc) return fail(GBO_ERR_INVALID_ARG, "abc is NULL");
  if (opts->precision != GBO_NS_BF16 && opts->precision != GBO_NS_F32)
    return fail(GBO_ERR_INVALID_ARG, "precision must be GBO_NS_BF16 or GBO_NS_F32");
  if (opts->route != GBO_ROUTE_AUTO && opts->route != GBO_ROUTE_X && opts->route != GBO_ROUTE_GRAM)
    return fail(GBO_ERR_INVALID_ARG, "route must be GBO_ROUTE_AUTO, GBO_ROUTE_X or GBO_ROUTE_GRAM");
  if (!std::isfinite(opts->mu)) return fail(GBO_ERR_INVALID_ARG, "mu is not finite");
  if (opts->normuon && (!(opts->beta2 >= 0.f && opts->beta2 <= 1.f) || !(opts->eps >= 0.f)))
    return fail(GBO_ERR_INVALID_ARG, "NorMuon needs 0 <= beta2 <= 1 and eps >= 0");
  if (!(opts->rms_target >= 0.f) || !std::isfinite(opts->rms_target))
    return fail(GBO_ERR_INVALID_ARG, "rms_target must be finite and >= 0");
  if (opts->rms_target > 0.f && !opts->normuon)
    return fail(GBO_ERR_INVALID_ARG, "rms_target needs NorMuon");
  gbo_plan *P = new gbo_plan();
  P->descs.assign(descs, descs + n);
  if (pool_len > 0) P->pool.assign(split_pool, split_pool + pool_len);
  P->opts = *opts;
  P->opts.abc = nullptr;
  const int k = opts->ns_steps;
  P->abc.resize(3 * k);
  for (int it = 0; it < k; ++it)
    for (int j = 0; j < 3; ++j) {
      const float v = opts->abc_per_step ? opts->abc[3 * it + j] : opts->abc[j];
      if (!std::isfinite(v)) {
        delete P;
        return fail(GBO_ERR_INVALID_ARG, "coefficient %d of iteration %d is not finite", j, it);
      }
      P->abc[3 * it + j] = v;
    }
  for (int it = 0; it < k; ++it) P->any_c |= P->abc[3 * it + 2] != 0.f;
  P->x_dtype = opts->precision == GBO_NS_F32 ? GBO_F32 : GBO_BF16;
  P->small_chain = g_small_chain.load() != 0;
  P->fused_gram = g_fused_gram.load() != 0;
  P->fused_mom = g_fused_mom.load() != 0;
  const int rc = validate_and_expand(P);
  if (rc != GBO_OK) {
    delete P;
    return rc;
  }
  P->hash = layout_hash(P);
  int64_t gemm = 0;
  for (const TcStep &st : build_schedule(P, nullptr)) gemm += tc_step_launches(st);
  P->info.launches_per_step =
      P->subs.empty() ? 0
                      : (P->n_tiles > 0) + (P->n_unfused > 0) + gemm +
                            (opts->normuon ? (opts->rms_target > 0.f ? 3 : (P->rows_streamed ? 2 : 1)) : 0);
  *out = P;
  return ok();
}

// The plan of descriptors t0 .. t1 - 1 alone (no cap), or nullptr with the
// error recorded.
gbo_plan *group_plan(const gbo_muon_desc *descs, int32_t t0, int32_t t1, const int64_t *pool, int32_t pool_len,
                     const gbo_muon_opts *opts) {
  gbo_muon_opts o = *opts;
  o.workspace_cap = 0;
  gbo_plan *q = nullptr;
  return make_plan(descs + t0, t1 - t0, pool, pool_len, &o, &q) == GBO_OK ? q : nullptr;
}

// Split the table into groups of consecutive descriptors, each the longest
// run from its first descriptor whose plan's workspace fits the cap (found
// by doubling, then bisection: a longer run never needs less workspace).
int split_into_groups(gbo_plan *P, const gbo_muon_desc *descs, int32_t n, const int64_t *pool, int32_t pool_len,
                      const gbo_muon_opts *opts) {
  const int64_t cap = opts->workspace_cap;
  auto fits = [&](int32_t t0, int32_t t1) {
    gbo_plan *q = group_plan(descs, t0, t1, pool, pool_len, opts);
    const bool f = q && (int64_t)q->ws_bytes <= cap;
    gbo_muon_plan_destroy(q);
    return f;
  };
  int64_t base = 0, mats = 0;
  for (int32_t t0 = 0; t0 < n;) {
    if (!fits(t0, t0 + 1)) {
      gbo_plan *q = group_plan(descs, t0, t0 + 1, pool, pool_len, opts);
      const size_t need = q ? q->ws_bytes : 0;
      gbo_muon_plan_destroy(q);
      return fail(GBO_ERR_WORKSPACE, "desc %d alone needs %zu bytes of workspace, above the cap of %lld", t0, need,
                  (long long)cap);
    }
    int32_t good = t0 + 1, bad = -1;
    while (good < n) {
      const int32_t cand = std::min<int64_t>(n, t0 + 2 * (int64_t)(good - t0));
      if (fits(t0, cand)) {
        good = cand;
      } else {
        bad = cand;
        break;
      }
    }
    while (bad > good + 1) {
      const int32_t mid = good + (bad - good) / 2;
      if (fits(t0, mid)) good = mid;
      else bad = mid;
    }
    gbo_plan *q = group_plan(descs, t0, good, pool, pool_len, opts);
    if (!q) return GBO_ERR_INVALID_ARG;
    q->dbg_base = base;
    q->mat_base = mats;
    mats += (int64_t)q->subs.size();
    for (int32_t t = t0; t < good; ++t) base += descs[t].rows * descs[t].cols;
    P->kids.push_back(q);
    t0 = good;
  }
  size_t ws = 0;
  int64_t launches = 0;
  for (const gbo_plan *q : P->kids) {
    ws = std::max(ws, q->ws_bytes);
    launches += q->info.launches_per_step;
  }
  P->ws_bytes = ws;
  P->info.launches_per_step = launches;
  return GBO_OK;
}

}  // namespace

extern "C" {

int gbo_muon_plan_create(const gbo_muon_desc *descs, int32_t n, const int64_t *split_pool,
                         int32_t pool_len, const gbo_muon_opts *opts, gbo_plan **out) {
  if (opts && opts->workspace_cap < 0) return fail(GBO_ERR_INVALID_ARG, "workspace_cap must be >= 0");
  const int rc = make_plan(descs, n, split_pool, pool_len, opts, out);
  if (rc != GBO_OK) return rc;
  gbo_plan *P = *out;
  if (opts->workspace_cap > 0 && (int64_t)P->ws_bytes > opts->workspace_cap) {
    const int src = split_into_groups(P, descs, n, split_pool, pool_len, opts);
    if (src != GBO_OK) {
      gbo_muon_plan_destroy(P);
      *out = nullptr;
      return src;
    }
  }
  return ok();
}

void gbo_muon_plan_destroy(gbo_plan *P) {
  if (!P) return;
  for (gbo_plan *q : P->kids) gbo_muon_plan_destroy(q);
  if (P->d_subs) cudaFree(P->d_subs);
  if (P->d_wmaps) cudaFree(P->d_wmaps);
  if (P->d_gbmaps) cudaFree(P->d_gbmaps);
  for (auto &iv : P->pending) {
    cudaEventDestroy(iv.a);
    cudaEventDestroy(iv.b);
  }
  for (cudaEvent_t e : P->event_pool) cudaEventDestroy(e);
  delete P;
}

size_t gbo_muon_workspace_bytes(const gbo_plan *P) { return P ? P->ws_bytes : 0; }

uint64_t gbo_desc_hash(const gbo_plan *P) { return P ? P->hash : 0; }

int gbo_muon_plan_info(const gbo_plan *P, gbo_plan_info *out) {
  if (!P || !out) return fail(GBO_ERR_INVALID_ARG, "NULL argument");
  *out = P->info;
  return ok();
}

int gbo_muon_plan_desc_flops(const gbo_plan *P, double *flops, int32_t n) {
  if (!P || !flops || n != (int32_t)P->descs.size())
    return fail(GBO_ERR_INVALID_ARG, "plan, output or descriptor count (%d) does not match", n);
  for (int32_t t = 0; t < n; ++t) flops[t] = 0.0;
  for (const DevSub &S : P->subs) flops[S.desc] += P->class_flops[S.cls];
  return ok();
}

int gbo_muon_plan_set_stats(gbo_plan *P, float *dev_stats) {
  if (!P) return fail(GBO_ERR_INVALID_ARG, "plan is NULL");
  if (!aligned(dev_stats, 4)) return fail(GBO_ERR_INVALID_ARG, "dev_stats misaligned");
  P->stats = dev_stats;
  for (gbo_plan *q : P->kids) q->stats = dev_stats ? dev_stats + 2 * q->mat_base : nullptr;
  return ok();
}

int gbo_muon_plan_set_free_sms(gbo_plan *P, int32_t n) {
  if (!P) return fail(GBO_ERR_INVALID_ARG, "plan is NULL");
  if (n < 0 || n > kMaxFreeSms) return fail(GBO_ERR_INVALID_ARG, "free SMs must be in 0 .. %d", kMaxFreeSms);
  P->free_sms = n;
  for (gbo_plan *q : P->kids) q->free_sms = n;
  return ok();
}

int gbo_muon_plan_set_timing(gbo_plan *P, int32_t enable) {
  if (!P) return fail(GBO_ERR_INVALID_ARG, "plan is NULL");
  P->timing = enable != 0;
  for (gbo_plan *q : P->kids) q->timing = P->timing;
  return ok();
}

int gbo_muon_plan_set_event(gbo_plan *P, int32_t phase, void *event) {
  if (!P || phase < 0 || phase >= GBO_N_PHASES) return fail(GBO_ERR_INVALID_ARG, "bad plan or phase");
  // in groups, the last group's occurrence of the phase is the step's last
  gbo_plan *target = P->kids.empty() ? P : P->kids.back();
  target->after_phase[phase] = static_cast<cudaEvent_t>(event);
  return ok();
}

int gbo_muon_plan_phase_times(gbo_plan *P, float *ms, int64_t *launches, int32_t n_phases) {
  if (!P || n_phases < 0 || (n_phases > 0 && (!ms || !launches)))
    return fail(GBO_ERR_INVALID_ARG, "bad argument");
  for (int i = 0; i < n_phases; ++i) {
    ms[i] = 0.f;
    launches[i] = 0;
  }
  if (!P->kids.empty()) {  // the sum over the groups
    std::vector<float> km(n_phases);
    std::vector<int64_t> kl(n_phases);
    for (gbo_plan *q : P->kids) {
      const int rc = gbo_muon_plan_phase_times(q, km.data(), kl.data(), n_phases);
      if (rc != GBO_OK) return rc;
      for (int i = 0; i < n_phases; ++i) {
        ms[i] += km[i];
        launches[i] += kl[i];
      }
    }
    return ok();
  }
  if (!P->pending.empty()) {
    cudaError_t e = cudaEventSynchronize(P->pending.back().b);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
  }
  for (auto &iv : P->pending) {
    float t = 0.f;
    cudaError_t e = cudaEventElapsedTime(&t, iv.a, iv.b);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    if (iv.phase < n_phases) {
      ms[iv.phase] += t;
      launches[iv.phase] += iv.launches;
    }
    P->event_pool.push_back(iv.a);
    P->event_pool.push_back(iv.b);
  }
  P->pending.clear();
  return ok();
}

int gbo_muon_step(gbo_plan *P, float lr, void *workspace, size_t ws_bytes, float *dbg_update,
                  int32_t *dev_status, gbo_stream_t stream) {
  if (!P) return fail(GBO_ERR_INVALID_ARG, "plan is NULL");
  if (!std::isfinite(lr)) return fail(GBO_ERR_INVALID_ARG, "lr is not finite");
  if (!P->kids.empty()) {  // the groups in turn, on the same workspace
    if (!workspace || ws_bytes < P->ws_bytes)
      return fail(GBO_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", P->ws_bytes, ws_bytes);
    for (gbo_plan *q : P->kids) {
      const int rc = gbo_muon_step(q, lr, workspace, ws_bytes, dbg_update ? dbg_update + q->dbg_base : nullptr,
                                   dev_status, stream);
      if (rc != GBO_OK) return rc;
    }
    return ok();
  }
  if (P->subs.empty()) return ok();
  if (!workspace || ws_bytes < P->ws_bytes)
    return fail(GBO_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", P->ws_bytes, ws_bytes);
  if (!aligned(workspace, 256)) return fail(GBO_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (!aligned(dbg_update, 4) || !aligned(dev_status, 4))
    return fail(GBO_ERR_INVALID_ARG, "dbg_update / dev_status misaligned");
  int dev = -1;
  DeviceInfo di;
  int rc = current_device(&dev, &di);
  if (rc != GBO_OK) return rc;
  if (P->device < 0) {
    // first call on a device: upload the matrix table
    cudaError_t e = cudaMalloc(&P->d_subs, P->subs.size() * sizeof(DevSub));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(matrix table)");
    e = cudaMemcpy(P->d_subs, P->subs.data(), P->subs.size() * sizeof(DevSub), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(matrix table)");
    if (P->x_dtype == GBO_BF16) {
      const int me = build_weight_maps(P->descs.data(), (int32_t)P->descs.size(), &P->d_wmaps);
      if (me) return cuda_fail(me, "weight tensor maps");
    }
    if (!P->gb_pairs.empty()) {  // the fused momentum pass's G and B maps, two per pair
      const size_t map_bytes = 128;  // sizeof(CUtensorMap), 64-byte aligned
      const size_t bytes = P->gb_pairs.size() * 2 * map_bytes;
      std::unique_ptr<unsigned char, void (*)(void *)> maps(static_cast<unsigned char *>(std::aligned_alloc(64, bytes)),
                                                           std::free);
      if (!maps) return fail(GBO_ERR_CUDA, "host memory for the G and B tensor maps");
      std::memset(maps.get(), 0, bytes);
      for (size_t k = 0; k < P->gb_pairs.size(); ++k) {
        const gbo_muon_desc &d = P->descs[P->gb_pairs[k].first];
        if (!encode_gb_maps(maps.get() + k * 2 * map_bytes, d.g, d.mom, d.rows, d.cols, P->gb_pairs[k].second))
          return fail(GBO_ERR_CUDA, "G and B tensor maps of desc %d refused", P->gb_pairs[k].first);
      }
      e = cudaMalloc(&P->d_gbmaps, bytes);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(G and B tensor maps)");
      e = cudaMemcpy(P->d_gbmaps, maps.get(), bytes, cudaMemcpyHostToDevice);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(G and B tensor maps)");
    }
    P->device = dev;
    P->sm_count = di.sm_count;
  } else if (P->device != dev) {
    return fail(GBO_ERR_INVALID_ARG, "plan was set up on device %d, current device is %d", P->device, dev);
  }
  char *ws = static_cast<char *>(workspace);
  void *x[2] = {ws + P->off_x[0], ws + P->off_x[1]};
  float *alpha = reinterpret_cast<float *>(ws + P->off_alpha);
  float *partials = reinterpret_cast<float *>(ws + P->off_part);
  void *st = stream;
  cudaEvent_t last = nullptr;
  // the caller's event after the momentum pass (the gradients are no longer
  // read) follows the chain launch that runs the fused matrices' momentum
  // pass, if there is one
  bool mom_event_due = P->after_phase[kPhaseMomentum] != nullptr;
  auto mark = [&](int phase, int64_t n_launch, bool mom_done = true) {
    if (phase == kPhaseMomentum) {
      if (mom_event_due && mom_done) {
        cudaEventRecord(P->after_phase[phase], reinterpret_cast<cudaStream_t>(stream));
        mom_event_due = false;
      }
    } else if (P->after_phase[phase]) {
      cudaEventRecord(P->after_phase[phase], reinterpret_cast<cudaStream_t>(stream));
    }
    if (mom_event_due && mom_done && phase != kPhaseMomentum) {
      cudaEventRecord(P->after_phase[kPhaseMomentum], reinterpret_cast<cudaStream_t>(stream));
      mom_event_due = false;
    }
    if (!P->timing) return;
    cudaEvent_t b = take_event(P);
    cudaEventRecord(b, reinterpret_cast<cudaStream_t>(stream));
    P->pending.push_back({last, b, phase, n_launch});
    last = take_event(P);
    cudaEventRecord(last, reinterpret_cast<cudaStream_t>(stream));
  };
  if (P->timing) {
    last = take_event(P);
    cudaEventRecord(last, reinterpret_cast<cudaStream_t>(stream));
  }
  const int32_t nsub = (int32_t)P->subs.size();
  void *x0t = P->x_dtype == GBO_F32 ? ws + P->off_xt[0] : nullptr;
  int err = launch_momentum(P->d_subs, nsub, P->n_tiles, P->opts.mu, P->opts.nesterov, x[0], x0t, P->x_dtype,
                            partials, P->mom_stream_g, dev_status, P->sm_count, st);
  if (err) return cuda_fail(err, "momentum kernel");
  if (P->n_unfused > 0) {
    err = launch_prenorm_finalize(P->d_subs, nsub, partials, alpha, dev_status, P->stats, P->sm_count, st);
    if (err) return cuda_fail(err, "pre-normalisation kernel");
  }
  mark(kPhaseMomentum, (P->n_tiles > 0) + (P->n_unfused > 0), !P->any_mom_fused);
  PhaseArgs A{};
  A.subs = P->d_subs;
  A.wmaps = P->d_wmaps;
  A.alpha = alpha;
  A.dbg = dbg_update;
  A.status = dev_status;
  A.lr = lr;
  A.gbmaps = P->d_gbmaps;
  A.alpha_out = alpha;
  A.mu = P->opts.mu;
  A.nesterov = P->opts.nesterov;
  A.stats = P->stats;
  bool fused_left = P->any_mom_fused;  // a fused momentum pass is still to be launched
  // the persistent Newton-Schulz kernels' SMs: all but the free ones
  const int ns_sms = std::max(2, P->sm_count - P->free_sms);
  for (const TcStep &step : build_schedule(P, ws)) {
    int64_t nl = 0;
    err = P->x_dtype == GBO_BF16
              ? launch_ns_gemm_tc(step.jobs.data(), (int32_t)step.jobs.size(), A, ns_sms, st, &nl)
              : launch_ns_gemm_tf32(step.jobs.data(), (int32_t)step.jobs.size(), A, ns_sms, st, &nl);
    if (err) return cuda_fail(err, "Newton-Schulz kernel");
    if (fused_left)
      for (const GemmJob &J : step.jobs)
        if (J.mode == kChain && J.cls->mom_fused) fused_left = false;
    mark(step.phase, nl, !fused_left);
  }
  if (P->opts.normuon) {
    err = launch_normuon_rows(P->d_subs, nsub, P->n_row_blocks, x[0], x[1], P->x_dtype, P->opts.beta2,
                              P->opts.eps, lr, dbg_update, dev_status, P->opts.rms_target,
                              reinterpret_cast<float *>(ws + P->off_rowf),
                              reinterpret_cast<float *>(ws + P->off_rowpart),
                              reinterpret_cast<float *>(ws + P->off_mscale),
                              P->x_dtype == GBO_BF16 ? reinterpret_cast<const float *>(ws + P->off_rowss) : nullptr,
                              P->rows_streamed, P->stats != nullptr, P->sm_count, st);
    if (err) return cuda_fail(err, "NorMuon rows kernel");
    mark(kPhaseRows, P->opts.rms_target > 0.f ? 3 : 1);
  }
  if (P->stats) {  // ||U||_F of every matrix, from the partial sums the step left
    err = launch_stats_finalize(P->d_subs, nsub, P->opts.normuon, P->opts.rms_target,
                                reinterpret_cast<const float *>(ws + P->off_rowss),
                                reinterpret_cast<const float *>(ws + P->off_rowpart), P->stats, st);
    if (err) return cuda_fail(err, "statistics kernel");
  }
  if (P->timing && last) P->event_pool.push_back(last);
  return ok();
}

int gbo_normuon_rownorm(const float *O, int64_t rows, int64_t cols, float *row_v, void *w,
                        int32_t w_dtype, float beta2, float eps, float scale, float lr, float wd,
                        float *dbg_update, gbo_stream_t stream) {
  if (rows < 0 || cols < 0) return fail(GBO_ERR_INVALID_ARG, "negative size");
  if (rows == 0 || cols == 0) return ok();
  if (!O || !row_v || !w) return fail(GBO_ERR_INVALID_ARG, "NULL pointer");
  if (!valid_dtype(w_dtype)) return fail(GBO_ERR_DTYPE, "w_dtype must be GBO_F32 or GBO_BF16");
  if (!aligned(O, 4) || !aligned(row_v, 4) || !aligned(w, dtype_size(w_dtype)) || !aligned(dbg_update, 4))
    return fail(GBO_ERR_INVALID_ARG, "misaligned pointer");
  int dev;
  DeviceInfo di;
  int rc = current_device(&dev, &di);
  if (rc != GBO_OK) return rc;
  const int err = launch_normuon_rownorm_plain(O, rows, cols, row_v, w, w_dtype, beta2, eps, scale, lr,
                                               wd, dbg_update, stream);
  if (err) return cuda_fail(err, "NorMuon rownorm kernel");
  return ok();
}

int32_t gbo_testing_set_small_chain(int32_t enable) { return g_small_chain.exchange(enable != 0 ? 1 : 0); }

int32_t gbo_testing_set_fused_gram(int32_t enable) { return g_fused_gram.exchange(enable != 0 ? 1 : 0); }

int32_t gbo_testing_set_fused_momentum(int32_t enable) { return g_fused_mom.exchange(enable != 0 ? 1 : 0); }

int32_t gbo_testing_set_tail_split(int32_t enable) { return gbo::set_tail_split(enable); }

int32_t gbo_testing_set_momentum_stream(int32_t enable) { return gbo::set_momentum_stream(enable); }

int32_t gbo_testing_pair_residency(void) { return gbo::pair_residency(); }

int32_t gbo_testing_set_pdl(int32_t mode) {
  if (mode < 0 || mode > 2) return -1;
  return gbo::g_pdl.exchange(mode);
}

int gbo_testing_wait_timeout(int32_t *dev_status, uint32_t limit_us, gbo_stream_t stream) {
  if (!dev_status || !aligned(dev_status, 4)) return fail(GBO_ERR_INVALID_ARG, "dev_status is NULL or misaligned");
  if (limit_us == 0 || limit_us > 10000000u) return fail(GBO_ERR_INVALID_ARG, "limit_us must be in 1..10^7");
  int dev;
  DeviceInfo di;
  int rc = current_device(&dev, &di);
  if (rc != GBO_OK) return rc;
  const int err = launch_wait_timeout(dev_status, (uint64_t)limit_us * 1000u, stream);
  if (err) return cuda_fail(err, "wait time-out kernel");
  return ok();
}

size_t gbo_clip_norm_workspace_bytes(void) { return (size_t)kClipBlocks * sizeof(float); }

int gbo_clip_norm(const gbo_tensor *grads, int32_t n, float max_norm, float *dev_total_norm,
                  float *dev_coef, int32_t *dev_status, void *workspace, size_t ws_bytes,
                  gbo_stream_t stream) {
  if (n < 0 || (n > 0 && !grads)) return fail(GBO_ERR_INVALID_ARG, "bad gradient table");
  if (n > 64 * kClipBlocks) return fail(GBO_ERR_INVALID_ARG, "more than %d tensors", 64 * kClipBlocks);
  if (!(max_norm > 0.f) || !std::isfinite(max_norm)) return fail(GBO_ERR_INVALID_ARG, "max_norm must be > 0");
  if (!workspace || ws_bytes < gbo_clip_norm_workspace_bytes())
    return fail(GBO_ERR_WORKSPACE, "clip workspace of %zu bytes needed", gbo_clip_norm_workspace_bytes());
  if (!aligned(workspace, 16)) return fail(GBO_ERR_WORKSPACE, "workspace must be 16-byte aligned");
  for (int32_t i = 0; i < n; ++i) {
    if (!valid_dtype(grads[i].dtype)) return fail(GBO_ERR_DTYPE, "tensor %d: bad dtype", i);
    if (grads[i].numel < 0) return fail(GBO_ERR_INVALID_ARG, "tensor %d: negative numel", i);
    if (grads[i].numel > 0 && (!grads[i].ptr || !aligned(grads[i].ptr, dtype_size(grads[i].dtype))))
      return fail(GBO_ERR_INVALID_ARG, "tensor %d: NULL or misaligned pointer", i);
  }
  int dev;
  DeviceInfo di;
  int rc = current_device(&dev, &di);
  if (rc != GBO_OK) return rc;
  const int err = launch_clip_norm(grads, n, max_norm, dev_total_norm, dev_coef, dev_status,
                                   static_cast<float *>(workspace), di.sm_count, stream);
  if (err) return cuda_fail(err, "clip-norm kernels");
  return ok();
}

int gbo_adamw_step(const gbo_adamw_desc *descs, int32_t n, const gbo_adamw_opts *opts,
                   const float *dev_coef, int32_t *dev_status, gbo_stream_t stream) {
  if (n < 0 || (n > 0 && !descs) || !opts) return fail(GBO_ERR_INVALID_ARG, "bad argument");
  if (!opts->dev_step && opts->step < 1) return fail(GBO_ERR_INVALID_ARG, "step must be >= 1");
  if (!aligned(opts->dev_step, 4)) return fail(GBO_ERR_INVALID_ARG, "dev_step misaligned");
  if (!(opts->beta1 >= 0.f && opts->beta1 < 1.f) || !(opts->beta2 >= 0.f && opts->beta2 < 1.f))
    return fail(GBO_ERR_INVALID_ARG, "betas must be in [0, 1)");
  if (!std::isfinite(opts->lr) || !std::isfinite(opts->eps) || !std::isfinite(opts->weight_decay))
    return fail(GBO_ERR_INVALID_ARG, "non-finite hyper-parameter");
  for (int32_t i = 0; i < n; ++i) {
    const gbo_adamw_desc &d = descs[i];
    if (!valid_dtype(d.g_dtype)) return fail(GBO_ERR_DTYPE, "tensor %d: bad g dtype", i);
    if (d.numel < 0) return fail(GBO_ERR_INVALID_ARG, "tensor %d: negative numel", i);
    if (d.numel > 0 && (!d.p || !d.g || !d.m || !d.v))
      return fail(GBO_ERR_INVALID_ARG, "tensor %d: NULL pointer", i);
    if (!aligned(d.p, 4) || !aligned(d.m, 4) || !aligned(d.v, 4) || !aligned(d.g, dtype_size(d.g_dtype)))
      return fail(GBO_ERR_INVALID_ARG, "tensor %d: misaligned pointer", i);
  }
  if (!aligned(dev_coef, 4)) return fail(GBO_ERR_INVALID_ARG, "dev_coef misaligned");
  int dev;
  DeviceInfo di;
  int rc = current_device(&dev, &di);
  if (rc != GBO_OK) return rc;
  const int err = launch_adamw(descs, n, opts, dev_coef, dev_status, di.sm_count, stream);
  if (err) return cuda_fail(err, "AdamW kernel");
  return ok();
}

}  // extern "C"
