"""ctypes binding of libgbo.so: argument marshalling only.

Every function here has the name of the C entry point it calls (see
``include/gbo.h``), turns torch tensors into device pointers and Python
numbers into C scalars, and raises :class:`GboError` on a non-zero status.
All arithmetic runs in the library's CUDA kernels; there is no fallback.
"""

import ctypes
import os

import torch

from . import build as _build

GBO_OK = 0
GBO_F32 = 0
GBO_BF16 = 1
GBO_NS_BF16 = 0
GBO_NS_F32 = 1
GBO_ROUTE_AUTO = 0
GBO_ROUTE_X = 1
GBO_ROUTE_GRAM = 2
GBO_STATUS_NONFINITE = 1
GBO_STATUS_TIMEOUT = 2
GBO_MAX_VIEW_DIMS = 6
GBO_N_PHASES = 6
PHASE_NAMES = ("momentum", "gram", "product", "square", "rows", "final")

c_void_p, c_int32, c_int64, c_float, c_size_t = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                                 ctypes.c_float, ctypes.c_size_t)


class GboError(RuntimeError):
    def __init__(self, code, message):
        super().__init__("libgbo error %d: %s" % (code, message))
        self.code = code


class MuonDesc(ctypes.Structure):
    _fields_ = [("w", c_void_p), ("g", c_void_p), ("mom", c_void_p), ("row_v", c_void_p),
                ("rows", c_int64), ("cols", c_int64), ("view", c_int64 * GBO_MAX_VIEW_DIMS),
                ("w_dtype", c_int32), ("g_dtype", c_int32), ("view_ndim", c_int32),
                ("n_split", c_int32), ("split_off", c_int32), ("lr_mult", c_float), ("wd", c_float),
                ("reserved", c_int32)]


class MuonOpts(ctypes.Structure):
    _fields_ = [("abc", ctypes.POINTER(c_float)), ("mu", c_float), ("beta2", c_float),
                ("eps", c_float), ("nesterov", c_int32), ("ns_steps", c_int32),
                ("abc_per_step", c_int32), ("precision", c_int32), ("normuon", c_int32),
                ("route", c_int32), ("rms_target", c_float), ("reserved", c_int32),
                ("workspace_cap", c_int64)]


class Tensor(ctypes.Structure):
    _fields_ = [("ptr", c_void_p), ("numel", c_int64), ("dtype", c_int32), ("reserved", c_int32)]


class AdamWDesc(ctypes.Structure):
    _fields_ = [("p", c_void_p), ("g", c_void_p), ("m", c_void_p), ("v", c_void_p),
                ("numel", c_int64), ("g_dtype", c_int32), ("reserved", c_int32)]


class AdamWOpts(ctypes.Structure):
    _fields_ = [("lr", c_float), ("beta1", c_float), ("beta2", c_float), ("eps", c_float),
                ("weight_decay", c_float), ("step", c_int32), ("dev_step", c_void_p)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("n_weights", c_int64), ("n_active", c_int64), ("n_matrices", c_int64),
                ("n_shape_classes", c_int64), ("muon_params", c_int64), ("ns_flops", ctypes.c_double),
                ("ns_flops_executed", ctypes.c_double), ("launches_per_step", c_int64),
                ("n_gram_route", c_int64), ("n_mom_fused", c_int64)]


_STRUCTS = (MuonDesc, MuonOpts, Tensor, AdamWDesc, AdamWOpts, PlanInfo)
_lib = None


def library_path():
    return _build.LIB_PATH


def lib():
    """Load libgbo.so (built by ``adamw_optimizer_step_gb300.build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError("libgbo.so is not built (%s); run adamw_optimizer_step_gb300.build.build()" % path)
    L = ctypes.CDLL(path)
    sig = {
        "gbo_muon_plan_create": (c_int32, [ctypes.POINTER(MuonDesc), c_int32, ctypes.POINTER(c_int64),
                                           c_int32, ctypes.POINTER(MuonOpts), ctypes.POINTER(c_void_p)]),
        "gbo_muon_plan_destroy": (None, [c_void_p]),
        "gbo_muon_workspace_bytes": (c_size_t, [c_void_p]),
        "gbo_desc_hash": (ctypes.c_uint64, [c_void_p]),
        "gbo_muon_step": (c_int32, [c_void_p, c_float, c_void_p, c_size_t, c_void_p, c_void_p, c_void_p]),
        "gbo_normuon_rownorm": (c_int32, [c_void_p, c_int64, c_int64, c_void_p, c_void_p, c_int32, c_float,
                                          c_float, c_float, c_float, c_float, c_void_p, c_void_p]),
        "gbo_clip_norm_workspace_bytes": (c_size_t, []),
        "gbo_clip_norm": (c_int32, [ctypes.POINTER(Tensor), c_int32, c_float, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_size_t, c_void_p]),
        "gbo_h2d_copy": (c_int32, [c_void_p, c_void_p, ctypes.c_int64, c_int32, c_void_p]),
        "gbo_muon_plan_set_free_sms": (c_int32, [c_void_p, c_int32]),
        "gbo_clip_norm_noalloc": (c_int32, [ctypes.POINTER(Tensor), c_int32, c_float, c_void_p, c_void_p,
                                            c_void_p, c_void_p]),
        "gbo_adamw_step": (c_int32, [ctypes.POINTER(AdamWDesc), c_int32, ctypes.POINTER(AdamWOpts), c_void_p,
                                     c_void_p, c_void_p]),
        "gbo_testing_wait_timeout": (c_int32, [c_void_p, ctypes.c_uint32, c_void_p]),
        "gbo_testing_set_small_chain": (c_int32, [c_int32]),
        "gbo_testing_set_fused_gram": (c_int32, [c_int32]),
        "gbo_testing_set_fused_momentum": (c_int32, [c_int32]),
        "gbo_testing_set_tail_split": (c_int32, [c_int32]),
        "gbo_testing_set_momentum_stream": (c_int32, [c_int32]),
        "gbo_testing_pair_residency": (c_int32, []),
        "gbo_testing_set_pdl": (c_int32, [c_int32]),
        "gbo_last_error": (ctypes.c_char_p, []),
        "gbo_abi_version": (c_int32, []),
        "gbo_struct_size": (c_size_t, [c_int32]),
        "gbo_launch_count": (ctypes.c_uint64, []),
        "gbo_muon_plan_info": (c_int32, [c_void_p, ctypes.POINTER(PlanInfo)]),
        "gbo_muon_plan_desc_flops": (c_int32, [c_void_p, ctypes.POINTER(ctypes.c_double), c_int32]),
        "gbo_muon_plan_set_timing": (c_int32, [c_void_p, c_int32]),
        "gbo_muon_plan_set_stats": (c_int32, [c_void_p, c_void_p]),
        "gbo_muon_plan_set_event": (c_int32, [c_void_p, c_int32, c_void_p]),
        "gbo_muon_plan_phase_times": (c_int32, [c_void_p, ctypes.POINTER(c_float), ctypes.POINTER(c_int64),
                                                c_int32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    for i, S in enumerate(_STRUCTS):
        if L.gbo_struct_size(i) != ctypes.sizeof(S):
            raise ImportError("ABI mismatch for %s: C %d bytes, Python %d" %
                              (S.__name__, L.gbo_struct_size(i), ctypes.sizeof(S)))
    _lib = L
    return L


def _check(code):
    if code != GBO_OK:
        raise GboError(code, lib().gbo_last_error().decode())


def _dtype(t):
    if t.dtype == torch.float32:
        return GBO_F32
    if t.dtype == torch.bfloat16:
        return GBO_BF16
    raise TypeError("tensor dtype must be float32 or bfloat16, got %s" % t.dtype)


def _dev_ptr(t, what, allow_host=False):
    if t is None:
        return None
    if not t.is_cuda and not allow_host:
        raise ValueError("%s must be a CUDA tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------------------
# Muon

class MuonPlan:
    """Owns a ``gbo_plan*`` and keeps the tensors it points to alive."""

    def __init__(self, handle, keepalive, n_descs=0):
        self.handle = handle
        self._keep = keepalive
        self.n_descs = n_descs

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.gbo_muon_plan_destroy(self.handle)
            self.handle = None


def muon_desc_table(entries, allow_host=False):
    """Marshal Muon weights into a ``gbo_muon_desc`` array and a split pool.

    Each entry is a dict with ``w`` (rows x cols, float32/bfloat16), ``g``
    (same shape, or None to skip), ``mom`` (float32), optional ``row_v``
    (float32, rows), ``view`` (tuple), ``split`` (tuple), ``lr_mult``, ``wd``.
    ``allow_host``: accept host tensors, for a plan that is only queried
    (plan creation never dereferences the pointers; such a plan must never
    be stepped).
    """
    arr = (MuonDesc * len(entries))()
    pool = []
    keep = []
    for d, e in zip(arr, entries):
        w, g, mom, rv = e["w"], e.get("g"), e.get("mom"), e.get("row_v")
        if w.dim() != 2:
            raise ValueError("Muon weights are 2-D")
        d.w = _dev_ptr(w, "w", allow_host)
        d.g = _dev_ptr(g, "g", allow_host)
        d.mom = _dev_ptr(mom, "mom", allow_host)
        d.row_v = _dev_ptr(rv, "row_v", allow_host)
        d.rows, d.cols = w.shape
        d.w_dtype = _dtype(w)
        d.g_dtype = _dtype(g) if g is not None else d.w_dtype
        view = e.get("view")
        if view is not None:
            if len(view) > GBO_MAX_VIEW_DIMS:
                raise ValueError("view has more than %d axes" % GBO_MAX_VIEW_DIMS)
            d.view_ndim = len(view)
            for k, s in enumerate(view):
                d.view[k] = int(s)
        split = e.get("split")
        if split is not None:
            d.n_split = len(split)
            d.split_off = len(pool)
            pool += [int(s) for s in split]
        d.lr_mult = float(e.get("lr_mult", 1.0))
        d.wd = float(e.get("wd", 0.0))
        keep += [w, g, mom, rv]
    return arr, pool, keep


def gbo_muon_plan_create(entries, *, abc=(1.5, -0.5, 0.0), ns_steps=5, mu=0.95, nesterov=True,
                         precision=GBO_NS_BF16, normuon=False, beta2=0.95, eps=1e-8, route=GBO_ROUTE_AUTO,
                         rms_target=0.0, workspace_cap=0, _query_only=False):
    """Validate a Muon table and build a plan (``abc``: one triple or one per step;
    ``route``: GBO_ROUTE_AUTO, GBO_ROUTE_X or GBO_ROUTE_GRAM; ``rms_target`` > 0
    with NorMuon: each matrix's update is scaled to that RMS; ``workspace_cap``
    > 0: the step runs the table in groups whose workspace fits the cap)."""
    L = lib()
    arr, pool, keep = muon_desc_table(entries, allow_host=_query_only)
    flat = []
    for t in ([abc] if len(abc) and not hasattr(abc[0], "__len__") else abc):
        flat += [float(x) for x in t]
    per_step = len(flat) > 3
    cabc = (c_float * len(flat))(*flat)
    opts = MuonOpts(ctypes.cast(cabc, ctypes.POINTER(c_float)), mu, beta2, eps, int(bool(nesterov)),
                    int(ns_steps), int(per_step), int(precision), int(bool(normuon)), int(route),
                    float(rms_target), 0, int(workspace_cap))
    cpool = (c_int64 * max(1, len(pool)))(*pool)
    out = c_void_p()
    _check(L.gbo_muon_plan_create(arr, len(entries), cpool, len(pool), ctypes.byref(opts), ctypes.byref(out)))
    return MuonPlan(out.value, keep, len(entries))


def gbo_muon_plan_destroy(plan):
    if plan.handle:
        lib().gbo_muon_plan_destroy(plan.handle)
        plan.handle = None


def gbo_muon_workspace_bytes(plan):
    return int(lib().gbo_muon_workspace_bytes(plan.handle))


def gbo_desc_hash(plan):
    return int(lib().gbo_desc_hash(plan.handle))


def gbo_muon_plan_info(plan):
    info = PlanInfo()
    _check(lib().gbo_muon_plan_info(plan.handle, ctypes.byref(info)))
    return {k: getattr(info, k) for k, _ in PlanInfo._fields_}


def muon_desc_flops(entries, **opts):
    """Executed Newton-Schulz FLOPs per step of every entry (host or device
    tensors), from a plan built only to be queried and then dropped."""
    plan = gbo_muon_plan_create(entries, _query_only=True, **opts)
    try:
        return gbo_muon_plan_desc_flops(plan)
    finally:
        gbo_muon_plan_destroy(plan)


def gbo_muon_plan_desc_flops(plan):
    """Executed Newton-Schulz FLOPs per step of every descriptor, in table order."""
    n = plan.n_descs
    out = (ctypes.c_double * max(1, n))()
    _check(lib().gbo_muon_plan_desc_flops(plan.handle, out, n))
    return [float(out[i]) for i in range(n)]


def gbo_muon_step(plan, lr, workspace, dbg_update=None, dev_status=None, stream=None):
    """One Muon step on ``stream`` (default: torch's current stream)."""
    ws = _dev_ptr(workspace, "workspace") if workspace is not None else None
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().gbo_muon_step(plan.handle, float(lr), ws, nbytes, _dev_ptr(dbg_update, "dbg_update"),
                               _dev_ptr(dev_status, "dev_status"), _stream(stream)))


def gbo_muon_plan_set_free_sms(plan, n):
    """Leave ``n`` SMs free of the plan's persistent Newton-Schulz kernels in
    later steps (for gbo_h2d_copy with ``n`` blocks on another stream)."""
    _check(lib().gbo_muon_plan_set_free_sms(plan.handle, int(n)))


def gbo_muon_plan_set_stats(plan, stats):
    """Per-matrix norms from later steps: ``stats`` is a float32 CUDA tensor of
    2 * n_matrices values (||D||_F, ||U||_F per matrix, table order), or None
    to stop."""
    if stats is not None and (stats.dtype != torch.float32 or stats.numel() < 2 * plan_matrices(plan)):
        raise ValueError("stats must be float32 with 2 values per matrix")
    plan._stats = stats  # kept alive while the plan writes to it
    _check(lib().gbo_muon_plan_set_stats(plan.handle, _dev_ptr(stats, "stats")))


def plan_matrices(plan):
    return gbo_muon_plan_info(plan)["n_matrices"]


def gbo_muon_plan_set_timing(plan, enable=True):
    _check(lib().gbo_muon_plan_set_timing(plan.handle, int(bool(enable))))


def gbo_muon_plan_set_event(plan, phase, event):
    """Record ``event`` (a torch.cuda.Event, or None to stop) after ``phase``
    (0 = momentum) of every later step, on the step's stream."""
    handle = None
    if event is not None:
        if not event.cuda_event:  # torch creates the CUDA event on first use
            event.record()
        handle = event.cuda_event
    _check(lib().gbo_muon_plan_set_event(plan.handle, int(phase), handle))
    plan._event = event  # keep it alive while the plan records it


def gbo_muon_plan_phase_times(plan):
    ms = (c_float * GBO_N_PHASES)()
    n = (c_int64 * GBO_N_PHASES)()
    _check(lib().gbo_muon_plan_phase_times(plan.handle, ms, n, GBO_N_PHASES))
    return {name: (float(ms[i]), int(n[i])) for i, name in enumerate(PHASE_NAMES)}


def gbo_normuon_rownorm(O, row_v, w, *, beta2, eps, scale, lr, wd=0.0, dbg_update=None, stream=None):
    rows, cols = O.shape
    if O.dtype != torch.float32:
        raise TypeError("O must be float32")
    _check(lib().gbo_normuon_rownorm(_dev_ptr(O, "O"), rows, cols, _dev_ptr(row_v, "row_v"), _dev_ptr(w, "w"),
                                     _dtype(w), float(beta2), float(eps), float(scale), float(lr), float(wd),
                                     _dev_ptr(dbg_update, "dbg_update"), _stream(stream)))


# ---------------------------------------------------------------------------
# AdamW

def gbo_clip_norm_workspace_bytes():
    return int(lib().gbo_clip_norm_workspace_bytes())


def gbo_clip_norm(grads, max_norm, total_norm, coef, workspace, dev_status=None, stream=None):
    """Global norm of ``grads`` into ``total_norm`` and the clip factor into ``coef``."""
    arr = (Tensor * max(1, len(grads)))()
    for d, g in zip(arr, grads):
        d.ptr = _dev_ptr(g, "grad")
        d.numel = g.numel()
        d.dtype = _dtype(g)
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().gbo_clip_norm(arr, len(grads), float(max_norm), _dev_ptr(total_norm, "total_norm"),
                               _dev_ptr(coef, "coef"), _dev_ptr(dev_status, "dev_status"),
                               _dev_ptr(workspace, "workspace"), nbytes, _stream(stream)))


def gbo_clip_norm_noalloc(grads, max_norm, total_norm, coef, dev_status=None, stream=None):
    """gbo_clip_norm without a workspace: the library's fixed device scratch
    is used, so nothing is allocated (for callers that cannot allocate)."""
    arr = (Tensor * max(1, len(grads)))()
    for d, g in zip(arr, grads):
        d.ptr = _dev_ptr(g, "grad")
        d.numel = g.numel()
        d.dtype = _dtype(g)
    _check(lib().gbo_clip_norm_noalloc(arr, len(grads), float(max_norm), _dev_ptr(total_norm, "total_norm"),
                                       _dev_ptr(coef, "coef"), _dev_ptr(dev_status, "dev_status"),
                                       _stream(stream)))


def gbo_h2d_copy(dst, src, blocks=0, stream=None):
    """Copy the page-locked host tensor ``src`` into the device tensor
    ``dst`` (both contiguous, the same number of bytes) with the library's
    copy kernel (``blocks`` SMs; 0: all), asynchronously on ``stream``."""
    if not (dst.is_cuda and dst.is_contiguous()):
        raise ValueError("dst must be a contiguous CUDA tensor")
    if src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous host tensor")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst and src differ in size")
    _check(lib().gbo_h2d_copy(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), nbytes,
                              int(blocks), _stream(stream)))


def gbo_adamw_step(params, *, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0, step=1,
                   coef=None, dev_status=None, stream=None, dev_step=None):
    """AdamW on ``params``: a list of (p, g, m, v) tensors (p, m, v float32).
    ``dev_step``: an int32 CUDA tensor holding t, read when the kernel runs
    (for CUDA graph replay), instead of the host ``step``."""
    arr = (AdamWDesc * max(1, len(params)))()
    for d, (p, g, m, v) in zip(arr, params):
        for t, nm in ((p, "p"), (m, "m"), (v, "v")):
            if t.dtype != torch.float32:
                raise TypeError("%s must be float32" % nm)
        d.p, d.g, d.m, d.v = (_dev_ptr(p, "p"), _dev_ptr(g, "g"), _dev_ptr(m, "m"), _dev_ptr(v, "v"))
        d.numel = p.numel()
        d.g_dtype = _dtype(g)
    if dev_step is not None and dev_step.dtype != torch.int32:
        raise TypeError("dev_step must be int32")
    opts = AdamWOpts(lr, beta1, beta2, eps, weight_decay, int(step), _dev_ptr(dev_step, "dev_step"))
    _check(lib().gbo_adamw_step(arr, len(params), ctypes.byref(opts), _dev_ptr(coef, "coef"),
                                _dev_ptr(dev_status, "dev_status"), _stream(stream)))


# ---------------------------------------------------------------------------
# diagnostics

def gbo_last_error():
    return lib().gbo_last_error().decode()


def gbo_abi_version():
    return int(lib().gbo_abi_version())


def gbo_struct_size(which):
    return int(lib().gbo_struct_size(which))


def gbo_testing_set_small_chain(enable):
    """Whether plans created from now on run the Gram route's p x p
    iterations of matrices with p <= 192 (bf16) in one on-chip chain launch.
    Returns the previous setting."""
    return bool(lib().gbo_testing_set_small_chain(1 if enable else 0))


def gbo_testing_set_fused_gram(enable):
    """Whether plans created from now on run the Gram of the chain's wide
    matrices with p <= 128 inside the chain launch (X_0 streamed through
    shared memory) rather than as a launch of its own.  Returns the previous
    setting."""
    return bool(lib().gbo_testing_set_fused_gram(1 if enable else 0))


def gbo_testing_set_fused_momentum(enable):
    """Whether plans created from now on run the momentum pass of the chain's
    wide p <= 128 matrices with bf16 gradients inside the chain launch (G and
    B streamed through shared memory) rather than in the momentum kernel
    (the default).  Returns the previous setting."""
    return bool(lib().gbo_testing_set_fused_momentum(1 if enable else 0))


def gbo_testing_set_tail_split(enable):
    """Whether launches of the bf16 CTA-pair kernel from now on run a last
    wave of at most half the resident pairs as 256 x 128 half tiles (the
    default).  Returns the previous setting."""
    return bool(lib().gbo_testing_set_tail_split(1 if enable else 0))


def gbo_testing_set_momentum_stream(enable):
    """Whether momentum passes from now on stream their tiles through shared
    memory where the plan allows it (the default) or take the register
    kernel; the results are bitwise the same.  Returns the previous
    setting."""
    return bool(lib().gbo_testing_set_momentum_stream(1 if enable else 0))


def gbo_testing_pair_residency():
    """CTA pairs of the bf16 Newton-Schulz kernel the current device holds at
    once (its pair launches' persistent grid)."""
    return int(lib().gbo_testing_pair_residency())


def gbo_testing_set_pdl(mode):
    """When launches from now on carry the programmatic-dependent-launch
    attribute: 0 never, 1 always, 2 (the default) in CUDA graph capture only.
    Returns the previous mode."""
    return int(lib().gbo_testing_set_pdl(int(mode)))


def gbo_testing_wait_timeout(dev_status, limit_us, stream=None):
    """Test hook: the GEMM's bounded wait on a barrier nothing arrives on."""
    _check(lib().gbo_testing_wait_timeout(_dev_ptr(dev_status, "dev_status"), int(limit_us), _stream(stream)))


def gbo_launch_count():
    return int(lib().gbo_launch_count())
