"""The C-ABI library builds, loads, exports every declared symbol, and its
host-side plan logic (validation, view expansion, workspace sizing, layout
hash) behaves as documented.  No GPU needed: plan creation touches no
device, and the fake addresses below are never dereferenced."""

import ctypes
import os
import re

import pytest

from adamw_optimizer_step_gb300 import _binding as B
from adamw_optimizer_step_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return B.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(gbo_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "gbo_muon_step" in names and "gbo_adamw_step" in names
    for n in names:
        assert hasattr(L, n), n
    assert B.gbo_abi_version() == 5
    for i, S in enumerate(B._STRUCTS):
        assert B.gbo_struct_size(i) == ctypes.sizeof(S)


FAKE = 1 << 20  # aligned fake device addresses; plan creation never dereferences them


def desc(i, rows, cols, view=None, split_off=0, n_split=0, w_dtype=B.GBO_BF16, g=True, row_v=False):
    d = B.MuonDesc()
    base = FAKE * (4 * i + 1)
    d.w = base
    d.g = base + FAKE if g else None
    d.mom = base + 2 * FAKE
    d.row_v = base + 3 * FAKE if row_v else None
    d.rows, d.cols = rows, cols
    d.w_dtype = w_dtype
    d.g_dtype = w_dtype
    if view:
        d.view_ndim = len(view)
        for k, s in enumerate(view):
            d.view[k] = s
    d.n_split = n_split
    d.split_off = split_off
    d.lr_mult = 1.0
    return d


def create(L, descs, pool=(), ns_steps=5, abc=(1.5, -0.5, 0.0), precision=B.GBO_NS_BF16, normuon=0,
           route=B.GBO_ROUTE_AUTO, rms_target=0.0, workspace_cap=0):
    arr = (B.MuonDesc * max(1, len(descs)))(*descs)
    cabc = (ctypes.c_float * len(abc))(*abc)
    opts = B.MuonOpts(ctypes.cast(cabc, ctypes.POINTER(ctypes.c_float)), 0.95, 0.95, 1e-8, 1, ns_steps,
                      int(len(abc) > 3), precision, normuon, route, rms_target, 0, workspace_cap)
    cpool = (ctypes.c_int64 * max(1, len(pool)))(*pool)
    out = ctypes.c_void_p()
    rc = L.gbo_muon_plan_create(arr, len(descs), cpool, len(pool), ctypes.byref(opts), ctypes.byref(out))
    return rc, out.value


def info(L, plan):
    i = B.PlanInfo()
    assert L.gbo_muon_plan_info(plan, ctypes.byref(i)) == 0
    return i


def test_page_views_expand(L):
    """The worked view shapes of the build_parameter_groups page."""
    descs = [desc(0, 32, 8, (2, 16, 8)), desc(1, 24, 8, (3, 2, 4, 8)), desc(2, 20, 8, (2, 10, 8), 0, 2)]
    rc, plan = create(L, descs, pool=(4, 6))
    assert rc == 0, L.gbo_last_error()
    i = info(L, plan)
    assert (i.n_weights, i.n_active, i.n_matrices) == (3, 3, 2 + 6 + 4)
    # oriented shapes: (16,8)->(8,16); (4,8); (6,8)
    assert i.n_shape_classes == 3
    assert i.muon_params == 32 * 8 + 24 * 8 + 20 * 8
    assert L.gbo_muon_workspace_bytes(plan) > 0
    L.gbo_muon_plan_destroy(plan)


@pytest.mark.parametrize("case,code", [
    (dict(rows=32, cols=8, view=(2, 15, 8)), -2),
    (dict(rows=32, cols=8, view=(2, 16, 4)), -2),
    (dict(rows=32, cols=8, view=(0, 16, 8)), -2),
    (dict(rows=20, cols=8, view=(2, 10, 8), split=(4, 5)), -2),
    (dict(rows=20, cols=8, view=(2, 10, 8), split=(10, 0)), -2),
    (dict(rows=0, cols=8), -2),
    (dict(rows=20, cols=8, view=(160,)), -2),
])
def test_view_rules_refused(L, case, code):
    split = case.get("split")
    d = desc(0, case["rows"], case["cols"], case.get("view"), 0, len(split) if split else 0)
    rc, plan = create(L, [d], pool=split or ())
    assert rc == code, L.gbo_last_error()
    assert plan is None
    assert L.gbo_last_error()


def test_other_refusals(L):
    # empty table
    rc, _ = create(L, [])
    assert rc == -4
    # the same weight twice
    d0 = desc(0, 8, 8)
    d1 = desc(1, 8, 8)
    d1.w = d0.w
    rc, _ = create(L, [d0, d1])
    assert rc == -3
    # bad dtype
    d = desc(0, 8, 8)
    d.w_dtype = 7
    assert create(L, [d])[0] == -5
    # NorMuon without row_v
    assert create(L, [desc(0, 8, 8)], normuon=1)[0] == -1
    # ns_steps out of range, NaN coefficient
    assert create(L, [desc(0, 8, 8)], ns_steps=0)[0] == -1
    assert create(L, [desc(0, 8, 8)], abc=(float("nan"), 0.0, 0.0))[0] == -1
    # misaligned weight pointer for bf16
    d = desc(0, 8, 8)
    d.w += 1
    assert create(L, [d])[0] == -1
    # split sizes outside the pool
    assert create(L, [desc(0, 20, 8, (2, 10, 8), 1, 2)], pool=(4, 6))[0] == -1
    # the RMS-keeping scale: finite and >= 0, and only with NorMuon
    assert create(L, [desc(0, 8, 8)], rms_target=0.2)[0] == -1
    assert create(L, [desc(0, 8, 8)], rms_target=-1.0)[0] == -1
    assert create(L, [desc(0, 8, 8)], rms_target=float("inf"))[0] == -1


def test_missing_gradient_skips(L):
    rc, plan = create(L, [desc(0, 16, 16), desc(1, 32, 16, g=False)])
    assert rc == 0
    i = info(L, plan)
    assert (i.n_weights, i.n_active, i.n_matrices, i.muon_params) == (2, 1, 1, 256)
    L.gbo_muon_plan_destroy(plan)


def test_flop_count_and_launches(L):
    descs = lambda: [desc(0, 5632 * 2, 2048, (2, 5632, 2048)), desc(1, 2048, 5632)]
    # p = 2048, q = 5632 on CTA pairs: 256 x 256 output tiles, K padded to 64.
    # A symmetric 2048 x 2048 output runs the 8 * 9 / 2 = 36 tiles on or above
    # the diagonal; a 2048 x 5632 output runs 8 x 22 tiles.
    tile = 2 * 256 * 256
    gram, sym, prod = 36 * tile * 5632, 36 * tile * 2048, 8 * 22 * tile * 2048
    rc, plan = create(L, descs(), route=B.GBO_ROUTE_X)
    assert rc == 0
    i = info(L, plan)
    # the tall gate/up halves and the wide down projection: two classes (X kept in stored orientation)
    assert i.n_matrices == 3 and i.n_shape_classes == 2 and i.n_gram_route == 0
    assert i.ns_flops == 3 * 5 * 4 * 2048 ** 2 * 5632
    assert i.ns_flops_executed == 3 * 5 * (gram + prod)
    # momentum + finalize + 5 x (Gram + product)
    assert i.launches_per_step == 12
    L.gbo_muon_plan_destroy(plan)
    # the automatic route takes the Gram route for q > p: the Gram, 12
    # symmetric 2048^3 products, one product with X_0, in 2k + 1 launches
    for route in (B.GBO_ROUTE_AUTO, B.GBO_ROUTE_GRAM):
        rc, plan = create(L, descs(), route=route)
        i = info(L, plan)
        assert i.n_gram_route == 3 and i.ns_flops == 3 * 5 * 4 * 2048 ** 2 * 5632
        assert i.ns_flops_executed == 3 * (gram + 12 * sym + prod)
        assert i.launches_per_step == 2 + 11
        L.gbo_muon_plan_destroy(plan)
    # square matrices stay on the X route unless forced; k = 1 never takes
    # the Gram route; c != 0 (one square of A per iteration) and the fp32
    # mode take it as the cubic in bf16 does
    rc, plan = create(L, [desc(0, 256, 256)])
    assert info(L, plan).n_gram_route == 0
    L.gbo_muon_plan_destroy(plan)
    rc, plan = create(L, [desc(0, 256, 256)], route=B.GBO_ROUTE_GRAM)
    assert info(L, plan).n_gram_route == 1
    L.gbo_muon_plan_destroy(plan)
    rc, plan = create(L, descs(), route=B.GBO_ROUTE_GRAM, ns_steps=1)
    assert rc == 0 and info(L, plan).n_gram_route == 0
    L.gbo_muon_plan_destroy(plan)
    rc, plan = create(L, descs(), abc=(15 / 8, -5 / 4, 3 / 8))
    i = info(L, plan)
    # Gram (+ square), then per iteration T / Q, A and a square: 1 + 1 + 4 x 3 + Q_5 + X_5
    assert i.n_gram_route == 3 and i.launches_per_step == 2 + 16
    assert i.ns_flops_executed == 3 * (gram + (12 + 5) * sym + prod)
    L.gbo_muon_plan_destroy(plan)
    rc, plan = create(L, descs(), precision=B.GBO_NS_F32)
    assert rc == 0 and info(L, plan).n_gram_route == 3 and info(L, plan).launches_per_step == 2 + 11
    L.gbo_muon_plan_destroy(plan)
    assert create(L, descs(), route=3)[0] == -1
    rc, plan = create(L, [desc(0, 64, 64)], abc=(15 / 8, -5 / 4, 3 / 8), route=B.GBO_ROUTE_X)
    assert info(L, plan).launches_per_step == 2 + 5 * 3
    L.gbo_muon_plan_destroy(plan)
    # a matrix of at most 192 rows takes the Gram route with the on-chip
    # chain automatically, square or not.  p = 64: the chain from X_0 (its
    # Gram and square on chip), then the product on single CTAs; p = 150:
    # the Gram (and the square of A_0) on CTA pairs, the chain, the product.
    # The chain from X_0 runs in the step of the other chain, so the products
    # share a step, and one single-CTA launch (the weight-writing last product
    # of a class of at most 256 rows runs on single CTAs).  Launches by step,
    # cubic: {Gram}, {both chains}, {both products}; quintic: {Gram},
    # {square}, {both chains}, {both products}
    for abc, launches in (((1.5, -0.5, 0.0), 2 + 1 + 2 + 1), ((15 / 8, -5 / 4, 3 / 8), 2 + 1 + 1 + 2 + 1)):
        rc, plan = create(L, [desc(0, 64, 64), desc(1, 150, 150)], abc=abc)
        i = info(L, plan)
        assert i.n_gram_route == 2 and i.launches_per_step == launches
        L.gbo_muon_plan_destroy(plan)


# eleven shape classes of at most 128 rows, wide and tall, with K ragged
CHAIN_CLASSES = [(8, 200, None), (200, 8, None), (24, 72, None), (130, 60, None), (64, 64, None),
                 (100, 1000, None), (1000, 100, None), (127, 129, None), (129, 127, None),
                 (2 * 40, 520, (2, 40, 520)), (3 * 16, 48, (3, 16, 48))]


def test_chain_gram_launch_groups(L):
    """Eleven Gram-route classes of at most 128 rows: the chain with its
    Gram on chip takes eight classes to a launch, so two chain launches and
    two product launches follow momentum and the pre-normalisation, for
    the cubic and for c != 0 (whose square of A_0 also runs on chip)."""
    ds = [desc(i, r, c, v) for i, (r, c, v) in enumerate(CHAIN_CLASSES)]
    for abc in ((1.5, -0.5, 0.0), (15 / 8, -5 / 4, 3 / 8)):
        rc, plan = create(L, ds, route=B.GBO_ROUTE_GRAM, abc=abc)
        assert rc == 0, L.gbo_last_error()
        i = info(L, plan)
        assert i.n_shape_classes == 11 and i.n_gram_route == 9 + 2 + 3
        assert i.launches_per_step == 2 + 2 + 2
        L.gbo_muon_plan_destroy(plan)


def test_small_chain_counts(L):
    """Gram-route matrices of at most 192 rows (bf16) run their p x p
    iterations in one on-chip launch.  For a wide matrix of p <= 128 the
    chain starts from X_0 (the Gram, and the square of A_0 when c != 0, on
    chip: 128 x 128 tiles, K padded to 64), then the product with X_0: two
    launches.  Otherwise the Gram is a tile-kernel launch of its own.  Each
    op of the chain is one 128 x 128 tile (128 x 256 when T and Q are formed
    together) with K padded to 64; with the chain switched off every p x p
    product is a tile-kernel launch of its own."""
    d = lambda: [desc(0, 4 * 96, 1000, (4, 96, 1000))]  # four 96 x 1000 matrices: p = 96, q = 1000
    tile = 2 * 128 * 256            # one single-CTA tile of the tile kernel, per unit of K
    gram, prod, sym = tile * 1024, 4 * tile * 128, tile * 128
    op128, op256 = 2 * 128 * 128 * 128, 2 * 128 * 256 * 128
    gram_chip = 2 * 128 * 128 * 1024  # the on-chip Gram: one 128 x 128 tile, K = 1000 padded to 1024
    # cubic, k = 5: T, A_1/P_1, then 3 x (T with Q, A/P), Q_5
    cubic_chain = 6 * op128 + 3 * op256
    # quintic, k = 5: T, A_1, square; 3 x (T with Q, A, square); Q_5 -- plus the square of A_0
    quintic_chain = 10 * op128 + 3 * op256
    rc, plan = create(L, d(), route=B.GBO_ROUTE_GRAM)
    i = info(L, plan)
    assert i.n_gram_route == 4 and i.n_mom_fused == 0 and i.launches_per_step == 2 + 2
    assert i.ns_flops_executed == 4 * (gram_chip + cubic_chain + prod)
    L.gbo_muon_plan_destroy(plan)
    rc, plan = create(L, d(), route=B.GBO_ROUTE_GRAM, abc=(15 / 8, -5 / 4, 3 / 8))
    i = info(L, plan)
    assert i.launches_per_step == 2 + 2
    assert i.ns_flops_executed == 4 * (gram_chip + op128 + quintic_chain + prod)
    L.gbo_muon_plan_destroy(plan)
    # with the momentum pass in the chain launch too (bf16 G on 16-byte rows):
    # no momentum or pre-normalisation launch
    prev = L.gbo_testing_set_fused_momentum(1)
    try:
        rc, plan = create(L, d(), route=B.GBO_ROUTE_GRAM)
        i = info(L, plan)
        assert i.n_mom_fused == 4 and i.launches_per_step == 2
        assert i.ns_flops_executed == 4 * (gram_chip + cubic_chain + prod)
        L.gbo_muon_plan_destroy(plan)
    finally:
        L.gbo_testing_set_fused_momentum(prev)
    # with the Gram as a launch of its own (and the square of A_0 another)
    prev = L.gbo_testing_set_fused_gram(0)
    try:
        rc, plan = create(L, d(), route=B.GBO_ROUTE_GRAM)
        i = info(L, plan)
        assert i.launches_per_step == 2 + 3 and i.ns_flops_executed == 4 * (gram + cubic_chain + prod)
        L.gbo_muon_plan_destroy(plan)
        rc, plan = create(L, d(), route=B.GBO_ROUTE_GRAM, abc=(15 / 8, -5 / 4, 3 / 8))
        i = info(L, plan)
        assert i.launches_per_step == 2 + 4 and i.ns_flops_executed == 4 * (gram + sym + quintic_chain + prod)
        L.gbo_muon_plan_destroy(plan)
    finally:
        L.gbo_testing_set_fused_gram(prev)
    # a matrix held tall (its stored rows > columns: X is q x p) too: its
    # Gram X^T X reads X_0 in 64-row blocks; 200 x 96 stored, p = 96, q = 200
    # (K padded to 256); the product runs on X held tall (q x p output)
    rc, plan = create(L, [desc(0, 200, 96)], route=B.GBO_ROUTE_GRAM)
    i = info(L, plan)
    assert i.launches_per_step == 2 + 2
    assert i.ns_flops_executed == 2 * 128 * 128 * 256 + cubic_chain + 2 * tile * 128  # 200 output rows: two tiles
    L.gbo_muon_plan_destroy(plan)
    # 128 < p <= 192: two 128-row halves with N = 192, T and Q as separate
    # products: T, A_1/P_1, 3 x (T, Q, A/P), Q_5; the Gram runs on CTA pairs
    # (256 x 256 tiles, K padded to 128), the weight-writing product with X_0
    # on single CTAs (two 128-row tiles x 6 column tiles, K = 192 in 64-wide
    # blocks)
    rc, plan = create(L, [desc(0, 2 * 192, 1536, (2, 192, 1536))], route=B.GBO_ROUTE_GRAM)
    i = info(L, plan)
    pair = 2 * 256 * 256
    single = 2 * 128 * 256
    chain192 = 12 * 2 * (2 * 128 * 192 * 192)
    assert i.launches_per_step == 2 + 3
    assert i.ns_flops_executed == 2 * (pair * 1536 + chain192 + 12 * single * 192)
    L.gbo_muon_plan_destroy(plan)
    # the fp32 mode and larger p keep one launch per product
    rc, plan = create(L, d(), route=B.GBO_ROUTE_GRAM, precision=B.GBO_NS_F32)
    assert info(L, plan).launches_per_step == 2 + 11
    L.gbo_muon_plan_destroy(plan)
    rc, plan = create(L, [desc(0, 200, 1536)], route=B.GBO_ROUTE_GRAM)
    assert info(L, plan).launches_per_step == 2 + 11
    L.gbo_muon_plan_destroy(plan)
    prev = L.gbo_testing_set_small_chain(0)
    try:
        rc, plan = create(L, d(), route=B.GBO_ROUTE_GRAM)
        i = info(L, plan)
        assert i.launches_per_step == 2 + 11 and i.ns_flops_executed == 4 * (gram + 12 * sym + prod)
        L.gbo_muon_plan_destroy(plan)
    finally:
        assert L.gbo_testing_set_small_chain(prev) == 0


def test_layout_hash(L):
    """Equal layouts hash equal whatever the pointers; a different view or
    split changes the hash (the checkpoint compatibility check)."""
    _, p1 = create(L, [desc(0, 20, 8, (2, 10, 8), 0, 2)], pool=(4, 6))
    d = desc(5, 20, 8, (2, 10, 8), 0, 2)
    _, p2 = create(L, [d], pool=(4, 6))
    _, p3 = create(L, [desc(0, 20, 8, (2, 10, 8), 0, 2)], pool=(6, 4))
    _, p4 = create(L, [desc(0, 20, 8)])
    h = [L.gbo_desc_hash(p) for p in (p1, p2, p3, p4)]
    assert h[0] == h[1] and h[0] != h[2] and h[0] != h[3] and h[0] != 0
    for p in (p1, p2, p3, p4):
        L.gbo_muon_plan_destroy(p)
    assert L.gbo_desc_hash(None) == 0


def test_step_without_device_reports_error(L):
    """On a host without a GPU a step fails with a status, never silently."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("host has a GPU")
    _, plan = create(L, [desc(0, 8, 8)])
    rc = L.gbo_muon_step(plan, 0.02, FAKE, L.gbo_muon_workspace_bytes(plan), None, None, None)
    assert rc in (-7, -8)
    L.gbo_muon_plan_destroy(plan)
    # workspace too small is reported before any device call
    _, plan = create(L, [desc(0, 8, 8)])
    assert L.gbo_muon_step(plan, 0.02, FAKE, 16, None, None, None) == -6
    L.gbo_muon_plan_destroy(plan)


def test_h2d_copy_argument_refusals(L):
    """gbo_h2d_copy checks its arguments before it touches a device."""
    assert L.gbo_h2d_copy(FAKE, FAKE, 0, 0, None) == 0
    assert L.gbo_h2d_copy(FAKE, FAKE, -1, 0, None) == -1
    assert L.gbo_h2d_copy(FAKE, FAKE, 16, -1, None) == -1
    assert L.gbo_h2d_copy(None, FAKE, 16, 0, None) == -1
    assert L.gbo_h2d_copy(FAKE, None, 16, 0, None) == -1
    assert L.gbo_h2d_copy(FAKE + 8, FAKE, 16, 0, None) == -1
    assert L.gbo_h2d_copy(FAKE, FAKE + 4, 16, 0, None) == -1
    import torch
    if not torch.cuda.is_available():
        assert L.gbo_h2d_copy(FAKE, FAKE, 16, 4, None) in (-7, -8)


def test_free_sms_setting(L):
    """gbo_muon_plan_set_free_sms takes 0 .. 64 and refuses the rest."""
    _, plan = create(L, [desc(0, 8, 8)])
    assert L.gbo_muon_plan_set_free_sms(plan, 0) == 0
    assert L.gbo_muon_plan_set_free_sms(plan, 4) == 0
    assert L.gbo_muon_plan_set_free_sms(plan, 64) == 0
    assert L.gbo_muon_plan_set_free_sms(plan, -1) == -1
    assert L.gbo_muon_plan_set_free_sms(plan, 65) == -1
    assert L.gbo_muon_plan_set_free_sms(None, 4) == -1
    L.gbo_muon_plan_destroy(plan)


def test_fused_momentum_eligibility(L):
    """Which matrices run their momentum pass inside the chain launch: wide
    (rows <= cols) matrices of at most 128 rows on the on-chip Gram, with
    bf16 gradients whose rows start on 16-byte boundaries; a class runs it
    there only if every one of its matrices can.  Everything else keeps the
    momentum kernel (and its pre-normalisation launch)."""
    ok = lambda i: desc(i, 2 * 64, 512, (2, 64, 512))  # two 64 x 512 matrices
    rc, plan = create(L, [ok(0)])
    assert rc == 0 and info(L, plan).n_mom_fused == 0  # off by default
    L.gbo_muon_plan_destroy(plan)
    prev = L.gbo_testing_set_fused_momentum(1)
    try:
        _eligibility_cases(L, ok)
    finally:
        L.gbo_testing_set_fused_momentum(prev)


def _eligibility_cases(L, ok):
    rc, plan = create(L, [ok(0)])
    i = info(L, plan)
    assert rc == 0 and i.n_mom_fused == 2 and i.launches_per_step == 2
    L.gbo_muon_plan_destroy(plan)
    cases = {
        "fp32 gradient": lambda: [dict_desc(ok(0), g_dtype=B.GBO_F32)],
        "row not a multiple of 8": lambda: [desc(0, 64, 500)],
        "gradient off 16 bytes": lambda: [dict_desc(ok(0), g_off=8)],
        "tall": lambda: [desc(0, 512, 64)],
        "more than 128 rows": lambda: [desc(0, 160, 1024)],
    }
    for why, make in cases.items():
        rc, plan = create(L, make())
        i = info(L, plan)
        assert rc == 0 and i.n_mom_fused == 0, why
        L.gbo_muon_plan_destroy(plan)
    for kw in (dict(route=B.GBO_ROUTE_X), dict(precision=B.GBO_NS_F32)):
        rc, plan = create(L, [ok(0)], **kw)
        assert rc == 0 and info(L, plan).n_mom_fused == 0, kw
        L.gbo_muon_plan_destroy(plan)
    # one matrix of a class that cannot keeps the whole class on the momentum
    # kernel; another class still fuses (plus the momentum kernel and its
    # pre-normalisation launch for the rest)
    mixed = [ok(0), dict_desc(desc(1, 64, 512), g_dtype=B.GBO_F32), desc(2, 96, 1024)]
    rc, plan = create(L, mixed)
    i = info(L, plan)
    assert rc == 0 and i.n_matrices == 4 and i.n_mom_fused == 1
    L.gbo_muon_plan_destroy(plan)


def dict_desc(d, g_dtype=None, g_off=0):
    if g_dtype is not None:
        d.g_dtype = g_dtype
    if g_off:
        d.g = d.g + g_off
    return d


def test_workspace_cap_groups(L):
    """With a workspace cap the plan runs its table in groups of consecutive
    descriptors: the workspace it asks for fits the cap, the layout hash,
    matrix count and per-descriptor FLOPs are those of the whole table, the
    step takes more launches, and a descriptor that alone exceeds the cap is
    refused."""
    descs = lambda: [desc(i, 512 * (1 + i % 3), 1024) for i in range(9)]
    rc, whole = create(L, descs())
    assert rc == 0
    wi = info(L, whole)
    full = L.gbo_muon_workspace_bytes(whole)
    h = L.gbo_desc_hash(whole)
    f_whole = (ctypes.c_double * 9)()
    assert L.gbo_muon_plan_desc_flops(whole, f_whole, 9) == 0
    for frac in (2, 3, 5):
        cap = full // frac
        rc, plan = create(L, descs(), workspace_cap=cap)
        assert rc == 0, B.gbo_last_error()
        i = info(L, plan)
        ws = L.gbo_muon_workspace_bytes(plan)
        assert 0 < ws <= cap
        assert L.gbo_desc_hash(plan) == h and i.n_matrices == wi.n_matrices
        assert i.launches_per_step > wi.launches_per_step
        f = (ctypes.c_double * 9)()
        assert L.gbo_muon_plan_desc_flops(plan, f, 9) == 0 and list(f) == list(f_whole)
        L.gbo_muon_plan_destroy(plan)
    # a cap the whole table fits: one schedule, as without a cap
    rc, plan = create(L, descs(), workspace_cap=full)
    assert rc == 0 and info(L, plan).launches_per_step == wi.launches_per_step
    assert L.gbo_muon_workspace_bytes(plan) == full
    L.gbo_muon_plan_destroy(plan)
    # below what one descriptor needs: refused
    rc, plan = create(L, descs(), workspace_cap=1024)
    assert rc == -6 and not plan and "above the cap" in B.gbo_last_error()  # GBO_ERR_WORKSPACE
    rc, plan = create(L, descs(), workspace_cap=-1)
    assert rc == -1  # GBO_ERR_INVALID_ARG
    L.gbo_muon_plan_destroy(whole)
