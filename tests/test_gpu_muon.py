"""GPU parity of the Muon path against the fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
from adamw_optimizer_step_gb300 import _binding as B
from adamw_optimizer_step_gb300 import workloads as wk
from tests.parity import (TOL, check_muon, f64, random_entries, rel_fro, run_muon_gpu,
                          run_muon_oracle)
from oracle.views import sub_matrices

pytestmark = pytest.mark.gpu

CUBIC = (1.5, -0.5, 0.0)
QUINTIC = (15.0 / 8.0, -5.0 / 4.0, 3.0 / 8.0)


@pytest.fixture(scope="module", autouse=True)
def built():
    from adamw_optimizer_step_gb300 import build
    build.build()
    B.lib()


def tiny_entries():
    wl = wk.workload(1)
    out = []
    for i, t in enumerate(wl.muon):
        W, G, Bm, v = wk.muon_tensor_inputs(wl, i)
        out.append(dict(w=W, g=G, mom=Bm, row_v=v, view=t.view, split=t.split))
    return out, wl


@pytest.mark.parametrize("precision", ["f32", "bf16"])
def test_tiny_views(precision):
    """The tiny fp32 set of the pages' worked views, four 64x64 and two
    64x128 matrices: one step, every matrix checked."""
    entries, wl = tiny_entries()
    gpu, status, _ = run_muon_gpu(entries, lr=wl.lr, precision=precision)
    ora = run_muon_oracle(entries, lr=wl.lr)
    assert status == 0
    check_muon(entries, gpu, ora, lr=wl.lr, precision=precision)


RAGGED = [
    (300, 700, None, None),
    (700, 300, None, None),
    (129, 257, None, None),
    (257, 129, None, None),
    (1, 300, None, None),
    (300, 1, None, None),
    (1000, 64, (4, 250, 64), None),
    (640, 192, (2, 5, 64, 192), (20, 44)),
    (520, 136, (2, 260, 136), (100, 160), 0.5, 0.1),
]


@pytest.mark.parametrize("precision", ["f32", "bf16"])
@pytest.mark.parametrize("wdt", [torch.bfloat16, torch.float32])
def test_ragged_multi_tile(precision, wdt):
    """Shapes spanning several GEMM and momentum tiles with ragged tails,
    both orientations, degenerate 1 x n / m x 1, views with splits."""
    entries = random_entries(RAGGED, seed=11, w_dtype=wdt, g_dtype=wdt, b_std=1e-3)
    gpu, status, _ = run_muon_gpu(entries, lr=0.02, precision=precision)
    ora = run_muon_oracle(entries, lr=0.02)
    assert status == 0
    check_muon(entries, gpu, ora, lr=0.02, precision=precision)


@pytest.mark.parametrize("precision", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [
    dict(abc=QUINTIC),
    dict(abc=CUBIC + QUINTIC + (2.0, -1.5, 0.5) + CUBIC + (1.2, -0.3, 0.1)),
    dict(abc=CUBIC, ns_steps=1),
    dict(abc=CUBIC, ns_steps=8),
    dict(abc=CUBIC, nesterov=False),
    dict(abc=CUBIC, mu=0.8),
])
def test_coefficients_and_options(precision, opts):
    shapes = [(200, 72, None, None), (72, 200, None, None), (96, 96, None, None, 2.0, 0.05)]
    entries = random_entries(shapes, seed=12, b_std=1e-3)
    kw = dict(opts)
    gpu, status, _ = run_muon_gpu(entries, lr=0.05, precision=precision, **kw)
    ora = run_muon_oracle(entries, lr=0.05, **kw)
    assert status == 0
    check_muon(entries, gpu, ora, lr=0.05, precision=precision, mu=kw.get("mu", 0.95))


@pytest.mark.parametrize("precision", ["bf16", "f32"])
@pytest.mark.parametrize("route", ["x", "gram"])
@pytest.mark.parametrize("ns_steps", [2, 3, 5, 8])
def test_routes(route, ns_steps, precision):
    """Both routes reach the oracle's k-step result in both precisions: the
    X route, and the Gram route forced on every shape (square, tall, 1 x n
    and split views included), for short and long k (the Gram route rotates
    its P and Q buffers by iteration)."""
    entries = random_entries(RAGGED, seed=21, b_std=1e-3)
    r = B.GBO_ROUTE_X if route == "x" else B.GBO_ROUTE_GRAM
    gpu, status, plan = run_muon_gpu(entries, lr=0.02, precision=precision, ns_steps=ns_steps, route=r)
    info = B.gbo_muon_plan_info(plan)
    assert info["n_gram_route"] == (0 if route == "x" else info["n_matrices"])
    ora = run_muon_oracle(entries, lr=0.02, ns_steps=ns_steps)
    assert status == 0
    check_muon(entries, gpu, ora, lr=0.02, precision=precision)


@pytest.mark.parametrize("precision", ["f32", "bf16"])
def test_normuon_rms_target(precision):
    """NorMuon with the RMS-keeping scale: statistics pass, per-matrix
    scale, write pass.  Parity with the oracle, and each matrix of the
    exported update (a split view included) has RMS rho."""
    shapes = [(300, 130, None, None), (130, 300, None, None), (64, 64, None, None, 1.5, 0.1),
              (200, 40, (2, 100, 40), (30, 70))]
    entries = random_entries(shapes, seed=23, normuon=True, b_std=1e-3)
    kw = dict(normuon=True, beta2=0.95, eps=1e-8, rms_target=0.2)
    gpu, status, plan = run_muon_gpu(entries, lr=0.02, precision=precision, **kw)
    ora = run_muon_oracle(entries, lr=0.02, **kw)
    assert status == 0
    check_muon(entries, gpu, ora, lr=0.02, precision=precision)
    for e, g in zip(entries, gpu):
        U = g["U"].double().numpy()
        rows, cols = U.shape
        for r0, m, n in sub_matrices(rows, cols, e.get("view"), e.get("split")):
            blk = U[r0:r0 + m]
            assert abs(np.sqrt(np.mean(blk * blk)) / 0.2 - 1.0) < 1e-3


@pytest.mark.parametrize("precision", ["bf16", "f32"])
@pytest.mark.parametrize("route", ["x", "gram"])
@pytest.mark.parametrize("abc", ["quintic", "schedule"])
def test_routes_with_square(route, precision, abc):
    """Iterations with c != 0 (P = a I + b A + c A^2, one square of A) on
    both routes: the textbook quintic triple, and a per-step schedule that
    mixes c == 0 and c != 0 iterations."""
    coeffs = QUINTIC if abc == "quintic" else CUBIC + QUINTIC + (2.0, -1.5, 0.5) + CUBIC + (1.2, -0.3, 0.1)
    entries = random_entries(RAGGED, seed=24, b_std=1e-3)
    r = B.GBO_ROUTE_X if route == "x" else B.GBO_ROUTE_GRAM
    gpu, status, plan = run_muon_gpu(entries, lr=0.02, precision=precision, abc=coeffs, route=r)
    info = B.gbo_muon_plan_info(plan)
    assert info["n_gram_route"] == (0 if route == "x" else info["n_matrices"])
    ora = run_muon_oracle(entries, lr=0.02, abc=coeffs)
    assert status == 0
    check_muon(entries, gpu, ora, lr=0.02, precision=precision)


SMALL = [(4 * 96, 1000, (4, 96, 1000), None), (300, 100, None, None), (40, 300, None, None),
         (128, 512, None, None), (640, 192, (2, 5, 64, 192), (20, 44)),
         (2 * 192, 1536, (2, 192, 1536), None), (700, 150, None, None), (129, 600, None, None),
         (2 * 160, 900, (2, 160, 900), None)]


@pytest.mark.parametrize("abc,ns_steps", [
    (CUBIC, 5), (CUBIC, 2), (QUINTIC, 3), (CUBIC, 16),
    (CUBIC + QUINTIC + (2.0, -1.5, 0.5) + CUBIC + (1.2, -0.3, 0.1), 5),
])
def test_small_chain_matches_launches(abc, ns_steps):
    """Matrices of at most 192 rows on the Gram route, three ways: one
    launch per p x p product; the on-chip chain (one launch for all p x p
    products) after a Gram launch; and, for the wide matrices of at most 128
    rows, the chain starting from X_0 (its Gram streamed through shared
    memory in the same launch).  p = 20 .. 192 (one and two 128-row halves),
    wide and tall, c == 0 and c != 0, k = 2 .. 16 (up to 32 ops a matrix,
    barrier phases over many products and X_0 blocks).  All round every
    p x p result to bf16 once; the launches mirror symmetric results from
    their upper triangle and the chain writes them whole, so they agree to
    bf16 rounding (1e-2 relative per weight, ten times inside the oracle
    tolerance) and all match the oracle."""
    entries = random_entries(SMALL, seed=31, b_std=1e-3)
    kw = dict(lr=0.02, precision="bf16", abc=abc, ns_steps=ns_steps, route=B.GBO_ROUTE_GRAM)
    prev = B.gbo_testing_set_small_chain(False)
    try:
        ref, st0, plan0 = run_muon_gpu(entries, **kw)
    finally:
        B.gbo_testing_set_small_chain(prev)
    B.gbo_testing_set_small_chain(True)
    prev_fused = B.gbo_testing_set_fused_gram(False)
    try:
        sep, st1, plan1 = run_muon_gpu(entries, **kw)
    finally:
        B.gbo_testing_set_fused_gram(prev_fused)
    B.gbo_testing_set_fused_gram(True)
    try:
        gpu, st2, plan2 = run_muon_gpu(entries, **kw)
    finally:
        B.gbo_testing_set_small_chain(prev)
        B.gbo_testing_set_fused_gram(prev_fused)
    assert st0 == 0 and st1 == 0 and st2 == 0
    n0, n1, n2 = (B.gbo_muon_plan_info(q)["launches_per_step"] for q in (plan0, plan1, plan2))
    assert n2 <= n1 < n0
    for a, b, c in zip(ref, sep, gpu):
        assert rel_fro(f64(b["U"]), f64(a["U"])) <= 1e-2
        assert rel_fro(f64(c["U"]), f64(a["U"])) <= 1e-2
    ora = run_muon_oracle(entries, lr=0.02, abc=abc, ns_steps=ns_steps)
    check_muon(entries, ref, ora, lr=0.02, precision="bf16")
    check_muon(entries, sep, ora, lr=0.02, precision="bf16")
    check_muon(entries, gpu, ora, lr=0.02, precision="bf16")


# eleven shape classes of at most 128 rows (p = 8 .. 127), wide and tall,
# with K ragged (q = 48 .. 1000): two launches of the chain with its Gram on
# chip, eight classes to a launch
CHAIN_CLASSES = [(8, 200, None, None), (200, 8, None, None), (24, 72, None, None), (130, 60, None, None),
                 (64, 64, None, None), (100, 1000, None, None), (1000, 100, None, None),
                 (127, 129, None, None), (129, 127, None, None), (2 * 40, 520, (2, 40, 520), None),
                 (3 * 16, 48, (3, 16, 48), None)]


@pytest.mark.parametrize("abc", [CUBIC, QUINTIC])
def test_chain_gram_launch_groups(abc):
    """The chain with its Gram on chip over two launches (classes 1-8 and
    9-11) against the same chain after a Gram launch of its own (agreement
    to bf16 rounding) and against the oracle."""
    entries = random_entries(CHAIN_CLASSES, seed=37, b_std=1e-3)
    kw = dict(lr=0.02, precision="bf16", abc=abc, ns_steps=5, route=B.GBO_ROUTE_GRAM)
    prev = B.gbo_testing_set_fused_gram(False)
    try:
        sep, st1, plan1 = run_muon_gpu(entries, **kw)
    finally:
        B.gbo_testing_set_fused_gram(prev)
    # the chain streaming X_0 for every class: classes 1-8 and 9-11
    prev_mom = B.gbo_testing_set_fused_momentum(False)
    try:
        x0s, st2, plan2 = run_muon_gpu(entries, **kw)
    finally:
        B.gbo_testing_set_fused_momentum(prev_mom)
    # the six wide classes on 16-byte rows stream G and B (one launch), the
    # other five X_0 (another)
    prev_mom = B.gbo_testing_set_fused_momentum(True)
    try:
        gpu, st3, plan3 = run_muon_gpu(entries, **kw)
    finally:
        B.gbo_testing_set_fused_momentum(prev_mom)
    assert st1 == 0 and st2 == 0 and st3 == 0
    assert B.gbo_muon_plan_info(plan2)["launches_per_step"] == 2 + 2 + 2
    assert B.gbo_muon_plan_info(plan3)["launches_per_step"] == 2 + 2 + 2
    assert B.gbo_muon_plan_info(plan3)["n_mom_fused"] == 1 + 1 + 1 + 1 + 2 + 3
    for a, b, c in zip(sep, x0s, gpu):
        assert rel_fro(f64(b["U"]), f64(a["U"])) <= 1e-2
        assert rel_fro(f64(c["U"]), f64(a["U"])) <= 1e-2
    ora = run_muon_oracle(entries, lr=0.02, abc=abc, ns_steps=5)
    check_muon(entries, x0s, ora, lr=0.02, precision="bf16")
    check_muon(entries, gpu, ora, lr=0.02, precision="bf16")


# wide matrices of at most 128 rows with bf16 gradients on 16-byte rows: the
# chain kernel runs their momentum pass (G and B streamed in 64-column
# stages); rows 1 .. 128, K ragged against the stages (q = 8 .. 4104), split
# views whose row blocks start mid-weight, plus classes that stay on the
# momentum kernel (a tall one, a row of 300 elements) in the same step
FUSED_MOM = [(1, 64, None, None), (3 * 7, 8, (3, 7, 8), None), (128, 4104, None, None), (96, 1000, None, None),
             (2 * 100, 520, (2, 100, 520), (37, 63)), (64, 64, None, None), (5 * 24, 72, (5, 24, 72), None),
             (300, 100, None, None), (40, 300, None, None)]


@pytest.mark.parametrize("nesterov", [True, False])
def test_fused_momentum_matches_momentum_kernel(nesterov):
    """Two steps from a nonzero momentum with the momentum pass inside the
    chain launch, against the same steps with it in the momentum kernel: the
    momentum buffers bitwise equal (the same fp32 operations per element),
    the updates equal to bf16 rounding (the pre-normalisation factor is
    reduced in another fixed order), and both match the oracle."""
    entries = random_entries(FUSED_MOM, seed=41, b_std=1e-3)
    kw = dict(lr=0.02, precision="bf16", steps=2, nesterov=nesterov, route=B.GBO_ROUTE_GRAM)
    prev = B.gbo_testing_set_fused_momentum(False)
    try:
        ref, st0, plan0 = run_muon_gpu(entries, **kw)
    finally:
        B.gbo_testing_set_fused_momentum(prev)
    B.gbo_testing_set_fused_momentum(True)
    try:
        gpu, st1, plan1 = run_muon_gpu(entries, **kw)
    finally:
        B.gbo_testing_set_fused_momentum(prev)
    assert st0 == 0 and st1 == 0
    i0, i1 = B.gbo_muon_plan_info(plan0), B.gbo_muon_plan_info(plan1)
    assert i0["n_mom_fused"] == 0 and i1["n_mom_fused"] == 1 + 3 + 1 + 1 + 4 + 1 + 5
    for a, b in zip(ref, gpu):
        assert torch.equal(a["B"], b["B"])
        assert rel_fro(f64(b["U"]), f64(a["U"])) <= 1e-2
        assert rel_fro(f64(b["W"]), f64(a["W"])) <= 1e-2
    # one step of the fused path against the oracle (every acceptance check)
    B.gbo_testing_set_fused_momentum(True)
    try:
        one, st2, plan2 = run_muon_gpu(entries, **dict(kw, steps=1))
    finally:
        B.gbo_testing_set_fused_momentum(prev)
    assert B.gbo_muon_plan_info(plan2)["n_mom_fused"] == i1["n_mom_fused"]
    assert st2 == 0
    ora = run_muon_oracle(entries, lr=0.02, nesterov=nesterov)
    check_muon(entries, one, ora, lr=0.02, precision="bf16")


@pytest.mark.parametrize("normuon", [False, True])
def test_workspace_cap_bitwise(normuon):
    """A workspace cap runs the table in groups of consecutive weights on one
    smaller workspace: weights, momentum, row moments and the exported
    update are bitwise those of the uncapped plan (every matrix is computed
    the same way), and match the oracle."""
    shapes = [(600, 130, None, None), (130, 600, None, None), (256, 256, None, None), (4 * 96, 1000, (4, 96, 1000), None),
              (200, 40, (2, 100, 40), (30, 70)), (2 * 192, 1536, (2, 192, 1536), None), (128, 512, None, None)]
    entries = random_entries(shapes, seed=43, normuon=normuon, b_std=1e-3)
    kw = dict(lr=0.02, precision="bf16", steps=2, normuon=normuon, beta2=0.95, eps=1e-8)
    ref, st0, plan0 = run_muon_gpu(entries, **kw)
    full = B.gbo_muon_workspace_bytes(plan0)
    gpu, st1, plan1 = run_muon_gpu(entries, workspace_cap=full // 2, **kw)
    assert st0 == 0 and st1 == 0
    assert 0 < B.gbo_muon_workspace_bytes(plan1) <= full // 2
    assert B.gbo_muon_plan_info(plan1)["launches_per_step"] > B.gbo_muon_plan_info(plan0)["launches_per_step"]
    for a, b in zip(ref, gpu):
        assert torch.equal(a["W"], b["W"]) and torch.equal(a["B"], b["B"]) and torch.equal(a["U"], b["U"])
        if normuon:
            assert torch.equal(a["v"], b["v"])
    one, st2, _ = run_muon_gpu(entries, workspace_cap=full // 2, **dict(kw, steps=1))
    assert st2 == 0
    ora = run_muon_oracle(entries, lr=0.02, normuon=normuon, beta2=0.95, eps=1e-8)
    check_muon(entries, one, ora, lr=0.02, precision="bf16")


@pytest.mark.parametrize("ns_steps", [3, 5])
def test_normuon_gram_route(ns_steps):
    """NorMuon rows read the last iterate from the buffer each route leaves
    it in: mixed X-route (square, above the chain's 192 rows) and Gram-route
    (rectangular) classes."""
    shapes = [(600, 130, None, None), (130, 600, None, None), (256, 256, None, None)]
    entries = random_entries(shapes, seed=22, normuon=True, b_std=1e-3)
    gpu, status, plan = run_muon_gpu(entries, lr=0.02, precision="bf16", normuon=True, beta2=0.95, eps=1e-8,
                                     ns_steps=ns_steps)
    assert B.gbo_muon_plan_info(plan)["n_gram_route"] == 2
    ora = run_muon_oracle(entries, lr=0.02, normuon=True, beta2=0.95, eps=1e-8, ns_steps=ns_steps)
    assert status == 0
    check_muon(entries, gpu, ora, lr=0.02, precision="bf16")


@pytest.mark.parametrize("precision", ["f32", "bf16"])
def test_normuon_rows(precision):
    shapes = [(300, 130, None, None), (130, 300, None, None), (64, 64, None, None),
              (200, 40, (2, 100, 40), (30, 70))]
    entries = random_entries(shapes, seed=13, normuon=True, b_std=1e-3)
    gpu, status, _ = run_muon_gpu(entries, lr=0.02, precision=precision, normuon=True, beta2=0.95, eps=1e-8)
    ora = run_muon_oracle(entries, lr=0.02, normuon=True, beta2=0.95, eps=1e-8)
    assert status == 0
    check_muon(entries, gpu, ora, lr=0.02, precision=precision)


@pytest.mark.parametrize("rms_target", [0.0, 0.2])
def test_normuon_streamed_write(rms_target):
    """bf16 weights whose rows all start on 16-byte boundaries take the
    streamed write pass (a statistics pass, then rows streamed through
    shared memory in 512-element segments): rows longer and shorter than a
    segment, ragged tails, wide and tall, X and Gram routes, a split view,
    with and without the RMS-keeping scale, from a nonzero v."""
    shapes = [(256, 4104, None, None), (4104, 256, None, None), (96, 96, None, None),
              (240, 512, (2, 120, 512), (40, 80)), (300, 2048, None, None, 1.5, 0.05)]
    entries = random_entries(shapes, seed=27, normuon=True, b_std=1e-3)
    kw = dict(normuon=True, beta2=0.95, eps=1e-8, rms_target=rms_target)
    gpu, status, plan = run_muon_gpu(entries, lr=0.02, precision="bf16", **kw)
    if not rms_target:  # one launch more than the single rows kernel: the statistics pass
        fp32w = [dict(e, w=e["w"].float()) for e in entries]
        _, _, plan32 = run_muon_gpu(fp32w, lr=0.02, precision="bf16", **kw)
        assert (B.gbo_muon_plan_info(plan)["launches_per_step"]
                == B.gbo_muon_plan_info(plan32)["launches_per_step"] + 1)
    ora = run_muon_oracle(entries, lr=0.02, **kw)
    assert status == 0
    check_muon(entries, gpu, ora, lr=0.02, precision="bf16")


@pytest.mark.parametrize("precision", ["bf16", "f32"])
@pytest.mark.parametrize("route", ["x", "gram"])
def test_skip_zero_and_nonfinite(route, precision):
    """Inactive weights stay untouched, a zero gradient gives a pure decay
    step (A_0 = 0 on the Gram route: Q_k = a^k I times a zero X_0), and a NaN
    gradient is reported in the status word, on both routes."""
    r = B.GBO_ROUTE_X if route == "x" else B.GBO_ROUTE_GRAM
    shapes = [(64, 96, None, None), (48, 48, None, None, 1.0, 0.1), (32, 32, None, None)]
    entries = random_entries(shapes, seed=14, b_std=0.0)
    entries[0]["g"] = None                        # inactive: untouched
    entries[1]["g"] = torch.zeros_like(entries[1]["g"])  # zero direction: pure decay
    gpu, status, _ = run_muon_gpu(entries, lr=0.1, precision=precision, route=r)
    assert status == 0
    assert torch.equal(gpu[0]["W"], entries[0]["w"]) and torch.equal(gpu[0]["B"], entries[0]["mom"])
    assert torch.count_nonzero(gpu[1]["U"]) == 0
    want = (entries[1]["w"].double() * (1 - 0.1 * 0.1)).to(entries[1]["w"].dtype)
    assert torch.equal(gpu[1]["W"], want)
    # a NaN gradient is reported in the status word
    bad = random_entries([(32, 32, None, None)], seed=15)
    bad[0]["g"][3, 4] = float("nan")
    _, status, _ = run_muon_gpu(bad, lr=0.1, precision=precision, route=r)
    assert status & B.GBO_STATUS_NONFINITE


@pytest.mark.parametrize("pdl", [0, 1, 2])
@pytest.mark.parametrize("precision", ["bf16", "f32"])
def test_cuda_graph_replay(precision, pdl):
    """Once a first call has set the plan up on the device, a Muon step
    captured in a CUDA graph replays the same launches: one direct step, a
    capture and three replays give bitwise the state of four direct steps,
    with programmatic dependent launch never, always or (the default) in
    the capture only."""
    prev = B.gbo_testing_set_pdl(pdl)
    try:
        _graph_replay_case(precision)
    finally:
        B.gbo_testing_set_pdl(prev)


def _graph_replay_case(precision):
    shapes = [(300, 700, None, None), (700, 300, None, None), (64, 64, None, None),
              (200, 40, (2, 100, 40), (30, 70))]
    entries = random_entries(shapes, seed=31, b_std=1e-3)
    prec = B.GBO_NS_F32 if precision == "f32" else B.GBO_NS_BF16

    def make():
        dev = [{k: (v.cuda().clone() if torch.is_tensor(v) else v) for k, v in e.items()} for e in entries]
        plan = B.gbo_muon_plan_create(dev, precision=prec)
        ws = torch.empty(max(1, B.gbo_muon_workspace_bytes(plan)), dtype=torch.uint8, device="cuda")
        return dev, plan, ws, torch.zeros(1, dtype=torch.int32, device="cuda")

    dev_a, plan_a, ws_a, st_a = make()
    dev_b, plan_b, ws_b, st_b = make()
    for _ in range(4):
        B.gbo_muon_step(plan_a, 0.02, ws_a, dev_status=st_a)
    B.gbo_muon_step(plan_b, 0.02, ws_b, dev_status=st_b)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.gbo_muon_step(plan_b, 0.02, ws_b, dev_status=st_b)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert int(st_a.item()) == 0 and int(st_b.item()) == 0
    for a, b in zip(dev_a, dev_b):
        assert torch.equal(a["w"], b["w"]) and torch.equal(a["mom"], b["mom"])


@pytest.mark.parametrize("precision", ["f32", "bf16"])
def test_deterministic(precision):
    entries = random_entries([(384, 260, None, None), (260, 384, None, None)], seed=16, b_std=1e-3)
    a, _, _ = run_muon_gpu(entries, lr=0.02, precision=precision)
    b, _, _ = run_muon_gpu(entries, lr=0.02, precision=precision)
    for x, y in zip(a, b):
        assert torch.equal(x["W"], y["W"]) and torch.equal(x["B"], y["B"]) and torch.equal(x["U"], y["U"])


def test_checkpoint_resume_bitwise():
    """Five steps straight equal three steps, a save/reload of weights and
    state into fresh buffers and a new plan, then two more steps."""
    entries = random_entries([(256, 160, None, None), (160, 256, (2, 80, 256), (30, 50))], seed=17,
                             normuon=True)
    straight, _, p1 = run_muon_gpu(entries, lr=0.02, precision="bf16", steps=5, normuon=True)
    mid, _, p2 = run_muon_gpu(entries, lr=0.02, precision="bf16", steps=3, normuon=True)
    resumed = []
    for e, m in zip(entries, mid):
        d = dict(e)
        d.update(w=m["W"].clone(), mom=m["B"].clone(), row_v=m["v"].clone())
        resumed.append(d)
    end, _, p3 = run_muon_gpu(resumed, lr=0.02, precision="bf16", steps=2, normuon=True)
    assert B.gbo_desc_hash(p1) == B.gbo_desc_hash(p3)
    for s, r in zip(straight, end):
        assert torch.equal(s["W"], r["W"]) and torch.equal(s["B"], r["B"]) and torch.equal(s["v"], r["v"])


def test_layer_d2048_full_size():
    """One d=2048 layer (Q, K, V, O 2048^2, gate_up (2, 5632, 2048), down
    2048 x 5632): step 1 checked on every matrix; ten consecutive steps run
    with the same gradients, the tenth checked on the gate matrix."""
    wl = wk.workload(2)
    entries = []
    for i, t in enumerate(wl.muon):
        W, G, Bm, v = wk.muon_tensor_inputs(wl, i)
        entries.append(dict(w=W, g=G, mom=Bm, view=t.view, split=t.split))
    gpu, status, _ = run_muon_gpu(entries, lr=wl.lr, precision="bf16")
    assert status == 0
    ora = run_muon_oracle(entries, lr=wl.lr)
    worst = check_muon(entries, gpu, ora, lr=wl.lr, precision="bf16")
    print("layer d2048 worst rel Frobenius error", worst)
    ten, status, _ = run_muon_gpu(entries, lr=wl.lr, precision="bf16", steps=10)
    assert status == 0
    e = entries[4]
    G = f64(e["g"])
    Bm = np.zeros_like(G)
    for _ in range(10):
        Bm = oracle.momentum_update(Bm, G, 0.95)
    D = oracle.nesterov_direction(G, Bm, 0.95)
    O = oracle.orthogonalize(D[:5632], [CUBIC] * 5) * oracle.rect_scale(5632, 2048)
    assert rel_fro(f64(ten[4]["U"])[:5632], O) <= TOL["bf16"]
    assert np.max(np.abs(f64(ten[4]["B"]) - Bm)) <= 1e-6 * np.max(np.abs(Bm))


def _sampled_large(idx, n_random=2, normuon=False):
    """Full-size workload generated on the device; every distinct matrix
    shape plus a few seeded random matrices are compared to the oracle."""
    wl = wk.workload(idx)
    dev = []
    for i, t in enumerate(wl.muon):
        W, G, Bm, v = wk.muon_tensor_inputs(wl, i, device="cuda")
        dev.append(dict(w=W, g=G, mom=Bm, row_v=v, view=t.view, split=t.split))
    originals = {}
    shapes = {}
    for i, t in enumerate(wl.muon):
        for r0, m, n in sub_matrices(t.rows, t.cols, t.view, t.split):
            shapes.setdefault((m, n), (i, r0))
    rng = np.random.default_rng(1000 + idx)
    picks = list(shapes.values())
    for _ in range(n_random):
        i = int(rng.integers(len(wl.muon)))
        t = wl.muon[i]
        subs = sub_matrices(t.rows, t.cols, t.view, t.split)
        picks.append((i, subs[int(rng.integers(len(subs)))][0]))
    for i, _ in picks:
        if i not in originals:
            e = dev[i]
            originals[i] = dict(w=e["w"].cpu(), g=e["g"].cpu(), mom=e["mom"].cpu(),
                                row_v=None if e["row_v"] is None else e["row_v"].cpu())
    plan = B.gbo_muon_plan_create(dev, normuon=normuon)
    ws = torch.empty(B.gbo_muon_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    offs = np.cumsum([0] + [t.numel for t in wl.muon])
    U = torch.empty(int(offs[-1]), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.gbo_muon_step(plan, wl.lr, ws, dbg_update=U, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i, r0 in picks:
        t = wl.muon[i]
        m = [s for s in sub_matrices(t.rows, t.cols, t.view, t.split) if s[0] == r0][0][1]
        o = originals[i]
        G = f64(o["g"])[r0:r0 + m]
        Bn = oracle.momentum_update(f64(o["mom"])[r0:r0 + m], G, 0.95)
        D = oracle.nesterov_direction(G, Bn, 0.95)
        O = oracle.orthogonalize(D, [CUBIC] * 5)
        if normuon:
            O, _ = oracle.normuon_rows(O, f64(o["row_v"])[r0:r0 + m], 0.95, 1e-8)
        O = O * oracle.rect_scale(m, t.cols)
        Ug = U[int(offs[i]) + r0 * t.cols: int(offs[i]) + (r0 + m) * t.cols].view(m, t.cols).cpu().double().numpy()
        err = rel_fro(Ug, O)
        print("workload %d matrix %s rows %d+%d: rel err %.3e" % (idx, t.name, r0, m, err))
        assert err <= TOL["bf16"]
        Bg = dev[i]["mom"][r0:r0 + m].cpu().double().numpy()
        assert np.all(np.abs(Bg - Bn) <= 1e-6 * (np.abs(G) + 1e-30))
    del dev, ws, U
    torch.cuda.empty_cache()


def test_omn_shaped_sampled():
    _sampled_large(3)


def test_many_small_sampled():
    _sampled_large(4, n_random=4)


def test_normuon_7b_sampled():
    _sampled_large(5, n_random=1, normuon=True)


def test_standalone_rownorm():
    gen = torch.Generator().manual_seed(21)
    O = torch.randn(77, 300, generator=gen)
    v = torch.rand(77, generator=gen) * 1e-2
    W = (torch.randn(77, 300, generator=gen) * 0.02).to(torch.bfloat16)
    Od, vd, Wd = O.cuda(), v.cuda(), W.cuda()
    U = torch.empty(77, 300, device="cuda")
    B.gbo_normuon_rownorm(Od, vd, Wd, beta2=0.95, eps=1e-8, scale=1.5, lr=0.02, wd=0.1, dbg_update=U)
    torch.cuda.synchronize()
    N, v_new = oracle.normuon_rows(f64(O), f64(v), 0.95, 1e-8)
    assert np.max(np.abs(f64(vd) - v_new) / v_new) < 1e-5
    assert rel_fro(f64(U), 1.5 * N) < 1e-5
    want = f64(W) - 0.02 * (0.1 * f64(W) + f64(U))
    assert np.max(np.abs(f64(Wd) - want)) <= 2 ** -7 * np.max(np.abs(want))


def test_after_momentum_event_and_side_stream():
    """An event recorded after the momentum phase lets another stream start
    (here: a copy of the updated momentum); results match a plain step.  The
    third weight's momentum pass runs in the chain launch, after which the
    event is recorded."""
    entries = random_entries([(256, 160, None, None), (160, 256, None, None), (128, 512, None, None)], seed=31,
                             b_std=1e-3)
    plain, _, _ = run_muon_gpu(entries, lr=0.02, precision="bf16")
    dev = []
    for e in entries:
        d = dict(e)
        for k in ("w", "g", "mom"):
            d[k] = d[k].cuda()
        dev.append(d)
    prev = B.gbo_testing_set_fused_momentum(True)
    try:
        plan = B.gbo_muon_plan_create(dev)
    finally:
        B.gbo_testing_set_fused_momentum(prev)
    ev = torch.cuda.Event()
    B.gbo_muon_plan_set_event(plan, 0, ev)
    ws = torch.empty(B.gbo_muon_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    B.gbo_muon_step(plan, 0.02, ws)
    side.wait_event(ev)
    with torch.cuda.stream(side):
        mom_copy = [d["mom"].clone() for d in dev]
    torch.cuda.synchronize()
    assert B.gbo_muon_plan_info(plan)["n_mom_fused"] == 1
    for m, p in zip(mom_copy, plain):
        assert torch.equal(m, p["B"].cuda())
    for d, p in zip(dev, plain):
        assert torch.equal(d["w"].cpu(), p["W"]) and torch.equal(d["mom"].cpu(), p["B"])
    B.gbo_muon_plan_set_event(plan, 0, None)


TAIL_SPLIT = [(1024, 1024, None, None), (2048, 2048, None, None), (384, 1536, None, None),
              (1536, 384, None, None), (1000, 700, None, None), (700, 1000, None, None),
              (3 * 320, 1280, (3, 320, 1280), None, 1.0, 0.1)]


@pytest.mark.parametrize("normuon", [False, True])
@pytest.mark.parametrize("shape", TAIL_SPLIT, ids=lambda s: "%dx%d" % s[:2])
def test_tail_split_bitwise(shape, normuon):
    """A weight alone in its plan gives launches of at most a few dozen CTA-pair
    tiles, so most run as 256 x 128 halves (Gram, products, the weight-writing
    last product, both routes, tall and wide): weights, momentum, row moments
    and the exported update are bitwise those of whole tiles, and match the
    oracle."""
    entries = random_entries([shape], seed=47, normuon=normuon, b_std=1e-3)
    kw = dict(lr=0.02, precision="bf16", steps=2, normuon=normuon, beta2=0.95, eps=1e-8)
    prev = B.gbo_testing_set_tail_split(False)
    try:
        whole, st0, _ = run_muon_gpu(entries, **kw)
        B.gbo_testing_set_tail_split(True)
        split, st1, _ = run_muon_gpu(entries, **kw)
        one, st2, _ = run_muon_gpu(entries, **dict(kw, steps=1))
    finally:
        B.gbo_testing_set_tail_split(prev)
    assert st0 == 0 and st1 == 0 and st2 == 0
    for a, b in zip(whole, split):
        assert torch.equal(a["W"], b["W"]) and torch.equal(a["B"], b["B"]) and torch.equal(a["U"], b["U"])
        if normuon:
            assert torch.equal(a["v"], b["v"])
    ora = run_muon_oracle(entries, lr=0.02, normuon=normuon, beta2=0.95, eps=1e-8)
    check_muon(entries, one, ora, lr=0.02, precision="bf16")


@pytest.mark.parametrize("g_kind", ["bf16", "f32", "mixed", "unaligned"])
def test_momentum_stream_bitwise(g_kind):
    """The momentum pass streamed through shared memory (bf16 mode, every
    matrix on 16-byte rows) against the register kernel: weights, momentum
    and the exported update bitwise equal over two steps, with bf16, fp32
    and mixed G (24 KB and 32 KB stages), ragged last tiles, matrices much
    smaller than a tile, tile ranges crossing matrices, split views and more
    tiles per block than ring stages; a table with a row off the 16-byte
    grid takes the register kernel either way.  Both match the oracle."""
    shapes = [(2048, 2048, None, None), (1536, 384, None, None), (136, 1000, None, None, 1.0, 0.1),
              (8, 8, None, None), (4 * 96, 1000, (4, 96, 1000), None), (24, 4104, None, None),
              (2 * 192, 1536, (2, 192, 1536), None), (72, 64, None, None)]
    if g_kind == "unaligned":
        shapes.append((40, 100, None, None))
    entries = random_entries(shapes, seed=59, b_std=1e-3)
    if g_kind == "f32":
        for e in entries:
            e["g"] = e["g"].float()
    elif g_kind == "mixed":
        for e in entries[1::2]:
            e["g"] = e["g"].float()
    kw = dict(lr=0.02, precision="bf16", steps=2)
    prev = B.gbo_testing_set_momentum_stream(False)
    try:
        reg, st0, _ = run_muon_gpu(entries, **kw)
        B.gbo_testing_set_momentum_stream(True)
        streamed, st1, _ = run_muon_gpu(entries, **kw)
        one, st2, _ = run_muon_gpu(entries, **dict(kw, steps=1))
    finally:
        B.gbo_testing_set_momentum_stream(prev)
    assert st0 == 0 and st1 == 0 and st2 == 0
    for a, b in zip(reg, streamed):
        assert torch.equal(a["W"], b["W"]) and torch.equal(a["B"], b["B"]) and torch.equal(a["U"], b["U"])
    ora = run_muon_oracle(entries, lr=0.02)
    check_muon(entries, one, ora, lr=0.02, precision="bf16")


@pytest.mark.parametrize("table", ["large", "small"])
@pytest.mark.parametrize("g_kind", ["bf16", "mixed"])
def test_momentum_stream_many_tiles_per_block(g_kind, table):
    """Tens of tiles per block, so every consumer group's ring of the
    streamed momentum pass wraps many times (24 KB stages with bf16 G, 32 KB
    with an fp32 G in the table), with tiles dealt out across the blocks
    (three large matrices) or in contiguous ranges (300 matrices of 8 tiles
    and one of 1024, so block ranges cross many matrices): bitwise the
    register kernel's weights, momentum and update over three steps."""
    if table == "large":
        shapes = [(4096, 4096, None, None), (4096, 1024, None, None), (1000, 4096, None, None, 1.0, 0.1)]
    else:
        shapes = [(4096, 1024, None, None)] + [(64, 512, None, None)] * 300
    entries = random_entries(shapes, seed=61, b_std=1e-3)
    if g_kind == "mixed":
        entries[1]["g"] = entries[1]["g"].float()
    kw = dict(lr=0.02, precision="bf16", steps=3)
    prev = B.gbo_testing_set_momentum_stream(False)
    try:
        reg, st0, _ = run_muon_gpu(entries, **kw)
        B.gbo_testing_set_momentum_stream(True)
        streamed, st1, _ = run_muon_gpu(entries, **kw)
    finally:
        B.gbo_testing_set_momentum_stream(prev)
    assert st0 == 0 and st1 == 0
    for a, b in zip(reg, streamed):
        assert torch.equal(a["W"], b["W"]) and torch.equal(a["B"], b["B"]) and torch.equal(a["U"], b["U"])


@pytest.mark.parametrize("free_sms", [4, 37])
def test_free_sms_bitwise(free_sms):
    """A plan that leaves SMs free runs its persistent kernels on fewer CTAs
    (CTA pairs, single CTAs and the on-chip chain, with a workspace cap's
    groups): the results are bitwise those of the whole device."""
    shapes = [(2048, 2048, None, None), (1536, 384, None, None), (4 * 96, 1000, (4, 96, 1000), None),
              (2 * 192, 1536, (2, 192, 1536), None), (130, 600, None, None), (64, 64, None, None)]
    entries = random_entries(shapes, seed=53, b_std=1e-3)
    kw = dict(lr=0.02, precision="bf16", steps=2)
    whole, st0, plan0 = run_muon_gpu(entries, **kw)
    part, st1, _ = run_muon_gpu(entries, free_sms=free_sms, **kw)
    full = B.gbo_muon_workspace_bytes(plan0)
    capped, st2, plan2 = run_muon_gpu(entries, free_sms=free_sms, workspace_cap=int(full * 0.85), **kw)
    assert st0 == 0 and st1 == 0 and st2 == 0
    assert B.gbo_muon_plan_info(plan2)["launches_per_step"] > B.gbo_muon_plan_info(plan0)["launches_per_step"]
    for a, b, c in zip(whole, part, capped):
        for k in ("W", "B", "U"):
            assert torch.equal(a[k], b[k]) and torch.equal(a[k], c[k]), k


def test_prenorm_finalize_independent_of_block_size():
    """The pre-normalisation factors reduce each matrix's partials as 1024
    virtual lanes in a fixed tree, run by 256-thread blocks when the table
    has at least as many matrices as SMs and by 1024-thread blocks when it
    has fewer: a table of 170 matrices and the same table stepped in
    capped groups of fewer matrices give the same bits."""
    shapes = [(2048, 2048, None, None)] + [(96, 320, None, None)] * 168 + [(1024, 3000, None, None)]
    entries = random_entries(shapes, seed=59, b_std=1e-3)
    kw = dict(lr=0.02, precision="bf16", steps=1)
    whole, st0, plan0 = run_muon_gpu(entries, **kw)
    full = B.gbo_muon_workspace_bytes(plan0)
    groups, st1, plan1 = run_muon_gpu(entries, workspace_cap=int(full * 0.6), **kw)
    assert st0 == 0 and st1 == 0
    assert B.gbo_muon_plan_info(plan1)["launches_per_step"] > B.gbo_muon_plan_info(plan0)["launches_per_step"]
    for a, b in zip(whole, groups):
        for k in ("W", "B", "U"):
            assert torch.equal(a[k], b[k]), k
    ora = run_muon_oracle(entries[:1] + entries[-1:], lr=0.02)
    check_muon(entries[:1] + entries[-1:], whole[:1] + whole[-1:], ora, lr=0.02, precision="bf16")
