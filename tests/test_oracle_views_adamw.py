"""Pins for the oracle's view expansion, the per-tensor Muon step and the
AdamW path (CPU only)."""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import adamw as oa
from oracle import muon as om
from oracle.views import ViewError, sub_matrices

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")))


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# views: the pages' worked shapes

@pytest.mark.parametrize("case", GOLDEN["views"]["cases"])
def test_page_view_shapes(case):
    rows, cols = case["stored"]
    subs = sub_matrices(rows, cols, tuple(case["view"]), case["split"] and tuple(case["split"]))
    assert [[m, n] for _, m, n in subs] == case["matrices"]
    # the blocks tile the stored rows exactly once, in order
    starts = [r0 for r0, _, _ in subs]
    assert starts[0] == 0
    for (r0, m, _), nxt in zip(subs, starts[1:] + [rows]):
        assert r0 + m == nxt


@pytest.mark.parametrize("bad", [
    dict(rows=32, cols=8, view=(2, 15, 8)),        # product mismatch
    dict(rows=32, cols=8, view=(2, 16, 4)),        # column mismatch
    dict(rows=32, cols=8, view=(0, 16, 8)),        # non-positive entry
    dict(rows=32, cols=8, view=(-2, -16, 8)),
    dict(rows=20, cols=8, view=(2, 10, 8), split=(4, 5)),   # split sum
    dict(rows=20, cols=8, view=(2, 10, 8), split=(10, 0)),  # empty split
    dict(rows=0, cols=8),
])
def test_view_rules_refuse(bad):
    with pytest.raises(ViewError):
        sub_matrices(bad["rows"], bad["cols"], bad.get("view"), bad.get("split"))


def _step(W, G, B, **kw):
    return om.muon_step_tensor(W, G, B, **kw)


def test_fused_view_equals_independent_matrices():
    """gate_up (32, 8) viewed (2, 16, 8) updates like two separate (16, 8)
    weights; the unsplit (32, 8) update differs (negative control)."""
    W = rng(1).standard_normal((32, 8))
    G = rng(2).standard_normal((32, 8))
    B = rng(3).standard_normal((32, 8))
    fused = _step(W, G, B, view=(2, 16, 8))
    top = _step(W[:16], G[:16], B[:16])
    bot = _step(W[16:], G[16:], B[16:])
    assert np.max(np.abs(fused[0] - np.vstack([top[0], bot[0]]))) < 1e-15
    assert np.max(np.abs(fused[3] - np.vstack([top[3], bot[3]]))) < 1e-15
    whole = _step(W, G, B)
    assert np.max(np.abs(whole[3] - fused[3])) > 1e-2
    # (16, 8) is tall: scale sqrt(2); its NS output is semi-orthogonal, so
    # each update block has Frobenius norm close to sqrt(2) * sqrt(8)
    assert om.rect_scale(16, 8) == math.sqrt(2.0)


def test_heads_and_kv_split_are_independent():
    """W_UKV (20, 8) viewed (2, 10, 8) split (4, 6): changing head 1's V
    gradient rows changes only those rows of the update."""
    W = rng(4).standard_normal((20, 8))
    G = rng(5).standard_normal((20, 8))
    B = np.zeros((20, 8))
    kw = dict(view=(2, 10, 8), split=(4, 6))
    base = _step(W, G, B, **kw)[3]
    G2 = G.copy()
    G2[14:20] += rng(6).standard_normal((6, 8))
    pert = _step(W, G2, B, **kw)[3]
    changed = np.any(np.abs(pert - base) > 0, axis=1)
    assert list(np.nonzero(changed)[0]) == list(range(14, 20))


def test_missing_gradient_skips_tensor():
    W = rng(7).standard_normal((6, 4))
    B = rng(8).standard_normal((6, 4))
    W2, B2, v2, U = _step(W, None, B)
    assert U is None and np.all(W2 == W) and np.all(B2 == B)


def test_rect_scale_orientation():
    assert om.rect_scale(16, 8) == math.sqrt(2.0)
    assert om.rect_scale(4, 8) == 1.0
    assert om.rect_scale(2048, 2048) == 1.0
    assert abs(om.rect_scale(5632, 2048) - 1.6583123951777) < 1e-12
    assert om.rect_scale(2048, 5632) == 1.0


def test_update_norm_and_decay():
    """lr * (wd * W + U): with zero gradient the update is pure decoupled
    decay; otherwise W moves by lr * lr_mult * U."""
    W = rng(9).standard_normal((8, 12))
    G = np.zeros((8, 12))
    B = np.zeros((8, 12))
    W2, _, _, U = _step(W, G, B, lr=0.1, lr_mult=2.0, wd=0.5)
    assert np.all(U == 0.0)
    assert np.max(np.abs(W2 - W * (1 - 0.1 * 2.0 * 0.5))) < 1e-15
    G = rng(10).standard_normal((8, 12))
    W3, _, _, U = _step(W, G, B, lr=0.1, lr_mult=2.0)
    assert np.max(np.abs(W3 - (W - 0.2 * U))) < 1e-15


def test_normuon_row_properties():
    """Row normalisation (NorMuon section 3.1): with beta2 = 0 every row of
    the normalised update has unit RMS (up to eps); for an exactly
    orthogonalised wide full-rank matrix every row already has norm 1, the
    page's remark that row normalisation then changes nothing but a uniform
    factor."""
    O = rng(11).standard_normal((6, 20))
    N, v = om.normuon_rows(O, np.zeros(6), 0.0, 1e-8)
    assert np.max(np.abs(np.sqrt(np.mean(N * N, axis=1)) - 1.0)) < 1e-7
    assert np.max(np.abs(v - np.mean(O * O, axis=1))) < 1e-15
    D = rng(12).standard_normal((6, 20))
    X = om.orthogonalize(D, [om.CUBIC] * 40)
    assert np.max(np.abs(np.linalg.norm(X, axis=1) - 1.0)) < 1e-10
    N, _ = om.normuon_rows(X, np.zeros(6), 0.0, 0.0)
    assert np.max(np.abs(N - X * math.sqrt(20))) < 1e-9
    # EMA with beta2: two updates of the same O from zero
    v1 = om.normuon_rows(O, np.zeros(6), 0.95, 1e-8)[1]
    v2 = om.normuon_rows(O, v1, 0.95, 1e-8)[1]
    assert np.max(np.abs(v2 - (1 - 0.95 ** 2) * np.mean(O * O, axis=1))) < 1e-15


def test_rms_match_pins():
    """NorMuon section 3.1, the learning-rate scale that keeps the update's
    RMS at a target (reading: per matrix, U * rho sqrt(mn) / ||U||_F).
    Worked value: [[3, 4]] at rho = 0.5 is [[3, 4]] * 0.5 sqrt(2) / 5, whose
    RMS is 0.5; the result keeps the direction; a positive multiple of U
    gives the same result; zero stays zero."""
    U = om.rms_match(np.array([[3.0, 4.0]]), 0.5)
    assert np.max(np.abs(U - np.array([[3.0, 4.0]]) * (0.5 * math.sqrt(2.0) / 5.0))) < 1e-15
    assert abs(math.sqrt(np.mean(U * U)) - 0.5) < 1e-15
    for shape in [(7, 3), (3, 7), (16, 16)]:
        X = rng(15).standard_normal(shape)
        Y = om.rms_match(X, 0.2)
        assert abs(math.sqrt(np.mean(Y * Y)) - 0.2) < 1e-14
        cos = np.sum(X * Y) / (np.linalg.norm(X) * np.linalg.norm(Y))
        assert abs(cos - 1.0) < 1e-14
        assert np.max(np.abs(om.rms_match(3.7 * X, 0.2) - Y)) < 1e-14
    assert np.all(om.rms_match(np.zeros((4, 5)), 0.2) == 0.0)


def test_normuon_rms_step():
    """In the step, each matrix of a view gets its own RMS (per-matrix
    granularity of the build_parameter_groups views), the rectangular scale
    is not applied on top, and rms_target = 0 is the plain NorMuon step."""
    m, n = 20, 8
    W = rng(16).standard_normal((m, n))
    G = rng(17).standard_normal((m, n))
    kw = dict(v_row=np.zeros(m), normuon=True, view=(2, 10, 8), split=(4, 6))
    _, _, _, U = _step(W, G, np.zeros((m, n)), rms_target=0.3, **kw)
    for r0, rows in [(0, 4), (4, 6), (10, 4), (14, 6)]:
        blk = U[r0:r0 + rows]
        assert abs(math.sqrt(np.mean(blk * blk)) - 0.3) < 1e-13
    _, _, _, U0 = _step(W, G, np.zeros((m, n)), **kw)
    for r0, rows in [(0, 4), (4, 6), (10, 4), (14, 6)]:
        a, b = U[r0:r0 + rows], U0[r0:r0 + rows]
        assert abs(np.sum(a * b) / (np.linalg.norm(a) * np.linalg.norm(b)) - 1.0) < 1e-13


def test_state_memory_formulas():
    """NorMuon section 3.3: Muon keeps m n state numbers, NorMuon m (n + 1)."""
    m, n = 20, 8
    W = rng(13).standard_normal((m, n))
    _, B, v, _ = _step(W, rng(14).standard_normal((m, n)), np.zeros((m, n)),
                       v_row=np.zeros(m), normuon=True)
    assert B.size == m * n and B.size + v.size == m * (n + 1)


# ---------------------------------------------------------------------------
# AdamW

def _torch_adamw(p, g, m, v, t, lr, b1, b2, eps, wd):
    """Library comparison: torch.optim.AdamW, single-tensor path, fp64."""
    P = torch.nn.Parameter(torch.tensor(p, dtype=torch.float64))
    P.grad = torch.tensor(g, dtype=torch.float64)
    opt = torch.optim.AdamW([P], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd,
                            foreach=False, fused=False)
    opt.state[P] = {"step": torch.tensor(float(t - 1), dtype=torch.float64),
                    "exp_avg": torch.tensor(m, dtype=torch.float64),
                    "exp_avg_sq": torch.tensor(v, dtype=torch.float64)}
    opt.step()
    st = opt.state[P]
    return P.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


@pytest.mark.parametrize("t,state,wd,coef", [(1, "zero", 0.0, 1.0), (7, "random", 0.0, 0.37),
                                             (3, "random", 0.1, 1.0), (1000, "random", 0.0, 0.5)])
def test_adamw_matches_torch(t, state, wd, coef):
    r = rng(20 + t)
    p = r.standard_normal(1000)
    g = r.standard_normal(1000) * 1e-3
    if state == "zero":
        m = np.zeros(1000)
        v = np.zeros(1000)
    else:
        m = r.standard_normal(1000) * 1e-3
        v = np.abs(r.standard_normal(1000)) * 1e-6
    kw = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=wd, t=t)
    got = oa.adamw_update(p, g, m, v, coef=coef, **kw)
    ref = _torch_adamw(p, coef * g, m, v, t, 3e-4, 0.9, 0.95, 1e-8, wd)
    for a, b in zip(got, ref):
        assert np.max(np.abs(a - b) / (np.abs(b) + 1e-30)) < 1e-12
    dp = got[0] - p
    assert np.max(np.abs(dp - (ref[0] - p))) < 1e-15


def test_adamw_first_step_and_constant_gradient():
    """From zero state the bias-corrected moments are g' and g'^2 exactly,
    for every step while the gradient stays constant: each step moves p by
    -lr g' / (|g'| + eps)."""
    g = rng(30).standard_normal(50)
    p = rng(31).standard_normal(50)
    m = np.zeros(50)
    v = np.zeros(50)
    for t in range(1, 6):
        p2, m, v = oa.adamw_update(p, g, m, v, coef=0.5, lr=1e-3, t=t)
        step = -1e-3 * (0.5 * g) / (np.abs(0.5 * g) + 1e-8)
        assert np.max(np.abs((p2 - p) - step)) < 1e-15
        p = p2


def test_adamw_zero_gradient_is_pure_decay():
    p = rng(32).standard_normal(10)
    p2, m, v = oa.adamw_update(p, np.zeros(10), np.zeros(10), np.zeros(10), lr=0.01, wd=0.1, t=1)
    assert np.max(np.abs(p2 - p * (1 - 0.001))) < 1e-16 and np.all(m == 0) and np.all(v == 0)


def test_clip_norm_and_coefficient():
    gs = [rng(40).standard_normal((100, 7)), rng(41).standard_normal(13), np.zeros(5)]
    N = oa.global_grad_norm(gs)
    assert abs(N - math.sqrt(math.fsum(float(x) ** 2 for g in gs for x in np.ravel(g)))) < 1e-12
    tnorm = torch.nn.utils.clip_grad_norm_([torch.nn.Parameter(torch.zeros(1, dtype=torch.float64))], 1.0)
    assert float(tnorm) == 0.0
    params = [torch.nn.Parameter(torch.zeros(g.shape, dtype=torch.float64)) for g in gs]
    for P, g in zip(params, gs):
        P.grad = torch.tensor(g, dtype=torch.float64)
    total = float(torch.nn.utils.clip_grad_norm_(params, 1.0))
    assert abs(total - N) < 1e-12 * N
    c = oa.clip_coefficient(N, 1.0)
    assert abs(c * N - 1.0) < 1e-15
    assert oa.global_grad_norm([c * g for g in gs]) == pytest.approx(1.0, abs=1e-14)
    assert oa.clip_coefficient(0.0, 1.0) == 1.0
    assert oa.clip_coefficient(0.5, 1.0) == 1.0
    assert math.isnan(oa.clip_coefficient(float("inf"), 1.0))
    assert math.isnan(oa.clip_coefficient(float("nan"), 1.0))
