"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case swaps one oracle function for a plausibly wrong variant (a
dropped term, a wrong sign, a missing transpose, an off-by-one exponent)
and checks that an independent pin now fails.
"""

import math

import numpy as np
import pytest

from oracle import adamw as oa
from oracle import muon as om

CUBIC = (1.5, -0.5, 0.0)
QUINTIC = (15.0 / 8.0, -5.0 / 4.0, 3.0 / 8.0)


def spectral_error(orthogonalize, shape, coeffs):
    m, n = shape
    r = min(m, n)
    rg = np.random.default_rng(m * 100 + n)
    U, _ = np.linalg.qr(rg.standard_normal((m, r)))
    V, _ = np.linalg.qr(rg.standard_normal((n, r)))
    sig = np.linspace(1.0, 0.05, r)
    D = (U * sig) @ V.T
    s = np.max(np.abs(D))
    x = sig / (np.linalg.norm(sig) + 1e-7 * s)
    for a, b, c in coeffs:
        x = a * x + b * x ** 3 + c * x ** 5
    try:
        got = orthogonalize(D, coeffs)
        return float(np.max(np.abs(got - (U * x) @ V.T)))
    except ValueError:
        return float("inf")


def ns_no_c(X, coeffs):
    for a, b, c in coeffs:
        A = X @ X.T
        X = a * X + b * (A @ X)
    return X


def ns_wrong_sign(X, coeffs):
    for a, b, c in coeffs:
        A = X @ X.T
        X = a * X - b * (A @ X) + c * ((A @ A) @ X)
    return X


def ns_transposed_operand(X, coeffs):
    for a, b, c in coeffs:
        A = X.T @ X
        X = a * X + b * (A @ X) + c * ((A @ A) @ X)
    return X


def orth_no_restore(D, coeffs):
    X = om.prenormalize(D)
    if X.shape[0] > X.shape[1]:
        X = X.T
    return om.newton_schulz(X, coeffs)


def prenorm_no_fro(D, clamp=1e-7, eps=1e-7):
    return D / max(np.max(np.abs(D)), clamp)


@pytest.mark.parametrize("name,patch,coeffs,shape", [
    ("dropped c term", ("newton_schulz", ns_no_c), [QUINTIC] * 5, (6, 10)),
    ("wrong sign of b", ("newton_schulz", ns_wrong_sign), [CUBIC] * 5, (6, 10)),
    ("transposed Gram operand", ("newton_schulz", ns_transposed_operand), [QUINTIC] * 5, (8, 8)),
    ("orientation not restored", ("orthogonalize", orth_no_restore), [CUBIC] * 5, (10, 6)),
    ("no Frobenius step", ("prenormalize", prenorm_no_fro), [CUBIC] * 5, (6, 10)),
])
def test_planted_ns_mistake_is_caught(monkeypatch, name, patch, coeffs, shape):
    assert spectral_error(om.orthogonalize, shape, coeffs) < 1e-12
    monkeypatch.setattr(om, patch[0], patch[1])
    assert spectral_error(om.orthogonalize, shape, coeffs) > 1e-6, name


def test_planted_rms_mistake_is_caught(monkeypatch):
    """An RMS factor over the rows only (sqrt(m) instead of sqrt(mn)) fails
    the RMS pin of the NorMuon step."""
    import tests.test_oracle_views_adamw as t

    def bad(U, rho):
        U = np.asarray(U, dtype=np.float64)
        f = float(np.sqrt(np.sum(U * U)))
        return U * (rho * np.sqrt(U.shape[0]) / f) if f > 0 else U.copy()

    monkeypatch.setattr(om, "rms_match", bad)
    with pytest.raises(AssertionError):
        t.test_normuon_rms_step()


def test_planted_scale_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(om, "rect_scale", lambda m, n: float(np.sqrt(max(1.0, n / m))))
    W = np.random.default_rng(0).standard_normal((32, 8))
    G = np.random.default_rng(1).standard_normal((32, 8))
    U = om.muon_step_tensor(W, G, np.zeros((32, 8)), view=(2, 16, 8))[3]
    # each (16, 8) block's NS output has Frobenius norm ~ sqrt(8) after five
    # steps only if scaled by sqrt(2) -> block norm ~ 4; the wrong scale gives ~ 2.8
    blk = np.linalg.norm(U[:16]) / np.linalg.norm(om.orthogonalize(
        om.nesterov_direction(G[:16], G[:16], 0.95), [CUBIC] * 5))
    assert abs(blk - math.sqrt(2.0)) > 0.1


def _adamw_off_by_one(p, g, m, v, *, coef=1.0, lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.0, t=1):
    g = g * coef
    m = beta1 * m + (1 - beta1) * g
    v = beta2 * v + (1 - beta2) * g * g
    return p - lr * wd * p - lr * (m / (1 - beta1 ** (t + 1))) / (np.sqrt(v / (1 - beta2 ** (t + 1))) + eps), m, v


def _adamw_eps_inside(p, g, m, v, *, coef=1.0, lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.0, t=1):
    g = g * coef
    m = beta1 * m + (1 - beta1) * g
    v = beta2 * v + (1 - beta2) * g * g
    return p - lr * wd * p - lr * (m / (1 - beta1 ** t)) / np.sqrt(v / (1 - beta2 ** t) + eps), m, v


@pytest.mark.parametrize("bad", [_adamw_off_by_one, _adamw_eps_inside])
def test_planted_adamw_mistake_is_caught(bad):
    from tests.test_oracle_views_adamw import _torch_adamw
    r = np.random.default_rng(5)
    p, g = r.standard_normal(100), r.standard_normal(100) * 1e-3
    m, v = r.standard_normal(100) * 1e-3, np.abs(r.standard_normal(100)) * 1e-6
    ref = _torch_adamw(p, g, m, v, 4, 3e-4, 0.9, 0.95, 1e-8, 0.0)
    good = oa.adamw_update(p, g, m, v, t=4)
    assert np.max(np.abs(good[0] - ref[0])) < 1e-15
    wrong = bad(p, g, m, v, t=4)
    assert np.max(np.abs(wrong[0] - ref[0])) > 1e-7
