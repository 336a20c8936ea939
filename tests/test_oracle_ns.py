"""Pins for the oracle's Muon arithmetic (CPU only).

Each check ties the oracle to something other than itself: the spectral
closed form of odd matrix polynomials, the SVD polar factor, exact rational
arithmetic, invariances the mathematics fixes, and the pages' worked example
(diag(100, 1) has polar factor diag(1, 1)).
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import muon as om

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")))

CUBIC = (1.5, -0.5, 0.0)
# Second-order Newton-Schulz for the inverse square root: the binomial series
# of (1 - z)^(-1/2) truncated after z^2, written for x (1 - (1 - x^2))^(-1/2).
# Derived here, not taken from the pages; used to exercise the c term.
QUINTIC = (15.0 / 8.0, -5.0 / 4.0, 3.0 / 8.0)


def rng(seed):
    return np.random.default_rng(seed)


def orthonormal(m, r, seed):
    q, _ = np.linalg.qr(rng(seed).standard_normal((m, r)))
    return q


def scalar_iterate(x, coeffs):
    """The odd polynomial a x + b x^3 + c x^5 applied to each singular value."""
    for a, b, c in coeffs:
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def spectral_expected(U, sig, V, coeffs):
    D = (U * sig) @ V.T
    s = max(np.max(np.abs(D)), 1e-7)
    sig0 = sig / (np.sqrt(np.sum(sig ** 2)) + 1e-7 * s)
    return D, (U * scalar_iterate(sig0, coeffs)) @ V.T


@pytest.mark.parametrize("shape", [(6, 6), (5, 9), (9, 5), (1, 7), (7, 1), (12, 40), (40, 12)])
@pytest.mark.parametrize("coeffs", [[CUBIC] * 5, [QUINTIC] * 5,
                                    [CUBIC, QUINTIC, (2.0, -1.5, 0.5), CUBIC, (1.2, -0.3, 0.1)]])
def test_spectral_closed_form(shape, coeffs):
    m, n = shape
    r = min(m, n)
    U = orthonormal(m, r, 10 + m)
    V = orthonormal(n, r, 20 + n)
    sig = np.array([1.0, 0.3, 0.1, 0.01, 0.5, 0.05, 0.2, 0.7, 0.9, 0.03, 0.4, 0.6] * 4)[:r]
    D, expected = spectral_expected(U, sig, V, coeffs)
    got = om.orthogonalize(D, coeffs)
    assert got.shape == D.shape
    assert np.max(np.abs(got - expected)) < 1e-12


def test_polar_example_diag_100_1():
    ex = GOLDEN["polar_example"]
    D = np.array(ex["input"])
    got = om.orthogonalize(D, [CUBIC] * 30)
    assert np.max(np.abs(got - np.array(ex["polar_factor"]))) < 1e-12
    # five cubic steps do not reach it: the small direction grows by about
    # 1.5x per step from 0.01, the large one is already at 1
    five = om.orthogonalize(D, [CUBIC] * 5)
    x = scalar_iterate(np.array([1.0, 0.01]) / (math.sqrt(1.0001) + 1e-7), [CUBIC] * 5)
    assert np.max(np.abs(np.diag(five) - x)) < 1e-14
    # without the 1e-7 norm epsilon the small value would be 0.01 / sqrt(1.0001)
    # pushed through five cubic steps = 0.0758191302279601; the epsilon moves
    # it by about 1e-7 relative
    assert abs(five[1, 1] - 0.0758191302279601) < 1e-8
    assert five[0, 1] == 0.0 and five[1, 0] == 0.0


@pytest.mark.parametrize("shape", [(16, 24), (24, 16), (20, 20), (3, 50)])
def test_polar_factor_matches_svd(shape):
    D = rng(sum(shape)).standard_normal(shape)
    u, _, vt = np.linalg.svd(D, full_matrices=False)
    got = om.orthogonalize(D, [CUBIC] * 40)
    assert np.max(np.abs(got - u @ vt)) < 1e-10
    # the semi-orthogonality invariant on the small side
    p = min(shape)
    gram = got @ got.T if shape[0] <= shape[1] else got.T @ got
    assert np.max(np.abs(gram - np.eye(p))) < 1e-10


@pytest.mark.parametrize("shape", [(128, 1), (1, 128), (8, 16)])
def test_rank_one_is_not_zeroed(shape):
    """A Frobenius-normalised rank-1 matrix has singular value 1, a fixed
    point of every (a, b, c) with a + b + c = 1: Newton-Schulz returns u v^T
    and zero singular values stay zero."""
    m, n = shape
    u = rng(1).standard_normal((m, 1))
    v = rng(2).standard_normal((n, 1))
    D = u @ v.T
    for coeffs in ([CUBIC] * 5, [QUINTIC] * 5):
        got = om.orthogonalize(D, coeffs)
        assert abs(np.linalg.norm(got) - 1.0) < 1e-12
        assert np.max(np.abs(got - D / np.linalg.norm(D))) < 1e-12


def test_transpose_scale_zero_invariances():
    D = rng(3).standard_normal((13, 29))
    coeffs = [QUINTIC] * 5
    base = om.orthogonalize(D, coeffs)
    assert np.max(np.abs(om.orthogonalize(D.T, coeffs) - base.T)) < 1e-14
    for c in (1e-3, 7.0, 1e3):
        assert np.max(np.abs(om.orthogonalize(c * D, coeffs) - base)) < 1e-13
    z = om.orthogonalize(np.zeros((4, 6)), coeffs)
    assert np.all(z == 0.0)


def test_ema_momentum_form_gives_same_direction():
    """The MuonClip page's EMA momentum m = d m + (1 - d) g is (1 - d) times
    the sum form; the Frobenius step cancels the factor."""
    mu = 0.95
    B_sum = np.zeros((10, 14))
    B_ema = np.zeros((10, 14))
    for step in range(4):
        G = rng(40 + step).standard_normal((10, 14))
        B_sum = om.momentum_update(B_sum, G, mu)
        D_sum = om.nesterov_direction(G, B_sum, mu)
        B_ema = mu * B_ema + (1 - mu) * G
        D_ema = (1 - mu) * G + mu * B_ema
        assert np.max(np.abs(D_ema - (1 - mu) * D_sum)) < 1e-13
        a = om.orthogonalize(D_sum, [CUBIC] * 5)
        b = om.orthogonalize(D_ema, [CUBIC] * 5)
        assert np.max(np.abs(a - b)) < 1e-12


def test_momentum_two_step_closed_form():
    mu = 0.95
    G1 = rng(5).standard_normal((3, 4))
    G2 = rng(6).standard_normal((3, 4))
    B = om.momentum_update(om.momentum_update(np.zeros((3, 4)), G1, mu), G2, mu)
    assert np.max(np.abs(B - (mu * G1 + G2))) < 1e-15
    D = om.nesterov_direction(G2, B, mu)
    assert np.max(np.abs(D - ((1 + mu) * G2 + mu * mu * G1))) < 1e-15
    assert np.all(om.nesterov_direction(G2, B, mu, nesterov=False) == B)


# ---------------------------------------------------------------------------
# exact rational brute force

def _exact_sqrt(q):
    num, den = q.numerator, q.denominator
    rn, rd = math.isqrt(num), math.isqrt(den)
    assert rn * rn == num and rd * rd == den, "fixture needs a rational Frobenius norm"
    return Fraction(rn, rd)


def exact_orthogonalize(D, coeffs):
    """Pre-normalisation and iterations in exact rationals, with no
    transposition (X X^T X is orientation-free)."""
    X = [[Fraction(x) for x in row] for row in D]
    s = max(max(abs(x) for x in row) for row in X)
    s = max(s, Fraction(1e-7))
    X = [[x / s for x in row] for row in X]
    fro = _exact_sqrt(sum(x * x for row in X for x in row))
    X = [[x / (fro + Fraction(1e-7)) for x in row] for row in X]
    m, n = len(X), len(X[0])

    def mul(P, Q):
        return [[sum(P[i][k] * Q[k][j] for k in range(len(Q))) for j in range(len(Q[0]))]
                for i in range(len(P))]

    for a, b, c in coeffs:
        a, b, c = Fraction(a), Fraction(b), Fraction(c)
        Xt = [[X[i][j] for i in range(m)] for j in range(n)]
        A = mul(X, Xt)
        AX = mul(A, X)
        AAX = mul(A, AX)
        X = [[a * X[i][j] + b * AX[i][j] + c * AAX[i][j] for j in range(n)] for i in range(m)]
    return X


@pytest.mark.parametrize("D", [
    [[3]],
    [[1, 2], [2, 0]],
    [[2, 2, 1], [0, 0, 4]],
    [[1, 2], [2, 0], [0, 4]],
])
@pytest.mark.parametrize("coeffs", [[CUBIC] * 5, [QUINTIC] * 3])
def test_exact_rational_brute_force(D, coeffs):
    exact = exact_orthogonalize(D, coeffs)
    got = om.orthogonalize(np.array(D, dtype=np.float64), coeffs)
    want = np.array([[float(x) for x in row] for row in exact])
    assert np.max(np.abs(got - want)) < 1e-14


def test_prenormalize_edges():
    # the max-abs clamp: a tiny matrix is not blown up by the max rescale
    D = np.full((2, 2), 1e-9)
    X = om.prenormalize(D)
    Y = D / 1e-7
    assert np.allclose(X, Y / (np.linalg.norm(Y) + 1e-7), rtol=0, atol=1e-18)
    # huge entries do not overflow thanks to the max rescale
    D = np.array([[1e300, 1e300], [0.0, 1e300]])
    X = om.prenormalize(D)
    assert np.all(np.isfinite(X)) and abs(np.linalg.norm(X) - 1.0) < 1e-6


def test_ns_flop_count():
    # cubic: 4 p^2 q per iteration; quintic adds 2 p^3
    assert om.ns_flops(2048, 5632, 5, False) == 5 * 4 * 2048 * 2048 * 5632
    assert om.ns_flops(5632, 2048, 5, True) == 5 * (4 * 2048 * 2048 * 5632 + 2 * 2048 ** 3)
