"""fp64 Muon path: momentum, Nesterov direction, pre-normalisation,
Newton-Schulz iterations, orientation, rectangular scale, NorMuon rows and
the weight write.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy float64;
the only library primitive used is the matrix product.
"""

import numpy as np

from .views import sub_matrices

CUBIC = (1.5, -0.5, 0.0)


def expand_coeffs(abc, steps=None):
    """Turn the coefficient argument into one (a, b, c) triple per iteration.

    ``abc`` is either one triple, used for every iteration (the pages' fixed
    recurrence), or a sequence of triples, one per iteration (the per-step
    schedule the Qwen optimizer notes mention in section 2).
    """
    abc = [tuple(float(x) for x in t) for t in np.atleast_2d(np.asarray(abc, dtype=np.float64))]
    if steps is None:
        return abc
    if len(abc) == 1:
        return abc * int(steps)
    if len(abc) != steps:
        raise ValueError("one coefficient triple per iteration, or one shared triple")
    return abc


def momentum_update(B, G, mu):
    """Momentum buffer: B_t = mu * B_{t-1} + G_t.

    NorMuon paper (zskr.cn), section 2.2, eq. (1), with the buffer starting
    at zero; the OMN page's Muon path keeps one zeros-initialised buffer per
    parameter at coefficient 0.95.
    """
    return mu * B + G


def nesterov_direction(G, B, mu, nesterov=True):
    """Direction handed to the orthogonalisation.

    OMN page, Muon path: the Nesterov-style direction adds the scaled buffer
    back to the current gradient, D_t = G_t + mu * B_t.  With ``nesterov``
    off the direction is the buffer itself, as in eq. (2) of the NorMuon
    paper, O_t = NS5(M_t).  (Reading: the equation is missing from the OMN
    page; this is the sum form of eq. (1) plus the sentence describing it.)
    """
    if nesterov:
        return G + mu * B
    return np.array(B, dtype=np.float64, copy=True)


def prenormalize(D, clamp=1e-7, eps=1e-7):
    """Rescale by the largest absolute entry, then by the Frobenius norm.

    OMN page, Muon path: the direction is cast up, divided by its largest
    absolute element (clamped from below at 1e-7), then normalised by its
    Frobenius norm "with epsilon handling".  Reading: the epsilon is added to
    the norm, X0 = Y / (||Y||_F + 1e-7) with Y = D / max(max|D|, 1e-7).  The
    NorMuon paper, section 2.2, starts Newton-Schulz from X0 = M / ||M||_F,
    which this equals up to the epsilon.
    """
    D = np.asarray(D, dtype=np.float64)
    s = max(float(np.max(np.abs(D))) if D.size else 0.0, clamp)
    Y = D / s
    return Y / (np.sqrt(np.sum(Y * Y)) + eps)


def newton_schulz(X, coeffs):
    """Newton-Schulz polynomial iterations.

    NorMuon paper, section 2.2, eq. (5):
        X_k = a X_{k-1} + b (X_{k-1} X_{k-1}^T) X_{k-1} + c (X_{k-1} X_{k-1}^T)^2 X_{k-1}.
    The MuonClip page's cubic X <- 1.5 X - 0.5 X (X^T X) is the case
    (a, b, c) = (1.5, -0.5, 0), because X (X^T X) = (X X^T) X.
    ``coeffs`` holds one (a, b, c) per iteration.
    """
    X = np.asarray(X, dtype=np.float64)
    for a, b, c in coeffs:
        A = X @ X.T
        X = a * X + b * (A @ X) + c * ((A @ A) @ X)
    return X


def orthogonalize(D, coeffs):
    """Normalise, orient, iterate and restore one matrix.

    OMN page, Muon path order: normalisation, then the orientation
    adjustment (transpose when there are more rows than columns, so the Gram
    product is on the smaller side), the polynomial iterations, then the
    original orientation is restored.
    """
    X = prenormalize(D)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    X = newton_schulz(X, coeffs)
    if tall:
        X = X.T
    return X


def rect_scale(m, n):
    """Rectangular scale sqrt(max(1, m / n)).

    OMN page, Muon path (the rectangular shape scaling term), with m and n
    the matrix's rows and columns in the stored out-by-in orientation
    (reading: the formula itself is missing from the page text; the
    surrounding sentences fix the orientation).
    """
    return float(np.sqrt(max(1.0, m / n)))


def normuon_rows(O, v, beta2, eps):
    """NorMuon row-wise second moment and row normalisation.

    NorMuon paper, section 3.1: each row (neuron) keeps an exponential moving
    average, decay beta2, of the mean over columns of the squared update;
    the update rows are then divided by it.  Readings (the algorithm listing
    is not printed): no bias correction, epsilon outside the square root,
    statistics on the unscaled Newton-Schulz output.

    Returns the normalised rows and the new second-moment vector.
    """
    O = np.asarray(O, dtype=np.float64)
    ms = np.mean(O * O, axis=1)
    v_new = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * ms
    return O / (np.sqrt(v_new)[:, None] + eps), v_new


def rms_match(U, rms_target):
    """Scale a row-normalised update so that its root-mean-square is rms_target.

    NorMuon paper, section 3.1: the row normalisation leaves a direction of
    larger norm, so the update gets a learning-rate scale that keeps its RMS
    near Adam's.  Reading (the listing line is not printed): per matrix,
    U = rms_target * sqrt(m n) / ||U||_F * U, with the target supplied by
    the caller; an all-zero update stays zero.
    """
    U = np.asarray(U, dtype=np.float64)
    f = float(np.sqrt(np.sum(U * U)))
    if f == 0.0:
        return U.copy()
    return U * (rms_target * np.sqrt(U.size) / f)


def weight_update(W, U, lr, wd):
    """W_t = W_{t-1} - lr * wd * W_{t-1} - lr * U_t.

    NorMuon paper, section 2.2, eq. (3), plus decoupled weight decay as the
    Qwen optimizer notes describe for AdamW (decay applied to the weight,
    not through the gradient).  The OMN recipe uses no Muon decay (wd = 0).
    """
    W = np.asarray(W, dtype=np.float64)
    return W - lr * wd * W - lr * U


def muon_step_tensor(W, G, B, *, view=None, split=None, mu=0.95, nesterov=True,
                     coeffs=None, ns_steps=5, lr=0.02, lr_mult=1.0, wd=0.0,
                     v_row=None, normuon=False, beta2=0.95, eps=1e-8, rms_target=0.0):
    """One Muon step for one stored weight with its matrix view.

    Order (OMN page, Muon path): gradient -> momentum -> Nesterov direction
    -> per matrix: normalisation, orientation, iterations, restore -> the
    rectangular scale -> (optional NorMuon rows) -> weight update.  The view
    is expanded into independent matrices (build_parameter_groups docs); the
    norm, the orientation and the scale are per matrix (Qwen optimizer notes,
    section 4: the fused tensor would mix directions and give the scale a
    fake shape).  A missing gradient skips the weight untouched
    (build_parameter_groups: inactive experts).

    The per-tensor learning-rate multiplier scales both the decay and the
    update: W <- W - (lr * lr_mult) * (wd * W + U).

    With NorMuon and ``rms_target > 0`` each matrix's normalised update is
    rescaled to that RMS (:func:`rms_match`) in place of the rectangular
    scale, which the rescaling would cancel.

    Returns ``(W_new, B_new, v_new, U)`` in float64, where ``U`` is the update
    direction (scale times the normalised NS output), or ``None`` for ``U``
    when the gradient is missing.
    """
    W = np.asarray(W, dtype=np.float64)
    if G is None:
        return W.copy(), np.array(B, dtype=np.float64, copy=True), (
            None if v_row is None else np.array(v_row, dtype=np.float64, copy=True)), None
    G = np.asarray(G, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    rows, cols = W.shape
    if coeffs is None:
        coeffs = CUBIC
    coeffs = expand_coeffs(coeffs, ns_steps)
    B_new = momentum_update(B, G, mu)
    D = nesterov_direction(G, B_new, mu, nesterov)
    U = np.zeros_like(W)
    v_new = None if v_row is None else np.array(v_row, dtype=np.float64, copy=True)
    for r0, m, n in sub_matrices(rows, cols, view, split):
        O = orthogonalize(D[r0:r0 + m], coeffs)
        if normuon:
            O, v_new[r0:r0 + m] = normuon_rows(O, v_new[r0:r0 + m], beta2, eps)
        if normuon and rms_target > 0:
            U[r0:r0 + m] = rms_match(O, rms_target)
        else:
            U[r0:r0 + m] = rect_scale(m, n) * O
    W_new = weight_update(W, U, lr * lr_mult, wd)
    return W_new, B_new, v_new, U


def ns_flops(m, n, steps, quintic):
    """Dense-count Newton-Schulz FLOPs for one m x n matrix.

    Per iteration on the p x q oriented matrix (p = min, q = max): the Gram
    product (2 p^2 q), the product back onto X (2 p^2 q) and, when c != 0,
    the square of the Gram matrix (2 p^3).
    """
    p, q = min(m, n), max(m, n)
    return steps * (4 * p * p * q + (2 * p ** 3 if quintic else 0))
