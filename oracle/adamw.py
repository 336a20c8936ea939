"""fp64 AdamW path: the global gradient norm over AdamW parameters, the clip
coefficient, and the bias-corrected AdamW update with decoupled decay.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

import math

import numpy as np


def global_grad_norm(grads):
    """sqrt of the sum of squares of every AdamW gradient element.

    OMN page: gradient clipping at 1.0 applies to the AdamW parameters only,
    so the norm is taken over the AdamW gradients alone.  Reading: the
    textbook global-norm clip (all listed tensors pooled into one norm).
    """
    total = 0.0
    for g in grads:
        g = np.asarray(g, dtype=np.float64)
        total += float(np.sum(g * g))
    return math.sqrt(total)


def clip_coefficient(total_norm, max_norm=1.0):
    """Multiplier applied to every AdamW gradient: min(1, max_norm / N).

    Reading (only "clipping at 1.0" is stated): a zero norm leaves the
    gradients as they are, and a non-finite norm is propagated as NaN.
    """
    if not math.isfinite(total_norm):
        return float("nan")
    if total_norm > max_norm:
        return max_norm / total_norm
    return 1.0


def adamw_update(p, g, m, v, *, coef=1.0, lr=3e-4, beta1=0.9, beta2=0.95,
                 eps=1e-8, wd=0.0, t=1):
    """One AdamW step on one tensor, elementwise.

    OMN page: betas (0.90, 0.95), epsilon 1e-8, zero decay on every active
    group.  Qwen optimizer notes (the Adam/AdamW history and section 1):
    first and second moment estimates with bias correction; AdamW decouples
    the decay and shrinks the weight in proportion to itself.  Reading: the
    epsilon is added after the square root of the corrected second moment,
    and the step counter ``t`` starts at 1.

        g' = coef * g
        m  = beta1 m + (1 - beta1) g'
        v  = beta2 v + (1 - beta2) g'^2
        p  = p - lr wd p - lr (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)

    Returns ``(p, m, v)`` in float64.
    """
    p = np.asarray(p, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64) * coef
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    p = p - lr * wd * p - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p, m, v
