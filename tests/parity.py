"""Helpers for the GPU-vs-oracle parity tests: run the CUDA path through the
binding and the fp64 oracle on the same inputs, and compare.

Acceptance (per matrix of a view):
* update direction U = scale * O, relative Frobenius error <= 1e-4 with fp32
  Newton-Schulz arithmetic, <= 3e-2 with bf16 operands;
* momentum B: |B - B_oracle| <= 1e-6 (|mu B_old| + |G|) elementwise;
* weight, per matrix: ||W - W_oracle||_F within one rounding of W's dtype per
  element plus lr * lr_mult * tol * ||U_oracle||_F; and, as a consistency
  check, W equals W_old - lr lr_mult (wd W_old + U) of the exported U rounded
  once to W's dtype.
"""

import math

import numpy as np
import torch

import oracle
from oracle.views import sub_matrices
from adamw_optimizer_step_gb300 import _binding as B

TOL = {"f32": 1e-4, "bf16": 3e-2}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_fro(a, b):
    nb = float(np.linalg.norm(b))
    return float(np.linalg.norm(a - b)) / (nb if nb > 0 else 1.0)


def ulp(x, dtype):
    """One unit in the last place of |x| in ``dtype`` (float32 or bfloat16)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    mant = 23 if dtype == torch.float32 else 7
    e = np.floor(np.log2(np.maximum(x, 1e-38)))
    return np.exp2(e - mant)


def run_muon_gpu(entries, *, lr, precision, steps=1, dbg=True, free_sms=0, **opts):
    """Copy ``entries`` (CPU tensors) to the GPU, run ``steps`` Muon steps,
    return CPU results: list of dicts W, B, v, U plus the status word.
    ``free_sms``: SMs the plan's Newton-Schulz kernels leave free."""
    dev = []
    for e in entries:
        d = dict(e)
        for k in ("w", "g", "mom", "row_v"):
            if d.get(k) is not None:
                d[k] = d[k].cuda().contiguous()
        dev.append(d)
    plan = B.gbo_muon_plan_create(dev, precision=B.GBO_NS_F32 if precision == "f32" else B.GBO_NS_BF16,
                                  **opts)
    if free_sms:
        B.gbo_muon_plan_set_free_sms(plan, free_sms)
    ws = torch.empty(max(1, B.gbo_muon_workspace_bytes(plan)), dtype=torch.uint8, device="cuda")
    total = sum(e["w"].numel() for e in entries)
    U = torch.full((total,), float("nan"), dtype=torch.float32, device="cuda") if dbg else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(steps):
        B.gbo_muon_step(plan, lr, ws, dbg_update=U, dev_status=status)
    torch.cuda.synchronize()
    out = []
    off = 0
    for e, d in zip(entries, dev):
        n = e["w"].numel()
        out.append(dict(W=d["w"].cpu(), B=d["mom"].cpu(), v=None if d.get("row_v") is None else d["row_v"].cpu(),
                        U=None if U is None else U[off:off + n].view(e["w"].shape).cpu()))
        off += n
    return out, int(status.item()), plan


def run_muon_oracle(entries, *, lr, steps=1, abc=(1.5, -0.5, 0.0), ns_steps=5, mu=0.95, nesterov=True,
                    normuon=False, beta2=0.95, eps=1e-8, rms_target=0.0):
    coeffs = [tuple(abc[3 * i:3 * i + 3]) for i in range(len(abc) // 3)] if len(abc) > 3 else [tuple(abc)]
    res = []
    for e in entries:
        W, G, Bm = f64(e["w"]), None if e.get("g") is None else f64(e["g"]), f64(e["mom"])
        v = None if e.get("row_v") is None else f64(e["row_v"])
        U = None
        for _ in range(steps):
            W, Bm, v, U = oracle.muon_step_tensor(
                W, G, Bm, view=e.get("view"), split=e.get("split"), mu=mu, nesterov=nesterov,
                coeffs=coeffs, ns_steps=ns_steps, lr=lr, lr_mult=e.get("lr_mult", 1.0), wd=e.get("wd", 0.0),
                v_row=v, normuon=normuon, beta2=beta2, eps=eps, rms_target=rms_target)
        res.append(dict(W=W, B=Bm, v=v, U=U))
    return res


def check_muon(entries, gpu, ora, *, lr, precision, mu=0.95, check_w=True):
    """Assert the acceptance criteria; return the worst per-matrix error."""
    tol = TOL[precision]
    worst = 0.0
    for e, g, o in zip(entries, gpu, ora):
        rows, cols = e["w"].shape
        if e.get("g") is None:
            assert torch.equal(g["W"], e["w"]) and torch.equal(g["B"], e["mom"])
            continue
        Ug = f64(g["U"])
        for r0, m, n in sub_matrices(rows, cols, e.get("view"), e.get("split")):
            err = rel_fro(Ug[r0:r0 + m], o["U"][r0:r0 + m])
            worst = max(worst, err)
            assert err <= tol, "matrix rows %d..%d of %s: rel Frobenius error %.3e > %.0e" % (
                r0, r0 + m, tuple(e["w"].shape), err, tol)
        Bscale = mu * np.abs(f64(e["mom"])) + np.abs(f64(e["g"]))
        assert np.all(np.abs(f64(g["B"]) - o["B"]) <= 1e-6 * Bscale + 1e-30), "momentum mismatch"
        if check_w:
            W0 = f64(e["w"])
            Wg = f64(g["W"])
            lrm = lr * e.get("lr_mult", 1.0)
            for r0, m, n in sub_matrices(rows, cols, e.get("view"), e.get("split")):
                sl = slice(r0, r0 + m)
                # against the oracle: one rounding to W's dtype per element plus
                # the direction tolerance carried through lr
                bound = (np.linalg.norm(ulp(o["W"][sl], e["w"].dtype)) + lrm * tol * np.linalg.norm(o["U"][sl])
                         + 2.0 ** -22 * np.linalg.norm(np.abs(W0[sl]) + lrm * np.abs(o["U"][sl])))
                assert np.linalg.norm(Wg[sl] - o["W"][sl]) <= bound, "weight mismatch"
            # consistency: the write applies the exported update, elementwise
            want = W0 - lrm * (e.get("wd", 0.0) * W0 + Ug)
            want_r = f64(torch.tensor(want).to(e["w"].dtype))
            diff = np.abs(Wg - want_r)
            slack = 2.0 ** -22 * (np.abs(W0) + lrm * (e.get("wd", 0.0) * np.abs(W0) + np.abs(Ug)))
            assert np.all(diff <= ulp(want, e["w"].dtype) * 1.01 + slack + 1e-30), \
                "weight write inconsistent with the exported update %.3e" % diff.max()
        if o["v"] is not None:
            # v carries the squared rows of O: three times the direction tolerance
            assert np.all(np.abs(f64(g["v"]) - o["v"]) <= 3 * tol * np.abs(o["v"]) + 1e-30), "row moment mismatch"
    return worst


def random_entries(shapes, *, seed, w_dtype=torch.bfloat16, g_dtype=torch.bfloat16, b_std=0.0, normuon=False,
                   g_std=1e-3, w_std=0.02):
    """CPU inputs for a list of (rows, cols, view, split[, lr_mult, wd]) tuples."""
    gen = torch.Generator().manual_seed(seed)
    out = []
    for k, sh in enumerate(shapes):
        rows, cols, view, split = sh[:4]
        lr_mult = sh[4] if len(sh) > 4 else 1.0
        wd = sh[5] if len(sh) > 5 else 0.0
        W = (torch.randn(rows, cols, generator=gen) * w_std).to(w_dtype)
        G = (torch.randn(rows, cols, generator=gen) * g_std).to(g_dtype)
        Bm = torch.randn(rows, cols, generator=gen) * b_std if b_std else torch.zeros(rows, cols)
        rv = torch.rand(rows, generator=gen) * 1e-3 if normuon else None
        out.append(dict(w=W, g=G, mom=Bm, row_v=rv, view=view, split=split, lr_mult=lr_mult, wd=wd))
    return out
