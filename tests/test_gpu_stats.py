"""Per-matrix norms (gbo_muon_plan_set_stats): ||D||_F of the momentum
direction and ||U||_F of the update direction, for every matrix of the
active weights in table order, from the reductions the step already runs.
Checked against the step's own exported update (gbo_muon_step's dbg_update)
and against the fp64 oracle's D and U, in both precisions, with NorMuon
(single pass, streamed, RMS-keeping scale), fp32 and bf16 weights, a skipped
weight, and a plan split into groups by a workspace cap."""

import numpy as np
import pytest
import torch

import oracle
from oracle.views import sub_matrices
from tests.parity import TOL, f64, random_entries
from adamw_optimizer_step_gb300 import _binding as B

pytestmark = pytest.mark.gpu

SHAPES = [(600, 130, None, None), (130, 600, None, None), (256, 256, None, None),
          (4 * 96, 1000, (4, 96, 1000), None), (200, 40, (2, 100, 40), (30, 70)), (128, 512, None, None)]


def run(entries, precision, normuon, rms_target, cap_frac=0.0):
    dev = []
    for e in entries:
        d = dict(e)
        for k in ("w", "g", "mom", "row_v"):
            if d.get(k) is not None:
                d[k] = d[k].cuda().contiguous()
        dev.append(d)
    kw = dict(precision=B.GBO_NS_F32 if precision == "f32" else B.GBO_NS_BF16, normuon=normuon, beta2=0.95,
              eps=1e-8, rms_target=rms_target)
    plan = B.gbo_muon_plan_create(dev, **kw)
    if cap_frac:
        plan = B.gbo_muon_plan_create(dev, workspace_cap=int(B.gbo_muon_workspace_bytes(plan) * cap_frac), **kw)
    n = B.gbo_muon_plan_info(plan)["n_matrices"]
    stats = torch.full((2 * n,), float("nan"), device="cuda")
    B.gbo_muon_plan_set_stats(plan, stats)
    ws = torch.empty(max(1, B.gbo_muon_workspace_bytes(plan)), dtype=torch.uint8, device="cuda")
    U = torch.zeros(sum(e["w"].numel() for e in entries), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.gbo_muon_step(plan, 0.02, ws, dbg_update=U, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return stats.cpu().double().numpy().reshape(-1, 2), U.cpu().double().numpy()


@pytest.mark.parametrize("precision,normuon,rms_target,cap,fp32w", [
    ("bf16", False, 0.0, 0.0, True), ("bf16", True, 0.0, 0.0, True), ("bf16", True, 0.0, 0.0, False),
    ("bf16", True, 0.2, 0.0, False), ("f32", False, 0.0, 0.0, True), ("f32", True, 0.0, 0.0, True),
    ("bf16", False, 0.0, 0.7, True)])
def test_matrix_norms(precision, normuon, rms_target, cap, fp32w):
    """fp32w: one weight in fp32 (its write takes the register path, and
    NorMuon takes its single pass); else all bf16 (NorMuon's streamed write
    after a statistics pass)."""
    entries = random_entries(SHAPES, seed=51, normuon=normuon, b_std=1e-3)
    if fp32w:
        entries[2]["w"] = entries[2]["w"].float()
    entries[1]["g"] = None  # skipped: no matrices in the table of norms
    stats, U = run(entries, precision, normuon, rms_target, cap)
    j, off = 0, 0
    for e in entries:
        rows, cols = e["w"].shape
        if e["g"] is None:
            off += rows * cols
            continue
        G, B0 = f64(e["g"]), f64(e["mom"])
        D = oracle.nesterov_direction(G, oracle.momentum_update(B0, G, 0.95), 0.95)
        _, _, _, Uo = oracle.muon_step_tensor(f64(e["w"]), G, B0, view=e["view"], split=e["split"], lr=0.02,
                                              v_row=None if e["row_v"] is None else f64(e["row_v"]), normuon=normuon,
                                              beta2=0.95, eps=1e-8, rms_target=rms_target)
        Ug = U[off:off + rows * cols].reshape(rows, cols)
        for r0, m, n in sub_matrices(rows, cols, e["view"], e["split"]):
            nd, nu = stats[j]
            assert abs(nd - np.linalg.norm(D[r0:r0 + m])) <= 1e-5 * np.linalg.norm(D[r0:r0 + m]), (j, "D")
            # the step's own update, exported: the same values, summed another way
            assert abs(nu - np.linalg.norm(Ug[r0:r0 + m])) <= 2e-5 * np.linalg.norm(Ug[r0:r0 + m]), (j, "U")
            assert abs(nu - np.linalg.norm(Uo[r0:r0 + m])) <= TOL[precision] * np.linalg.norm(Uo[r0:r0 + m])
            j += 1
        off += rows * cols
    assert j == len(stats)
