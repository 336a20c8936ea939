"""gbo_clip_norm_noalloc, the clip norm for callers that cannot allocate
device memory (all of it owned by another allocator, or no cudaMalloc
allowed on their path): it must give what gbo_clip_norm gives with a
caller-provided workspace, on consecutive calls that reuse the library's
one fixed scratch array.

This file is collected last on purpose, so a run that stops at the first
failure has run every other test before it."""

import pytest
import torch

import oracle
from adamw_optimizer_step_gb300 import _binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from adamw_optimizer_step_gb300 import build
    build.build()
    B.lib()


def grad_set(seed, n_tensors, scale):
    gen = torch.Generator().manual_seed(seed)
    out = []
    for k in range(n_tensors):
        n = int(torch.randint(1, 40000, (1,), generator=gen))
        g = torch.randn(n, generator=gen) * scale
        if k % 4 == 1:
            g = g.to(torch.bfloat16)
        out.append(g.cuda())
    return out


def with_workspace(grads, max_norm):
    total = torch.zeros(1, device="cuda")
    coef = torch.zeros(1, device="cuda")
    ws = torch.empty(B.gbo_clip_norm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    B.gbo_clip_norm(grads, max_norm, total, coef, ws)
    torch.cuda.synchronize()
    return total.item(), coef.item()


def test_noalloc_matches_workspace_version_on_consecutive_calls():
    # two different gradient sets back to back: the second call reuses the
    # scratch array the first one filled (more tensors than one launch
    # takes, so several slices of the array are in use)
    sets = [grad_set(1, 150, 1e-4), grad_set(2, 70, 3.0)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    results = []
    for grads in sets:
        total = torch.full((1,), -1.0, device="cuda")
        coef = torch.full((1,), -1.0, device="cuda")
        B.gbo_clip_norm_noalloc(grads, 1.0, total, coef, dev_status=status)
        torch.cuda.synchronize()
        results.append((total.item(), coef.item()))
    assert status.item() == 0
    for grads, (total, coef) in zip(sets, results):
        ref_total, ref_coef = with_workspace(grads, 1.0)
        assert abs(total - ref_total) <= 1e-6 * ref_total
        assert abs(coef - ref_coef) <= 1e-6 * ref_coef
        # and the fp64 oracle's global norm and clip coefficient, on the same
        # values (bf16 gradients widened exactly)
        host = [g.double().cpu().numpy() for g in grads]
        o_total = oracle.global_grad_norm(host)
        o_coef = oracle.clip_coefficient(o_total, 1.0)
        assert abs(total - o_total) <= 1e-6 * o_total
        assert abs(coef - o_coef) <= 1e-6 * o_coef
    # the second set is large: clipping is active; the first is not
    assert results[0][1] == 1.0 and results[1][1] < 1.0


def test_noalloc_refuses_too_many_tensors():
    g = torch.zeros(1, device="cuda")
    total = torch.zeros(1, device="cuda")
    coef = torch.zeros(1, device="cuda")
    with pytest.raises(B.GboError) as e:
        B.gbo_clip_norm_noalloc([g] * 65537, 1.0, total, coef)
    assert e.value.code == -1 and "65536" in str(e.value)
