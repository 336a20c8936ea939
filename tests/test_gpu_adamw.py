"""GPU parity of the clip norm and AdamW against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

import oracle
from adamw_optimizer_step_gb300 import _binding as B
from adamw_optimizer_step_gb300 import workloads as wk
from tests.parity import f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from adamw_optimizer_step_gb300 import build
    build.build()
    B.lib()


def run(params, *, lr, t, max_norm=1.0, wd=0.0, clip=True):
    dev = [tuple(x.cuda().contiguous() for x in p) for p in params]
    total = torch.zeros(1, device="cuda")
    coef = torch.zeros(1, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.gbo_clip_norm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    if clip:
        B.gbo_clip_norm([d[1] for d in dev], max_norm, total, coef, ws, dev_status=status)
    B.gbo_adamw_step(dev, lr=lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=wd, step=t,
                     coef=coef if clip else None, dev_status=status)
    torch.cuda.synchronize()
    return dev, float(total.item()), float(coef.item()), int(status.item())


def check(params, dev, *, lr, t, coef, wd=0.0, b1=0.9, b2=0.95, eps=1e-8):
    """m, v, p within 1e-6 of the oracle relative to the size of the terms
    that form them (m can cancel to ~0: b1 m_old + (1 - b1) g'), plus one
    fp32 rounding of p itself."""
    for (p, g, m, v), (pd, _, md, vd) in zip(params, dev):
        P, G, M, V = f64(p), f64(g), f64(m), f64(v)
        po, mo, vo = oracle.adamw_update(P, G, M, V, coef=coef, lr=lr, beta1=b1, beta2=b2, eps=eps, wd=wd, t=t)
        m_scale = b1 * np.abs(M) + (1 - b1) * np.abs(coef * G)
        assert np.all(np.abs(f64(md) - mo) <= 1e-6 * m_scale + 1e-37), "m mismatch"
        assert np.all(np.abs(f64(vd) - vo) <= 1e-6 * np.abs(vo) + 1e-37), "v mismatch"
        step_scale = lr * wd * np.abs(P) + lr * (m_scale / (1 - b1 ** t)) / (np.sqrt(vo / (1 - b2 ** t)) + eps)
        slack = 1e-6 * step_scale + 2.0 ** -24 * np.abs(po) * 1.01 + 1e-37
        assert np.all(np.abs(f64(pd) - po) <= slack), "p mismatch"


def test_adamw_with_decay_rounds_p_once():
    """With weight decay the new p is the oracle's within one fp32 rounding
    of p (decay and Adam step summed before they meet p)."""
    params = tiny_params("random")
    dev, _, coef, _ = run(params, lr=3e-4, t=5, wd=0.1)
    check(params, [tuple(x.cpu() for x in d) for d in dev], lr=3e-4, t=5, coef=coef, wd=0.1)


def tiny_params(state):
    wl = wk.workload(1)
    return [wk.adamw_tensor_inputs(wl, i, state=state) for i in range(len(wl.adamw))]


@pytest.mark.parametrize("state,t", [("zero", 1), ("random", 7)])
def test_tiny_adamw_with_clip(state, t):
    params = tiny_params(state)
    dev, total, coef, status = run(params, lr=3e-4, t=t)
    N = oracle.global_grad_norm([f64(g) for _, g, _, _ in params])
    c = oracle.clip_coefficient(N, 1.0)
    assert status == 0
    assert abs(total - N) <= 1e-6 * N
    assert abs(coef - c) <= 2e-6 * c
    check(params, dev, lr=3e-4, t=t, coef=c)


def test_ragged_many_tensors_and_dtypes():
    """More tensors than one launch takes, odd sizes, bf16 gradients, and
    tensors that start off a 16-byte boundary (scalar path)."""
    gen = torch.Generator().manual_seed(5)
    params = []
    for k in range(150):
        n = int(torch.randint(1, 5000, (1,), generator=gen))
        p = torch.randn(n, generator=gen)
        g = torch.randn(n, generator=gen) * 1e-2
        if k % 3 == 0:
            g = g.to(torch.bfloat16)
        m = torch.randn(n, generator=gen) * 1e-3
        v = torch.rand(n, generator=gen) * 1e-6
        params.append((p, g, m, v))
    # a parameter that starts 4 bytes into its buffer (scalar path)
    p_host = torch.randn(4096, generator=gen)
    params.append((p_host, torch.randn(4096, generator=gen) * 1e-2, torch.zeros(4096), torch.zeros(4096)))
    dev = [tuple(x.cuda() for x in p) for p in params]
    big = torch.empty(4097, device="cuda")
    big[1:].copy_(dev[-1][0])
    dev[-1] = (big[1:],) + dev[-1][1:]
    total = torch.zeros(1, device="cuda")
    coef = torch.zeros(1, device="cuda")
    ws = torch.empty(B.gbo_clip_norm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    B.gbo_clip_norm([d[1] for d in dev], 1.0, total, coef, ws)
    B.gbo_adamw_step(dev, lr=1e-3, step=3, coef=coef)
    torch.cuda.synchronize()
    N = oracle.global_grad_norm([f64(g) for _, g, _, _ in params])
    assert abs(float(total.item()) - N) <= 1e-6 * N
    check(params, dev, lr=1e-3, t=3, coef=oracle.clip_coefficient(N, 1.0))


def test_clip_edges():
    ws = torch.empty(B.gbo_clip_norm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    total = torch.zeros(1, device="cuda")
    coef = torch.zeros(1, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # zero gradients: N = 0, coef = 1
    B.gbo_clip_norm([torch.zeros(1000, device="cuda")], 1.0, total, coef, ws, dev_status=status)
    torch.cuda.synchronize()
    assert total.item() == 0.0 and coef.item() == 1.0 and status.item() == 0
    # small gradients: no clipping
    g = torch.full((100,), 1e-3, device="cuda")
    B.gbo_clip_norm([g], 1.0, total, coef, ws, dev_status=status)
    torch.cuda.synchronize()
    assert abs(total.item() - 1e-2) < 1e-8 and coef.item() == 1.0
    # no tensors at all
    B.gbo_clip_norm([], 1.0, total, coef, ws, dev_status=status)
    torch.cuda.synchronize()
    assert total.item() == 0.0 and coef.item() == 1.0
    # NaN: flagged, coef NaN
    g = torch.ones(100, device="cuda")
    g[7] = float("inf")
    B.gbo_clip_norm([g], 1.0, total, coef, ws, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() & B.GBO_STATUS_NONFINITE and math.isnan(coef.item())


def test_omn_adamw_full_size():
    """The 128000 x 2048 tied embedding and 49 gains with 1% hot rows: the
    clip norm over all 262M gradients, then AdamW checked on a seeded sample
    of elements of every tensor (the update is elementwise)."""
    wl = wk.workload(3)
    params = [wk.adamw_tensor_inputs(wl, i, device="cuda", state="random") for i in range(len(wl.adamw))]
    host = [tuple(x.cpu() for x in p) for p in params]
    total = torch.zeros(1, device="cuda")
    coef = torch.zeros(1, device="cuda")
    ws = torch.empty(B.gbo_clip_norm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    B.gbo_clip_norm([p[1] for p in params], 1.0, total, coef, ws)
    B.gbo_adamw_step(params, lr=3e-4, step=5, coef=coef)
    torch.cuda.synchronize()
    N = oracle.global_grad_norm([f64(g) for _, g, _, _ in host])
    c = oracle.clip_coefficient(N, 1.0)
    assert abs(total.item() - N) <= 1e-6 * N and c < 0.1
    rng = np.random.default_rng(3)
    for (p, g, m, v), (pd, _, md, vd) in zip(host, params):
        n = p.numel()
        idx = torch.from_numpy(rng.choice(n, size=min(n, 200000), replace=False))
        sub = [x.reshape(-1)[idx] for x in (p, g, m, v)]
        got = [x.reshape(-1)[idx.cuda()].cpu() for x in (pd, md, vd)]
        check([tuple(sub)], [(got[0], None, got[1], got[2])], lr=3e-4, t=5, coef=c)


def test_device_step_in_cuda_graph():
    """With the step count on the device, clip + AdamW captured once in a
    CUDA graph (with the count's increment) replays steps t = 2, 3, 4 as
    direct launches with the host count give them."""
    params = tiny_params("random")
    devs = [[tuple(x.cuda().clone() for x in p) for p in params] for _ in range(2)]
    ws = [torch.empty(B.gbo_clip_norm_workspace_bytes(), dtype=torch.uint8, device="cuda") for _ in range(2)]
    tot = [torch.zeros(1, device="cuda") for _ in range(2)]
    coef = [torch.zeros(1, device="cuda") for _ in range(2)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step(k, **kw):
        B.gbo_clip_norm([d[1] for d in devs[k]], 1.0, tot[k], coef[k], ws[k], dev_status=status)
        B.gbo_adamw_step(devs[k], lr=3e-4, coef=coef[k], dev_status=status, **kw)

    for t in (1, 2, 3, 4):  # direct, host step count
        step(0, step=t)
    t_dev = torch.ones(1, dtype=torch.int32, device="cuda")
    step(1, dev_step=t_dev)  # t = 1, direct
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        t_dev.add_(1)
        step(1, dev_step=t_dev)
    for _ in range(3):  # t = 2, 3, 4
        graph.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(t_dev.item()) == 4
    for a, b in zip(devs[0], devs[1]):
        for x, y in zip(a, b):
            assert torch.equal(x, y)

