"""The HybridOptimizer front end on a toy model: one step through the
library matches the oracle route by route, and its state round-trips."""

import copy

import numpy as np
import pytest
import torch

import oracle
from oracle.views import sub_matrices
from tests.parity import TOL, f64, ulp
from tests.test_routing import LAYOUTS, Toy, ToyFused

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from adamw_optimizer_step_gb300 import build, _binding as B
    build.build()
    B.lib()


def make_model(seed, cls=Toy):
    torch.manual_seed(seed)
    m = cls().cuda()
    for p in m.parameters():
        if p.requires_grad:
            p.grad = torch.randn_like(p) * 1e-2
    return m


def check_step_against_oracle(model, **kw):
    """One HybridOptimizer step, route by route (row blocks of a fused
    weight included) against the oracle: Muon routes on their rows with
    their view, AdamW routes with the clip over every AdamW gradient."""
    from adamw_optimizer_step_gb300.routing import HybridOptimizer
    before = {n: (p.detach().clone(), p.grad.clone()) for n, p in model.named_parameters() if p.requires_grad}
    opt = HybridOptimizer(model, muon_lr=0.02, adamw_lr=1e-3, weight_decay=0.1, precision="bf16", **kw)
    norm = opt.step()
    torch.cuda.synchronize()
    assert int(opt.status.item()) == 0
    adam_grads = [f64(r.part(before[r.name][1])) for r in opt.adamw]
    N = oracle.global_grad_norm(adam_grads)
    assert abs(float(norm.item()) - N) <= 1e-6 * N
    c = oracle.clip_coefficient(N, 1.0)
    for r in opt.routes:
        W0, G = (f64(r.part(t)) for t in before[r.name])
        got = f64(r.part(r.param.detach()))
        if r.algorithm == "muon":
            Wn, _, _, U = oracle.muon_step_tensor(W0, G, np.zeros_like(G), view=r.view, split=r.split,
                                                  lr=0.02, wd=r.weight_decay)
            for r0, m, n in sub_matrices(W0.shape[0], W0.shape[1], r.view, r.split):
                sl = slice(r0, r0 + m)
                bound = (np.linalg.norm(ulp(Wn[sl], torch.float32)) + 0.02 * TOL["bf16"] * np.linalg.norm(U[sl])
                         + 1e-6 * np.linalg.norm(W0[sl]))
                assert np.linalg.norm(got[sl] - Wn[sl]) <= bound, r.key
        else:
            pn, _, _ = oracle.adamw_update(W0, G, np.zeros_like(G), np.zeros_like(G), coef=c, lr=1e-3,
                                           wd=r.weight_decay, t=1)
            assert np.max(np.abs(got - pn) - (1e-6 * 1e-3 + 2 ** -23 * np.abs(pn))) <= 0, r.key
    return opt


def test_hybrid_step_matches_oracle():
    check_step_against_oracle(make_model(1))


def test_hybrid_step_with_excluded_blocks_matches_oracle():
    """A fused projection whose gate and per-head vector rows are excluded
    from Muon: its Muon blocks match the oracle on their own rows and views,
    its excluded blocks take AdamW (and count in the clip norm)."""
    opt = check_step_against_oracle(make_model(4, ToyFused), layouts=LAYOUTS)
    kinds = [(r.algorithm, r.rows) for r in opt.routes if r.name == "gdn.in_proj.weight"]
    assert kinds == [("muon", (0, 16)), ("muon", (16, 28)), ("adamw", (28, 40)), ("adamw", (40, 44))]


def test_hybrid_state_round_trip():
    """Step, save, restore into a fresh optimizer on a copy of the model,
    step both: bitwise equal parameters."""
    from adamw_optimizer_step_gb300.routing import HybridOptimizer
    a = make_model(2)
    opt_a = HybridOptimizer(a, muon_lr=0.02, adamw_lr=1e-3)
    opt_a.step()
    sd = opt_a.state_dict()
    b = copy.deepcopy(a)
    for pa, pb in zip(a.parameters(), b.parameters()):
        if pa.requires_grad:
            pb.grad = pa.grad.clone()
    opt_b = HybridOptimizer(b, muon_lr=0.02, adamw_lr=1e-3)
    opt_b.load_state_dict(sd)
    opt_a.step()
    opt_b.step()
    torch.cuda.synchronize()
    for (na, pa), (nb, pb) in zip(a.named_parameters(), b.named_parameters()):
        assert torch.equal(pa, pb), na
    # a different Muon layout is refused
    c = Toy().cuda()
    c.ffn.intermediate_size = 8  # gate_up viewed (2, 8, 8) would not flatten -> use another layout
    c.ffn.gate_up_proj = torch.nn.Linear(8, 16, bias=False).cuda()
    for p in c.parameters():
        if p.requires_grad:
            p.grad = torch.zeros_like(p)
    opt_c = HybridOptimizer(c)
    with pytest.raises(ValueError):
        opt_c.load_state_dict(sd)


def test_graph_mode_matches_direct_steps():
    """graph=True (a direct first step, then replays of one captured step with
    the AdamW count on the device) gives bitwise the parameters and states
    of direct steps, in both precisions."""
    from adamw_optimizer_step_gb300.routing import HybridOptimizer
    for precision in ("bf16", "f32"):
        a = make_model(3)
        b = copy.deepcopy(a)
        for pa, pb in zip(a.parameters(), b.parameters()):
            if pa.grad is not None:
                pb.grad = pa.grad.clone()
        kw = dict(muon_lr=0.02, adamw_lr=1e-3, weight_decay=0.1, precision=precision)
        oa = HybridOptimizer(a, **kw)
        ob = HybridOptimizer(b, graph=True, **kw)
        for _ in range(4):
            oa.step()
            ob.step()
        torch.cuda.synchronize()
        assert ob._graph is not None and int(ob._step_t.item()) == 4
        assert int(oa.status.item()) == 0 and int(ob.status.item()) == 0
        for (na, pa), (nb, pb) in zip(a.named_parameters(), b.named_parameters()):
            assert torch.equal(pa, pb), na
        for k in oa.state:
            for n in oa.state[k]:
                assert torch.equal(oa.state[k][n], ob.state[k][n]), (k, n)
