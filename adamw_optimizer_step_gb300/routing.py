"""Role routing: which parameters of a torch module take the Muon path (and
with which matrix view), which take AdamW, and with what decay.

Rules ("build_parameter_groups", kimi-k3 docs, sections "Recording
independent matrix geometry", "Exclusion and decay rules" and
"Classification happens once per original parameter identity"; "Dual-
Manifold Optimization in OMN", routing paragraph: the role decides, not the
rank):

* module traversal records matrix views on projection weights by module
  structure -- a ``gate_up_proj`` Linear with ``intermediate_size`` is
  viewed (2, I, C); a ``QKV`` Linear with ``num_heads``, ``d_head`` and
  ``d_model`` is viewed (3, H, D, C); MLA ``W_UQ`` / ``W_UKV`` Linears are
  viewed per head, (H, D + D_s, R_q) and (H, D + D_v, R_kv) with split sizes
  (D, D_v) -- each view only describes how rows split into independent
  matrices, the parameter itself is untouched;
* embedding weights and output classifiers (``lm_head``, ``head``) are
  auxiliary: they never take the Muon path; norm gains and the learned
  residual query projections take no decay;
* every trainable parameter is classified exactly once, by identity (a tied
  embedding / head is visited once): fewer than two dimensions or no-decay
  -> AdamW without decay; a 2-D non-auxiliary matrix -> Muon with decay;
  anything else (auxiliary 2-D, 3-D filters) -> AdamW with decay;
* frozen parameters are skipped, and a model with nothing to train is
  refused with ``ValueError``.

This module only builds tables; the arithmetic runs in the library's
kernels (see :class:`HybridOptimizer`).
"""

from dataclasses import dataclass
from typing import Optional, Tuple

import torch
import torch.nn as nn

NO_DECAY_LINEARS = ("attn_res_proj", "mlp_res_proj", "output_attn_res_proj")
HEAD_NAMES = ("lm_head", "head")


@dataclass
class ParamRoute:
    name: str
    param: nn.Parameter
    algorithm: str                     # "muon" | "adamw"
    decay: bool
    view: Optional[Tuple[int, ...]] = None
    split: Optional[Tuple[int, ...]] = None


def _norm_types():
    kinds = [nn.LayerNorm]
    if hasattr(nn, "RMSNorm"):
        kinds.append(nn.RMSNorm)
    return tuple(kinds)


def _record_view(views, weight, shape, split=None):
    """Register a view for one weight, refusing bad or conflicting views.

    Every entry must be a positive int and the flattened leading axes must
    give back the stored 2-D shape; the split sizes must cut the row axis.
    """
    shape = tuple(shape)
    if any((not isinstance(s, int)) or s <= 0 for s in shape):
        raise ValueError("view entries must be positive integers: %r" % (shape,))
    lead = 1
    for s in shape[:-1]:
        lead *= s
    if weight.dim() != 2 or (lead, shape[-1]) != tuple(weight.shape):
        raise ValueError("view %r does not flatten to the stored shape %r" % (shape, tuple(weight.shape)))
    if split is not None:
        split = tuple(split)
        if any((not isinstance(s, int)) or s <= 0 for s in split) or sum(split) != shape[-2]:
            raise ValueError("split sizes %r must be positive and sum to %d" % (split, shape[-2]))
    key = id(weight)
    if key in views and views[key] != (shape, split):
        raise ValueError("conflicting views for one weight: %r and %r" % (views[key], (shape, split)))
    views[key] = (shape, split)


def _linear(module, name):
    m = getattr(module, name, None)
    return m if isinstance(m, nn.Linear) else None


def build_parameter_groups(model, weight_decay=0.0, auxiliary_decay=True):
    """Route every trainable parameter of ``model``.

    Returns a list of :class:`ParamRoute` in ``named_parameters()`` order;
    ``weight_decay`` is the decay of the decayed routes (0 for all others).
    ``auxiliary_decay=False`` puts embeddings and output heads in the
    no-decay AdamW group too: the OMN recipe, whose decayed AdamW group is
    empty.
    """
    views, auxiliary, no_decay = {}, set(), set()
    norms = _norm_types()
    for mname, module in model.named_modules():
        if isinstance(module, nn.Embedding):
            auxiliary.add(id(module.weight))
        if isinstance(module, norms):
            for p in module.parameters(recurse=False):
                no_decay.add(id(p))
        for attr in NO_DECAY_LINEARS:
            lin = _linear(module, attr)
            if lin is not None:
                for p in lin.parameters(recurse=False):
                    no_decay.add(id(p))
        for attr in HEAD_NAMES:
            lin = _linear(module, attr)
            if lin is not None:
                auxiliary.add(id(lin.weight))
        gate_up = _linear(module, "gate_up_proj")
        if gate_up is not None and hasattr(module, "intermediate_size"):
            _record_view(views, gate_up.weight, (2, int(module.intermediate_size), gate_up.in_features))
        qkv = _linear(module, "QKV")
        if qkv is not None and all(hasattr(module, a) for a in ("num_heads", "d_head", "d_model")):
            _record_view(views, qkv.weight, (3, int(module.num_heads), int(module.d_head), int(module.d_model)))
        uq, ukv = _linear(module, "W_UQ"), _linear(module, "W_UKV")
        if uq is not None and ukv is not None:
            H, D = int(module.num_heads), int(module.d_head)
            _record_view(views, uq.weight, (H, D + int(module.d_shared), int(module.q_latent_dim)))
            _record_view(views, ukv.weight, (H, D + int(module.dv_head), int(module.kv_latent_dim)),
                         (D, int(module.dv_head)))
    routes, seen = [], set()
    for name, p in model.named_parameters():
        if not p.requires_grad or id(p) in seen:
            continue
        seen.add(id(p))
        key = id(p)
        if p.dim() < 2 or key in no_decay:
            routes.append(ParamRoute(name, p, "adamw", False))
        elif p.dim() == 2 and key not in auxiliary:
            view, split = views.get(key, (None, None))
            routes.append(ParamRoute(name, p, "muon", True, view, split))
        else:
            routes.append(ParamRoute(name, p, "adamw", auxiliary_decay or key not in auxiliary))
    if not routes:
        raise ValueError("the model has no trainable parameters")
    for r in routes:
        r.weight_decay = float(weight_decay) if r.decay else 0.0
    return routes


# ---------------------------------------------------------------------------

class HybridOptimizer:
    """Muon on the routed matrices + clipped AdamW on the rest, stepped by
    the library's kernels on the current CUDA stream.

    State (all caller-side torch tensors): an fp32 momentum buffer per Muon
    weight (and a NorMuon row vector), fp32 AdamW moments, the step count.
    Muon weights may be bf16 or fp32; AdamW parameters must be fp32.  The
    Muon plan binds the gradient tensors; it is rebuilt when the set of
    gradient tensors changes (e.g. after ``zero_grad(set_to_none=True)``).

    ``precision`` "bf16" or "f32" (three TF32 products); ``route`` "auto",
    "x" or "gram" (see gbo_muon_opts); ``rms_target`` > 0 with NorMuon
    scales each matrix's update to that RMS.

    ``graph=True``: the first step (and the first after the parameter or
    gradient tensors change) runs directly, then one step is captured in a
    CUDA graph, with the AdamW step count kept on the device, and later
    steps replay it.  The learning rates are fixed at capture.
    """

    def __init__(self, model, *, muon_lr=0.01, adamw_lr=3e-4, weight_decay=0.0, auxiliary_decay=True, mu=0.95,
                 ns_steps=5, abc=(1.5, -0.5, 0.0), normuon=False, beta2_rows=0.95, eps_rows=1e-8,
                 rms_target=0.0, betas=(0.9, 0.95), eps=1e-8, max_norm=1.0, precision="bf16", route="auto",
                 graph=False):
        from . import _binding as B
        self.B = B
        self.routes = build_parameter_groups(model, weight_decay, auxiliary_decay)
        self.muon = [r for r in self.routes if r.algorithm == "muon"]
        self.adamw = [r for r in self.routes if r.algorithm == "adamw"]
        for r in self.adamw:
            if r.param.dtype != torch.float32:
                raise TypeError("AdamW parameter %s must be float32" % r.name)
        self.muon_lr, self.adamw_lr = muon_lr, adamw_lr
        self.betas, self.eps, self.max_norm = betas, eps, max_norm
        self.opts = dict(abc=abc, ns_steps=ns_steps, mu=mu, normuon=normuon, beta2=beta2_rows, eps=eps_rows,
                         rms_target=rms_target,
                         route={"auto": B.GBO_ROUTE_AUTO, "x": B.GBO_ROUTE_X, "gram": B.GBO_ROUTE_GRAM}[route],
                         precision=B.GBO_NS_F32 if precision == "f32" else B.GBO_NS_BF16)
        self.state = {}
        for r in self.muon:
            p = r.param
            self.state[r.name] = {"mom": torch.zeros(p.shape, dtype=torch.float32, device=p.device)}
            if normuon:
                self.state[r.name]["row_v"] = torch.zeros(p.shape[0], dtype=torch.float32, device=p.device)
        for r in self.adamw:
            p = r.param
            self.state[r.name] = {"m": torch.zeros_like(p, dtype=torch.float32),
                                  "v": torch.zeros_like(p, dtype=torch.float32)}
        self.step_count = 0
        self._plan = None
        self._plan_key = None
        self._ws = None
        dev = (self.muon or self.adamw)[0].param.device
        self.total_norm = torch.zeros(1, device=dev)
        self.coef = torch.zeros(1, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self._cws = torch.empty(B.gbo_clip_norm_workspace_bytes(), dtype=torch.uint8, device=dev)
        self.graph = graph
        self._graph = None      # torch.cuda.CUDAGraph of one step, or None
        self._graph_key = None  # the tensors it was captured with
        self._step_t = torch.zeros(1, dtype=torch.int32, device=dev)  # AdamW t on the device

    def _muon_entries(self):
        out = []
        for r in self.muon:
            st = self.state[r.name]
            out.append(dict(w=r.param.data, g=r.param.grad, mom=st["mom"], row_v=st.get("row_v"),
                            view=r.view, split=r.split, wd=r.weight_decay))
        return out

    def _ensure_plan(self):
        key = tuple((r.param.data_ptr(), None if r.param.grad is None else r.param.grad.data_ptr())
                    for r in self.muon)
        if self._plan is not None and key == self._plan_key:
            return
        self._plan = self.B.gbo_muon_plan_create(self._muon_entries(), **self.opts)
        self._plan_key = key
        need = self.B.gbo_muon_workspace_bytes(self._plan)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 1), dtype=torch.uint8, device=self.total_norm.device)

    def layout_hash(self):
        """Hash of the Muon layout (shapes, views, splits, dtypes), for checkpoints."""
        self._ensure_plan()
        return self.B.gbo_desc_hash(self._plan)

    def _launch(self, dev_step=None):
        """Enqueue one step on the current stream: the host step count, or
        with ``dev_step`` the device one."""
        if self.muon:
            self.B.gbo_muon_step(self._plan, self.muon_lr, self._ws, dev_status=self.status)
        active = [r for r in self.adamw if r.param.grad is not None]
        if active:
            self.B.gbo_clip_norm([r.param.grad for r in active], self.max_norm, self.total_norm, self.coef,
                                 self._cws, dev_status=self.status)
            for wd in sorted({r.weight_decay for r in active}):  # one call per decay value
                params = [(r.param.data, r.param.grad, self.state[r.name]["m"], self.state[r.name]["v"])
                          for r in active if r.weight_decay == wd]
                self.B.gbo_adamw_step(params, lr=self.adamw_lr, beta1=self.betas[0], beta2=self.betas[1],
                                      eps=self.eps, weight_decay=wd, step=self.step_count, coef=self.coef,
                                      dev_status=self.status, dev_step=dev_step)

    def _tensor_key(self):
        return tuple((r.param.data_ptr(), None if r.param.grad is None else r.param.grad.data_ptr())
                     for r in self.routes)

    @torch.no_grad()
    def step(self):
        """One hybrid step; returns the pre-clip AdamW gradient norm (a device
        tensor) and leaves the device status word in ``self.status``."""
        self.step_count += 1
        if self.muon:
            self._ensure_plan()
        if not self.graph:
            self._launch()
            return self.total_norm
        key = self._tensor_key()
        if self._graph is not None and key == self._graph_key:
            self._graph.replay()  # advances the device count, then the step
            return self.total_norm
        # direct step (sets the plan up on the device), then capture the next
        self._step_t.fill_(self.step_count)
        self._launch(dev_step=self._step_t)
        torch.cuda.synchronize()
        self._graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self._graph):
            self._step_t.add_(1)
            self._launch(dev_step=self._step_t)
        self._graph_key = key
        return self.total_norm

    def state_dict(self):
        return {"step": self.step_count, "layout_hash": self.layout_hash() if self.muon else 0,
                "state": {k: {n: t.clone() for n, t in v.items()} for k, v in self.state.items()}}

    def load_state_dict(self, sd):
        if self.muon and sd["layout_hash"] != self.layout_hash():
            raise ValueError("checkpoint was written for a different Muon layout (views, splits or shapes)")
        self.step_count = int(sd["step"])
        self._graph = None  # a captured step holds the old count
        for k, v in sd["state"].items():
            for n, t in v.items():
                self.state[k][n].copy_(t)
