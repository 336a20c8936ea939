"""Role routing: which parameters of a torch module take the Muon path (and
with which matrix view), which take AdamW, and with what decay.

The rules come from "build_parameter_groups" (kimi-k3 docs: "Recording
independent matrix geometry", "Exclusion and decay rules"), from the OMN
page's routing paragraph (the role of a parameter decides, not its rank),
and from the Qwen3.8-Flash-Next optimizer notes, section 4 (a fused tensor
is split by meaning, each real sub-matrix is orthogonalised on its own, and
gate or vector sub-blocks that do not suit Muon go to AdamW).  In this
module's terms:

Geometry.  A stored 2-D projection is a stack of row blocks.  A
:class:`Layout` names a projection attribute of a module, the module fields
it reads, and how the projection's rows divide into :class:`Block` runs.  A
Muon block carries the view that cuts it into independent matrices (and
optional split sizes along the view's row axis); an AdamW block is a run of
rows excluded from Muon.  :data:`STANDARD_LAYOUTS` declares the pages' four
layouts: a gate/up pair, a per-head Q/K/V stack, and the per-head MLA
up-projections, whose K and V parts are further cut by split sizes.  A
caller adds layouts of its own (fused projections with excluded blocks)
through ``layouts=``.  Declaring a geometry never changes the parameter:
the optimizer only reads it.

Roles.  Embedding tables and output classifiers are auxiliary and never
take Muon.  Norm gains and the learned residual query projections are
never decayed.  Every trainable parameter is routed once, by identity (a
tied embedding and head count once), in ``named_parameters()`` order:

* a vector, or a parameter the rules exempt from decay, goes to AdamW
  without decay;
* an auxiliary parameter goes to AdamW with decay (none when
  ``auxiliary_decay`` is False, as in the OMN recipe);
* any other 2-D matrix goes to Muon with decay, block by block when a
  layout declares its rows; an excluded block goes to AdamW with the
  matrix's decay;
* anything else (a 3-D convolution filter, say) goes to AdamW with decay,
  since its storage is not a hidden matrix.

Frozen parameters are skipped, and a model with nothing to train is refused
with ``ValueError``; so is a layout whose blocks do not tile the stored
rows, and two different layouts for one weight.

This module only builds tables; the arithmetic runs in the library's
kernels (see :class:`HybridOptimizer`).
"""

from dataclasses import dataclass
from types import SimpleNamespace
from typing import Callable, Optional, Tuple

import torch
import torch.nn as nn


# ---------------------------------------------------------------------------
# geometry: layouts of stored projections


@dataclass(frozen=True)
class Block:
    """A run of ``rows`` consecutive stored rows of a projection.

    ``path`` is "muon" (the rows are cut into independent matrices by
    ``view``, whose last entry is the column count, and ``split``) or
    "adamw" (the rows are excluded from Muon).  A Muon block without a view
    is one matrix.
    """

    rows: int
    path: str = "muon"
    view: Optional[Tuple[int, ...]] = None
    split: Optional[Tuple[int, ...]] = None


@dataclass(frozen=True)
class Layout:
    """Where a layout applies and what it declares.

    It applies to ``module.<attr>`` when that attribute is an ``nn.Linear``,
    every name in ``siblings`` is an ``nn.Linear`` of the same module too,
    and the module has every field in ``fields``.  ``blocks(f, lin)``
    receives those fields (``f.<name>``, as ints) and the Linear, and
    returns the projection's row blocks from first row to last.
    """

    attr: str
    fields: Tuple[str, ...]
    blocks: Callable[[SimpleNamespace, nn.Linear], Tuple[Block, ...]]
    siblings: Tuple[str, ...] = ()


def _gate_up(f, lin):
    # gate and up halves of one fused FFN input projection: two I x C matrices
    return (Block(2 * f.intermediate_size, view=(2, f.intermediate_size, lin.in_features)),)


def _per_head_qkv(f, lin):
    # Q, K and V of every head: 3 * H independent D x C matrices
    return (Block(3 * f.num_heads * f.d_head, view=(3, f.num_heads, f.d_head, f.d_model)),)


def _mla_query(f, lin):
    # one (D + D_s) x R_q up-projection per head
    return (Block(f.num_heads * (f.d_head + f.d_shared),
                  view=(f.num_heads, f.d_head + f.d_shared, f.q_latent_dim)),)


def _mla_key_value(f, lin):
    # per head a K part (D rows) and a V part (D_v rows) of the latent up-projection
    return (Block(f.num_heads * (f.d_head + f.dv_head),
                  view=(f.num_heads, f.d_head + f.dv_head, f.kv_latent_dim), split=(f.d_head, f.dv_head)),)


STANDARD_LAYOUTS = (
    Layout("gate_up_proj", ("intermediate_size",), _gate_up),
    Layout("QKV", ("num_heads", "d_head", "d_model"), _per_head_qkv),
    Layout("W_UQ", ("num_heads", "d_head", "d_shared", "q_latent_dim"), _mla_query, siblings=("W_UKV",)),
    Layout("W_UKV", ("num_heads", "d_head", "dv_head", "kv_latent_dim"), _mla_key_value, siblings=("W_UQ",)),
)

# Linear projections whose parameters are never decayed (learned residual
# query vectors), and output classifiers (auxiliary, like embeddings).
NO_DECAY_LINEARS = ("attn_res_proj", "mlp_res_proj", "output_attn_res_proj")
HEAD_NAMES = ("lm_head", "head")


def _positive_ints(values):
    return all(isinstance(v, int) and not isinstance(v, bool) and v > 0 for v in values)


def _checked_blocks(weight, blocks):
    """The blocks as a tuple, after checking that they tile the stored rows
    and that each Muon block's view flattens to its rows and the columns."""
    blocks = tuple(blocks)
    if weight.dim() != 2:
        raise ValueError("a layout needs a 2-D weight, got shape %r" % (tuple(weight.shape),))
    rows, cols = weight.shape
    if not blocks or not _positive_ints([b.rows for b in blocks]) or sum(b.rows for b in blocks) != rows:
        raise ValueError("row blocks %r do not tile the %d stored rows" % ([b.rows for b in blocks], rows))
    for b in blocks:
        if b.path not in ("muon", "adamw"):
            raise ValueError("block path must be 'muon' or 'adamw', got %r" % (b.path,))
        if b.path == "adamw" and (b.view is not None or b.split is not None):
            raise ValueError("an excluded block carries no view or split")
        if b.view is None:
            if b.split is not None:
                raise ValueError("split sizes need a view")
            continue
        view = tuple(b.view)
        if len(view) < 2 or not _positive_ints(view):
            raise ValueError("view entries must be positive integers: %r" % (view,))
        lead = 1
        for v in view[:-1]:
            lead *= v
        if (lead, view[-1]) != (b.rows, cols):
            raise ValueError("view %r does not flatten to the block's %d x %d" % (view, b.rows, cols))
        if b.split is not None and (not _positive_ints(b.split) or sum(b.split) != view[-2]):
            raise ValueError("split sizes %r must be positive and sum to %d" % (tuple(b.split), view[-2]))
    return blocks


def declared_geometry(model, layouts=STANDARD_LAYOUTS):
    """Map ``id(weight) -> tuple of Blocks`` for every projection of
    ``model`` a layout applies to.  One weight reached by two different
    layouts (or by one layout with different fields) is refused."""
    geometry = {}
    for _, module in model.named_modules():
        for lay in layouts:
            lin = getattr(module, lay.attr, None)
            if not isinstance(lin, nn.Linear):
                continue
            if not all(isinstance(getattr(module, s, None), nn.Linear) for s in lay.siblings):
                continue
            if not all(hasattr(module, name) for name in lay.fields):
                continue
            fields = SimpleNamespace(**{name: int(getattr(module, name)) for name in lay.fields})
            blocks = _checked_blocks(lin.weight, lay.blocks(fields, lin))
            known = geometry.setdefault(id(lin.weight), blocks)
            if known != blocks:
                raise ValueError("conflicting layouts for one weight: %r and %r" % (known, blocks))
    return geometry


# ---------------------------------------------------------------------------
# roles and routes


def _norm_types():
    kinds = [nn.LayerNorm]
    if hasattr(nn, "RMSNorm"):
        kinds.append(nn.RMSNorm)
    return tuple(kinds)


def _role_sets(model):
    """(auxiliary, never_decayed): identities of embedding / classifier
    weights and of norm gains and residual query projections."""
    auxiliary, never_decayed = set(), set()
    norms = _norm_types()
    for module in model.modules():
        if isinstance(module, nn.Embedding):
            auxiliary.add(id(module.weight))
        if isinstance(module, norms):
            never_decayed.update(id(p) for p in module.parameters(recurse=False))
        for attr in NO_DECAY_LINEARS + HEAD_NAMES:
            lin = getattr(module, attr, None)
            if not isinstance(lin, nn.Linear):
                continue
            if attr in HEAD_NAMES:
                auxiliary.add(id(lin.weight))
            else:
                never_decayed.update(id(p) for p in lin.parameters(recurse=False))
    return auxiliary, never_decayed


def classify(param, auxiliary, never_decayed):
    """The role of one trainable parameter: "gain" (AdamW, never decayed),
    "auxiliary" (AdamW), "matrix" (Muon) or "other" (AdamW, decayed)."""
    key = id(param)
    if param.dim() < 2 or key in never_decayed:
        return "gain"
    if key in auxiliary:
        return "auxiliary"
    if param.dim() == 2:
        return "matrix"
    return "other"


@dataclass
class ParamRoute:
    """One routed parameter, or one row block of it (``rows`` = (first,
    last + 1); None for the whole tensor)."""

    name: str
    param: nn.Parameter
    algorithm: str                     # "muon" | "adamw"
    decay: bool
    view: Optional[Tuple[int, ...]] = None
    split: Optional[Tuple[int, ...]] = None
    rows: Optional[Tuple[int, int]] = None
    weight_decay: float = 0.0

    @property
    def key(self):
        """Unique name of the route (the state dictionary's key)."""
        return self.name if self.rows is None else "%s[%d:%d]" % (self.name, self.rows[0], self.rows[1])

    def part(self, t):
        """The route's rows of ``t`` (the parameter, its data or gradient, or
        a state tensor of the parameter's shape): a contiguous view."""
        return t if self.rows is None or t is None else t[self.rows[0]:self.rows[1]]

    @property
    def shape(self):
        return tuple(self.part(self.param).shape)

    def numel(self):
        return self.part(self.param).numel()


def build_parameter_groups(model, weight_decay=0.0, auxiliary_decay=True, layouts=STANDARD_LAYOUTS):
    """Route every trainable parameter of ``model``.

    Returns a list of :class:`ParamRoute` in ``named_parameters()`` order
    (the row blocks of one parameter in row order).  ``weight_decay`` is the
    decay of the decayed routes (0 for all others).  ``auxiliary_decay=False``
    puts embeddings and output heads in the no-decay AdamW group too: the OMN
    recipe, whose decayed AdamW group is empty.  ``layouts`` declares the
    row geometry of fused projections (:data:`STANDARD_LAYOUTS` by default;
    add layouts with excluded blocks for gate or vector rows).
    """
    geometry = declared_geometry(model, layouts)
    auxiliary, never_decayed = _role_sets(model)
    routes, seen = [], set()
    for name, p in model.named_parameters():
        if not p.requires_grad or id(p) in seen:
            continue
        seen.add(id(p))
        role = classify(p, auxiliary, never_decayed)
        if role == "gain":
            routes.append(ParamRoute(name, p, "adamw", False))
        elif role == "auxiliary":
            routes.append(ParamRoute(name, p, "adamw", bool(auxiliary_decay)))
        elif role == "other":
            routes.append(ParamRoute(name, p, "adamw", True))
        else:
            blocks = geometry.get(id(p))
            if blocks is None or (len(blocks) == 1 and blocks[0].path == "muon"):
                b = blocks[0] if blocks else Block(p.shape[0])
                routes.append(ParamRoute(name, p, "muon", True, b.view, b.split))
                continue
            r0 = 0
            for b in blocks:
                rows = (r0, r0 + b.rows)
                if b.path == "muon":
                    routes.append(ParamRoute(name, p, "muon", True, b.view, b.split, rows))
                else:
                    routes.append(ParamRoute(name, p, "adamw", True, rows=rows))
                r0 += b.rows
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
    Muon weights may be bf16 or fp32; AdamW parameters (and the excluded
    row blocks of a fused projection) must be fp32.  A fused projection with
    excluded blocks steps its Muon blocks as weights of their own (views of
    its rows) and its excluded blocks with the AdamW path.  The Muon plan
    binds the gradient tensors; it is rebuilt when the set of gradient
    tensors changes (e.g. after ``zero_grad(set_to_none=True)``).

    ``precision`` "bf16" or "f32" (three TF32 products); ``route`` "auto",
    "x" or "gram" (see gbo_muon_opts); ``rms_target`` > 0 with NorMuon
    scales each matrix's update to that RMS.

    ``graph=True``: the first step (and the first after the parameter or
    gradient tensors change) runs directly, then one step is captured in a
    CUDA graph, with the AdamW step count kept on the device, and later
    steps replay it.  The learning rates are fixed at capture.

    ``process_group`` (data parallelism over more than one rank, gradients
    already all-reduced): each Muon weight gets one owner rank, by LPT over
    its executed Newton-Schulz FLOPs (:class:`.sharding.MuonShards`); a rank
    steps only the Muon weights it owns, and an all-gather after the Muon
    step hands every rank the owners' updated weights.  The AdamW path runs
    on every rank, on identical inputs.  Not combined with ``graph``.
    """

    def __init__(self, model, *, muon_lr=0.01, adamw_lr=3e-4, weight_decay=0.0, auxiliary_decay=True, mu=0.95,
                 ns_steps=5, abc=(1.5, -0.5, 0.0), normuon=False, beta2_rows=0.95, eps_rows=1e-8,
                 rms_target=0.0, betas=(0.9, 0.95), eps=1e-8, max_norm=1.0, precision="bf16", route="auto",
                 graph=False, layouts=STANDARD_LAYOUTS, process_group=None):
        from . import _binding as B
        self.B = B
        self.group = process_group
        self.shards = None
        if process_group is not None and graph:
            raise ValueError("graph mode is not combined with a process group")
        self.routes = build_parameter_groups(model, weight_decay, auxiliary_decay, layouts)
        self.muon = [r for r in self.routes if r.algorithm == "muon"]
        self.adamw = [r for r in self.routes if r.algorithm == "adamw"]
        for r in self.adamw:
            if r.param.dtype != torch.float32:
                raise TypeError("AdamW parameter %s must be float32" % r.key)
        self.muon_lr, self.adamw_lr = muon_lr, adamw_lr
        self.betas, self.eps, self.max_norm = betas, eps, max_norm
        self.opts = dict(abc=abc, ns_steps=ns_steps, mu=mu, normuon=normuon, beta2=beta2_rows, eps=eps_rows,
                         rms_target=rms_target,
                         route={"auto": B.GBO_ROUTE_AUTO, "x": B.GBO_ROUTE_X, "gram": B.GBO_ROUTE_GRAM}[route],
                         precision=B.GBO_NS_F32 if precision == "f32" else B.GBO_NS_BF16)
        self.state = {}
        for r in self.muon:
            dev = r.param.device
            self.state[r.key] = {"mom": torch.zeros(r.shape, dtype=torch.float32, device=dev)}
            if normuon:
                self.state[r.key]["row_v"] = torch.zeros(r.shape[0], dtype=torch.float32, device=dev)
        for r in self.adamw:
            self.state[r.key] = {"m": torch.zeros(r.shape, dtype=torch.float32, device=r.param.device),
                                 "v": torch.zeros(r.shape, dtype=torch.float32, device=r.param.device)}
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

    def _muon_entries(self, local=True):
        """Plan entries of the Muon routes; ``local``: with the gradients of
        weights another rank owns dropped."""
        out = []
        for r in self.muon:
            st = self.state[r.key]
            out.append(dict(w=r.part(r.param.data), g=r.part(r.param.grad), mom=st["mom"], row_v=st.get("row_v"),
                            view=r.view, split=r.split, wd=r.weight_decay))
        if local and self.group is not None:
            import torch.distributed as dist
            world, rank = dist.get_world_size(self.group), dist.get_rank(self.group)
            if world > 1:
                from .sharding import MuonShards
                if self.shards is None:
                    self.shards = MuonShards(self._muon_entries(local=False), world, rank, **self.opts)
                out = self.shards.local_entries(out)
        return out

    def _ensure_plan(self):
        key = tuple((r.part(r.param.data).data_ptr(),
                     None if r.param.grad is None else r.part(r.param.grad).data_ptr()) for r in self.muon)
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
            if self.shards is not None:  # every rank takes the owners' updated weights
                self.shards.gather([r.part(r.param.data) for r in self.muon], group=self.group)
        active = [r for r in self.adamw if r.param.grad is not None]
        if active:
            self.B.gbo_clip_norm([r.part(r.param.grad) for r in active], self.max_norm, self.total_norm,
                                 self.coef, self._cws, dev_status=self.status)
            for wd in sorted({r.weight_decay for r in active}):  # one call per decay value
                params = [(r.part(r.param.data), r.part(r.param.grad), self.state[r.key]["m"],
                           self.state[r.key]["v"]) for r in active if r.weight_decay == wd]
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
