"""Role routing (CPU): the build_parameter_groups rules on toy modules with
the pages' worked shapes, and the OMN model's counts on the meta device."""

import json
import os

import pytest
import torch
import torch.nn as nn

from adamw_optimizer_step_gb300.routing import build_parameter_groups

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")))


class DenseFFN(nn.Module):
    def __init__(self, C=8, I=16):
        super().__init__()
        self.intermediate_size = I
        self.gate_up_proj = nn.Linear(C, 2 * I, bias=False)
        self.down_proj = nn.Linear(I, C, bias=False)


class KDA(nn.Module):
    def __init__(self, H=2, D=4, C=8):
        super().__init__()
        self.num_heads, self.d_head, self.d_model = H, D, C
        self.QKV = nn.Linear(C, 3 * H * D, bias=False)


class MLA(nn.Module):
    def __init__(self, H=2, D=4, Ds=2, Dv=6, Rq=8, Rkv=8):
        super().__init__()
        self.num_heads, self.d_head, self.d_shared, self.dv_head = H, D, Ds, Dv
        self.q_latent_dim, self.kv_latent_dim = Rq, Rkv
        self.W_UQ = nn.Linear(Rq, H * (D + Ds), bias=False)
        self.W_UKV = nn.Linear(Rkv, H * (D + Dv), bias=False)
        self.W_O = nn.Linear(H * Dv, 8, bias=True)


class Toy(nn.Module):
    def __init__(self):
        super().__init__()
        self.embed_tokens = nn.Embedding(50, 8)
        self.norm = nn.RMSNorm(8)
        self.ffn = DenseFFN()
        self.kda = KDA()
        self.mla = MLA()
        self.attn_res_proj = nn.Linear(8, 1, bias=False)
        self.conv = nn.Conv1d(8, 8, 3, groups=8, bias=False)
        self.frozen = nn.Linear(8, 8, bias=False)
        self.frozen.weight.requires_grad_(False)
        self.lm_head = nn.Linear(8, 50, bias=False)
        self.lm_head.weight = self.embed_tokens.weight  # tied


def test_page_views_and_roles():
    routes = {r.name: r for r in build_parameter_groups(Toy(), weight_decay=0.1)}
    cases = {c["stored"][0]: c for c in GOLDEN["views"]["cases"]}
    ffn = routes["ffn.gate_up_proj.weight"]
    assert ffn.algorithm == "muon" and list(ffn.view) == cases[32]["view"] and ffn.weight_decay == 0.1
    kda = routes["kda.QKV.weight"]
    assert kda.algorithm == "muon" and list(kda.view) == cases[24]["view"]
    ukv = routes["mla.W_UKV.weight"]
    assert list(ukv.view) == cases[20]["view"] and list(ukv.split) == cases[20]["split"]
    assert routes["mla.W_UQ.weight"].view == (2, 6, 8)
    # plain matrices take Muon without a view; biases and norms AdamW without decay
    assert routes["ffn.down_proj.weight"].algorithm == "muon" and routes["ffn.down_proj.weight"].view is None
    assert routes["mla.W_O.bias"].algorithm == "adamw" and routes["mla.W_O.bias"].weight_decay == 0.0
    assert routes["norm.weight"].algorithm == "adamw" and not routes["norm.weight"].decay
    assert routes["attn_res_proj.weight"].algorithm == "adamw" and not routes["attn_res_proj.weight"].decay
    # the tied embedding / head: one AdamW route, decayed (auxiliary); a 3-D filter: AdamW with decay
    assert "embed_tokens.weight" in routes and "lm_head.weight" not in routes
    assert routes["embed_tokens.weight"].algorithm == "adamw" and routes["embed_tokens.weight"].decay
    assert routes["conv.weight"].algorithm == "adamw" and routes["conv.weight"].decay
    # frozen parameters are skipped; every trainable parameter appears once
    assert "frozen.weight" not in routes
    model = Toy()
    n_trainable = len({id(p) for p in model.parameters() if p.requires_grad})
    assert len(build_parameter_groups(model)) == n_trainable


def test_refusals():
    with pytest.raises(ValueError):
        build_parameter_groups(nn.Module())
    frozen = nn.Linear(4, 4)
    for p in frozen.parameters():
        p.requires_grad_(False)
    with pytest.raises(ValueError):
        build_parameter_groups(frozen)
    bad = DenseFFN()
    bad.intermediate_size = 15  # (2, 15, 8) does not flatten to (32, 8)
    with pytest.raises(ValueError):
        build_parameter_groups(bad)


class OMNBlock(nn.Module):
    def __init__(self):
        super().__init__()
        self.input_norm = nn.RMSNorm(2048)
        self.q_norm = nn.RMSNorm(128)
        self.k_norm = nn.RMSNorm(128)
        self.q = nn.Linear(2048, 2048, bias=False)
        self.k = nn.Linear(2048, 512, bias=False)
        self.v = nn.Linear(2048, 512, bias=False)
        self.o = nn.Linear(2048, 2048, bias=False)
        self.gate = nn.Linear(2048, 5504, bias=False)
        self.up = nn.Linear(2048, 5504, bias=False)
        self.down = nn.Linear(5504, 2048, bias=False)


class OMN(nn.Module):
    def __init__(self):
        super().__init__()
        self.embed_tokens = nn.Embedding(128256, 2048)
        self.blocks = nn.ModuleList([OMNBlock() for _ in range(28)])
        self.final_norm = nn.RMSNorm(2048)
        self.lm_head = nn.Linear(2048, 128256, bias=False)
        self.lm_head.weight = self.embed_tokens.weight


def test_omn_routing_counts():
    """The OMN routing paragraph: 196 Muon tensors with 1,240,465,408
    parameters; AdamW 262,734,848 parameters, all without decay (the
    decayed AdamW group is empty)."""
    c = GOLDEN["omn_counts"]
    with torch.device("meta"):
        model = OMN()
    routes = build_parameter_groups(model, weight_decay=0.01, auxiliary_decay=False)
    muon = [r for r in routes if r.algorithm == "muon"]
    adamw = [r for r in routes if r.algorithm == "adamw"]
    assert len(muon) == c["muon_tensors"]
    assert sum(r.param.numel() for r in muon) == c["muon_params"]
    assert sum(r.param.numel() for r in adamw) == c["adamw_params"]
    assert all(not r.decay for r in adamw)


# ---------------------------------------------------------------------------
# fused projections with excluded row blocks (Qwen3.8-Flash-Next optimizer
# notes, section 4: split by meaning, orthogonalise each real sub-matrix,
# send gate and vector sub-blocks to AdamW, gather back into the fused layout)

from adamw_optimizer_step_gb300.routing import STANDARD_LAYOUTS, Block, Layout  # noqa: E402


class FusedGDN(nn.Module):
    """One fused input projection of a gated linear-attention block: per-head
    Q and K rows, per-head V rows, an output-gate block, and one decay and one
    beta row per head (scalars per head, vector-like), stored as one Linear."""

    def __init__(self, H=2, D=4, Dv=6, C=8):
        super().__init__()
        self.num_heads, self.d_head, self.dv_head = H, D, Dv
        self.in_proj = nn.Linear(C, 2 * H * D + 2 * H * Dv + 2 * H, bias=False)


def _gdn_blocks(f, lin):
    H, D, Dv, C = f.num_heads, f.d_head, f.dv_head, lin.in_features
    return (Block(2 * H * D, view=(2, H, D, C)),   # Q and K per head: Muon
            Block(H * Dv, view=(H, Dv, C)),         # V per head: Muon
            Block(H * Dv, path="adamw"),            # output gate: excluded
            Block(2 * H, path="adamw"))             # decay and beta rows: excluded


GDN_LAYOUT = Layout("in_proj", ("num_heads", "d_head", "dv_head"), _gdn_blocks)
LAYOUTS = STANDARD_LAYOUTS + (GDN_LAYOUT,)


class ToyFused(Toy):
    def __init__(self):
        super().__init__()
        self.gdn = FusedGDN()


def test_excluded_blocks_route_every_row_once():
    model = ToyFused()
    routes = build_parameter_groups(model, weight_decay=0.1, layouts=LAYOUTS)
    w = model.gdn.in_proj.weight
    parts = [r for r in routes if r.param is w]
    assert [(r.algorithm, r.rows) for r in parts] == [
        ("muon", (0, 16)), ("muon", (16, 28)), ("adamw", (28, 40)), ("adamw", (40, 44))]
    # every row of the fused weight exactly once, in order
    covered = [i for r in parts for i in range(*r.rows)]
    assert covered == list(range(w.shape[0]))
    assert parts[0].view == (2, 2, 4, 8) and parts[1].view == (2, 6, 8)
    # excluded blocks keep the matrix's decay; Muon blocks are decayed
    assert all(r.decay and r.weight_decay == 0.1 for r in parts)
    # the route keys are unique and name the rows
    keys = [r.key for r in routes]
    assert len(keys) == len(set(keys)) and "gdn.in_proj.weight[28:40]" in keys
    assert parts[2].shape == (12, 8) and parts[3].numel() == 4 * 8
    # row views are contiguous slices of the parameter
    assert parts[2].part(w).data_ptr() == w[28:].data_ptr() and parts[2].part(w).is_contiguous()
    # every trainable element is routed exactly once over the whole model
    n_routed = sum(r.numel() for r in routes)
    assert n_routed == sum(p.numel() for p in {id(p): p for p in model.parameters() if p.requires_grad}.values())
    # without the layout the fused weight is one Muon matrix
    plain = {r.key: r for r in build_parameter_groups(ToyFused())}
    assert plain["gdn.in_proj.weight"].algorithm == "muon" and plain["gdn.in_proj.weight"].rows is None


def test_layout_refusals():
    def bad(blocks):
        return (Layout("in_proj", ("num_heads", "d_head", "dv_head"), lambda f, lin: blocks),)

    with pytest.raises(ValueError):  # rows do not tile the weight
        build_parameter_groups(FusedGDN(), layouts=bad((Block(16), Block(20, path="adamw"))))
    with pytest.raises(ValueError):  # a view that does not flatten to its block
        build_parameter_groups(FusedGDN(), layouts=bad((Block(16, view=(2, 2, 5, 8)), Block(28, path="adamw"))))
    with pytest.raises(ValueError):  # split sizes that do not sum to the view's row axis
        build_parameter_groups(FusedGDN(), layouts=bad((Block(16, view=(2, 8, 8), split=(3, 4)),
                                                        Block(28, path="adamw"))))
    with pytest.raises(ValueError):  # an excluded block with a view
        build_parameter_groups(FusedGDN(), layouts=bad((Block(16, path="adamw", view=(2, 8, 8)),
                                                        Block(28, path="adamw"))))
    # two layouts declaring different geometry for one weight
    other = Layout("in_proj", ("num_heads",), lambda f, lin: (Block(44),))
    with pytest.raises(ValueError):
        build_parameter_groups(FusedGDN(), layouts=(GDN_LAYOUT, other))
