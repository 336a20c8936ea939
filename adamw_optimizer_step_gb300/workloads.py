"""Seeded synthetic workloads: parameter-set shapes and input generators.

This module holds shapes, seeds and random draws only -- none of the
optimizer's arithmetic -- so that both the CUDA path and the CPU checker can
take their inputs from it.

Shapes follow the models the source pages describe:

* the OMN model ("Dual-Manifold Optimization in OMN"): 28 blocks at width
  2048, K/V 512 x 2048, FFN 5504, a 128,256 x 2,048 tied embedding;
* the matrix views of "build_parameter_groups" (kimi-k3 docs): gate_up
  (2, I, C), QKV (3, H, D, C), W_UQ (H, D + D_s, R_q), W_UKV (H, D + D_v, R_kv)
  with split (D, D_v).

Every tensor draws from its own seed, ``seed(config, tensor_index, role)``.
Small workloads are drawn on the CPU and copied where needed, so both sides
see identical bits; large ones are drawn on the device by torch's Philox
generator and sampled tensors are copied to the host.
"""

from dataclasses import dataclass, field
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class MuonTensor:
    """One stored 2-D weight on the Muon path, with its optional view/split."""

    name: str
    rows: int
    cols: int
    view: Optional[Tuple[int, ...]] = None
    split: Optional[Tuple[int, ...]] = None

    @property
    def numel(self):
        return self.rows * self.cols


@dataclass(frozen=True)
class AdamWTensor:
    """One tensor on the AdamW path (embedding, norm gain)."""

    name: str
    shape: Tuple[int, ...]

    @property
    def numel(self):
        n = 1
        for s in self.shape:
            n *= s
        return n


@dataclass
class Workload:
    """A named synthetic parameter set plus the step's hyper-parameters."""

    name: str
    index: int
    muon: list
    adamw: list = field(default_factory=list)
    w_dtype: torch.dtype = torch.bfloat16
    g_dtype: torch.dtype = torch.bfloat16
    precision: str = "bf16"
    ns_steps: int = 5
    mu: float = 0.95
    lr: float = 0.02
    normuon: bool = False
    beta2_row: float = 0.95
    eps_row: float = 1e-8
    w_std: float = 0.02
    g_std: float = 1e-3
    b_std: float = 0.0
    hot_row_frac: float = 0.0
    hot_row_scale: float = 100.0
    adamw_lr: float = 3e-4
    adamw_g_std: float = 1e-3
    adamw_p_std: float = 0.02
    steps: int = 1
    description: str = ""

    @property
    def muon_params(self):
        return sum(t.numel for t in self.muon)

    @property
    def adamw_params(self):
        return sum(t.numel for t in self.adamw)


def layer_d2048(prefix=""):
    """One transformer layer at d = 2048, FFN 5632 (Q, K, V, O square)."""
    return [
        MuonTensor(prefix + "q", 2048, 2048),
        MuonTensor(prefix + "k", 2048, 2048),
        MuonTensor(prefix + "v", 2048, 2048),
        MuonTensor(prefix + "o", 2048, 2048),
        MuonTensor(prefix + "gate_up", 11264, 2048, (2, 5632, 2048)),
        MuonTensor(prefix + "down", 2048, 5632),
    ]


def layer_d4096(prefix=""):
    """One 7B-shaped layer: d = 4096, FFN 11008, gate/up fused."""
    return [
        MuonTensor(prefix + "q", 4096, 4096),
        MuonTensor(prefix + "k", 4096, 4096),
        MuonTensor(prefix + "v", 4096, 4096),
        MuonTensor(prefix + "o", 4096, 4096),
        MuonTensor(prefix + "gate_up", 22016, 4096, (2, 11008, 4096)),
        MuonTensor(prefix + "down", 4096, 11008),
    ]


def layer_mla_kda(prefix=""):
    """One many-small-matrix layer, H = 32: W_UQ, W_UKV (split), QKV."""
    return [
        MuonTensor(prefix + "w_uq", 6144, 1536, (32, 192, 1536)),
        MuonTensor(prefix + "w_ukv", 8192, 512, (32, 256, 512), (128, 128)),
        MuonTensor(prefix + "qkv", 12288, 4096, (3, 32, 128, 4096)),
    ]


def tiny_fp32():
    muon = [
        MuonTensor("gate_up", 32, 8, (2, 16, 8)),
        MuonTensor("qkv", 24, 8, (3, 2, 4, 8)),
        MuonTensor("w_ukv", 20, 8, (2, 10, 8), (4, 6)),
    ]
    muon += [MuonTensor("sq%d" % i, 64, 64) for i in range(4)]
    muon += [MuonTensor("wide%d" % i, 64, 128) for i in range(2)]
    return Workload(
        name="tiny_fp32_views", index=1, muon=muon,
        adamw=[AdamWTensor("embedding", (1000, 64)), AdamWTensor("gain", (64,))],
        w_dtype=torch.float32, g_dtype=torch.float32, precision="f32",
        w_std=1.0, g_std=1.0, b_std=1.0, adamw_g_std=1.0, adamw_p_std=1.0,
        lr=0.02, steps=1,
        description="tiny fp32 set: gate_up (32,8)->(2,16,8); QKV (24,8)->(3,2,4,8); "
                    "W_UKV (20,8)->(2,10,8) split (4,6); 4x 64x64; 2x 64x128; "
                    "AdamW 1000x64 embedding + 64 gain")


def one_layer():
    return Workload(
        name="layer_d2048_ffn5632", index=2, muon=layer_d2048(), steps=10,
        description="one layer d=2048 FFN 5632, bf16 W/G, fp32 momentum, 10 steps")


def omn_shaped():
    muon = []
    for layer in range(24):
        muon += layer_d2048("l%d." % layer)
    adamw = [AdamWTensor("embedding", (128000, 2048))]
    adamw += [AdamWTensor("gain%d" % i, (2048,)) for i in range(49)]
    return Workload(
        name="omn_1.23B_muon_262M_adamw", index=3, muon=muon, adamw=adamw,
        hot_row_frac=0.01, steps=1,
        description="24 x (Q,K,V,O 2048^2, gate_up (2,5632,2048), down 2048x5632) "
                    "+ 128000x2048 tied embedding + 49x2048 gains on AdamW")


def many_small():
    muon = []
    for layer in range(48):
        muon += layer_mla_kda("l%d." % layer)
    return Workload(
        name="mla_kda_9216_matrices", index=4, muon=muon, steps=1,
        description="48 layers, H=32: W_UQ (32,192,1536); W_UKV (32,256,512) split "
                    "(128,128); QKV (3,32,128,4096)")


def normuon_7b():
    muon = []
    for layer in range(32):
        muon += layer_d4096("l%d." % layer)
    adamw = [AdamWTensor("embedding", (32000, 4096))]
    adamw += [AdamWTensor("gain%d" % i, (4096,)) for i in range(65)]
    return Workload(
        name="normuon_7b_shape", index=5, muon=muon, adamw=adamw, normuon=True, steps=1,
        description="32 x (Q,K,V,O 4096^2, gate_up (2,11008,4096), down 4096x11008), "
                    "NorMuon rows; 32000x4096 embedding + 65x4096 gains on AdamW")


WORKLOADS = {1: tiny_fp32, 2: one_layer, 3: omn_shaped, 4: many_small, 5: normuon_7b}


def first_layers(wl, n):
    """The same workload restricted to its first ``n`` layers (tensors named
    ``l<k>.*`` with k < n), for small profiling cases; other tensors stay."""
    keep = []
    for t in wl.muon:
        head = t.name.split(".")[0]
        if not (head.startswith("l") and head[1:].isdigit()) or int(head[1:]) < n:
            keep.append(t)
    wl.muon = keep
    wl.name = "%s_first_%d_layers" % (wl.name, n)
    return wl


def workload(index):
    return WORKLOADS[index]()


def omn_param_set():
    """The OMN model's optimizer-visible tensors, for the parameter-count check.

    28 blocks: Q, O 2048 x 2048; K, V 512 x 2048; gate, up 5504 x 2048; down
    2048 x 5504 on Muon.  AdamW: the 128,256 x 2,048 tied embedding; per
    block one input RMSNorm gain (2048) and Q/K norm gains (128 each); one
    final norm gain (2048).  The norm decomposition is a reading: the page
    gives only the AdamW total.
    """
    muon, adamw = [], [AdamWTensor("embedding", (128256, 2048))]
    for b in range(28):
        p = "b%d." % b
        muon += [
            MuonTensor(p + "q", 2048, 2048), MuonTensor(p + "k", 512, 2048),
            MuonTensor(p + "v", 512, 2048), MuonTensor(p + "o", 2048, 2048),
            MuonTensor(p + "gate", 5504, 2048), MuonTensor(p + "up", 5504, 2048),
            MuonTensor(p + "down", 2048, 5504),
        ]
        adamw += [AdamWTensor(p + "norm", (2048,)), AdamWTensor(p + "q_norm", (128,)),
                  AdamWTensor(p + "k_norm", (128,))]
    adamw.append(AdamWTensor("final_norm", (2048,)))
    return muon, adamw


# ---------------------------------------------------------------------------
# seeded draws

ROLE_W, ROLE_G, ROLE_B, ROLE_V, ROLE_HOT = 0, 1, 2, 3, 4
ROLE_P, ROLE_AG, ROLE_M, ROLE_AV = 5, 6, 7, 8


def seed(cfg, tensor_index, role):
    """Seed of one tensor: distinct per (workload, tensor, role)."""
    return 1_000_000 * int(cfg) + 16 * int(tensor_index) + int(role)


def _gen(device, s):
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def normal(shape, std, s, device="cpu", dtype=torch.float32):
    """N(0, std^2) draw of ``shape`` from seed ``s``, cast to ``dtype``."""
    x = torch.randn(shape, generator=_gen(device, s), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def hot_rows(rows, frac, s):
    """Seeded choice of ``round(frac * rows)`` row indices (at least one)."""
    k = max(1, int(round(frac * rows)))
    perm = torch.randperm(rows, generator=_gen("cpu", s))
    return perm[:k].sort().values


def muon_tensor_inputs(wl, i, device="cpu"):
    """W, G, B (and the NorMuon row vector) for Muon tensor ``i`` of ``wl``."""
    t = wl.muon[i]
    shape = (t.rows, t.cols)
    W = normal(shape, wl.w_std, seed(wl.index, i, ROLE_W), device, wl.w_dtype)
    G = normal(shape, wl.g_std, seed(wl.index, i, ROLE_G), device, torch.float32)
    if wl.hot_row_frac > 0:
        idx = hot_rows(t.rows, wl.hot_row_frac, seed(wl.index, i, ROLE_HOT)).to(device)
        G[idx] *= wl.hot_row_scale
    G = G.to(wl.g_dtype)
    if wl.b_std > 0:
        B = normal(shape, wl.b_std, seed(wl.index, i, ROLE_B), device, torch.float32)
    else:
        B = torch.zeros(shape, device=device, dtype=torch.float32)
    v = torch.zeros((t.rows,), device=device, dtype=torch.float32) if wl.normuon else None
    return W, G, B, v


def adamw_tensor_inputs(wl, i, device="cpu", state="zero"):
    """p, g, m, v for AdamW tensor ``i``.

    ``state="zero"`` starts the moments at zero; ``state="random"`` draws
    m ~ N(0, 1e-3^2) and v = |N(0, 1e-6^2)| so that the moment update is not
    hidden by a zero state.
    """
    t = wl.adamw[i]
    p = normal(t.shape, wl.adamw_p_std, seed(wl.index, 100000 + i, ROLE_P), device)
    g = normal(t.shape, wl.adamw_g_std, seed(wl.index, 100000 + i, ROLE_AG), device)
    if wl.hot_row_frac > 0 and len(t.shape) == 2:
        idx = hot_rows(t.shape[0], wl.hot_row_frac, seed(wl.index, 100000 + i, ROLE_HOT)).to(device)
        g[idx] *= wl.hot_row_scale
    if state == "zero":
        m = torch.zeros(t.shape, device=device, dtype=torch.float32)
        v = torch.zeros(t.shape, device=device, dtype=torch.float32)
    else:
        m = normal(t.shape, 1e-3, seed(wl.index, 100000 + i, ROLE_M), device)
        v = normal(t.shape, 1e-6, seed(wl.index, 100000 + i, ROLE_AV), device).abs_()
    return p, g, m, v
