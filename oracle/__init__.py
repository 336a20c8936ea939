"""Plain fp64 CPU oracle for the hybrid Muon + AdamW optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code, constants or helpers with the
CUDA library under ``adamw_optimizer_step_gb300/csrc``.

Every function is written from the source pages, in fp64 numpy, step by step
in the order the pages give, with no blocking, fusion or reordering.  Each
docstring names the page and the section it follows.  The pages are:

* "Dual-Manifold Optimization in OMN" (aethrintelligence.in) -- the Muon path
  order, the 0.95 momentum, the max-abs rescale, the orientation rule, the
  rectangular scale, the AdamW hyper-parameters and the AdamW-only clip.
* "build_parameter_groups" (kimi-k3 docs) -- matrix views and split sizes.
* "MuonClip Optimizer" (wikifita) -- the cubic Newton-Schulz recurrence.
* The Chinese translation of the NorMuon paper (zskr.cn) -- Muon eqs. (1)-(5)
  in section 2.2 and the row-wise second moment of section 3.1.
* "Qwen3.8-Flash-Next notes / Optimizer" (cbphcr.github.io) -- the polar
  factor example, fused-matrix splitting, AdamW bias correction and
  decoupled decay.

Readings taken where the pages are silent or garbled are listed in the
docstrings of the functions that take them.

Parity unpinned: the NorMuon ordering choices (statistics on the unscaled
Newton-Schulz output, epsilon outside the square root, no bias correction on
the row second moment) and the form of its RMS-keeping learning-rate scale
(per matrix, to a caller-supplied target RMS, in place of the rectangular
scale).  The NorMuon algorithm listing is not printed on the page; the
oracle fixes these choices by reading and the tests pin only the properties
the page states (row normalisation, unit rows for an exactly orthogonal
update, an update RMS held at a target).
"""

from .views import sub_matrices, validate_view
from .muon import (
    momentum_update,
    nesterov_direction,
    prenormalize,
    newton_schulz,
    orthogonalize,
    rect_scale,
    normuon_rows,
    rms_match,
    weight_update,
    muon_step_tensor,
    ns_flops,
)
from .adamw import global_grad_norm, clip_coefficient, adamw_update

__all__ = [
    "sub_matrices",
    "validate_view",
    "momentum_update",
    "nesterov_direction",
    "prenormalize",
    "newton_schulz",
    "orthogonalize",
    "rect_scale",
    "normuon_rows",
    "rms_match",
    "weight_update",
    "muon_step_tensor",
    "ns_flops",
    "global_grad_norm",
    "clip_coefficient",
    "adamw_update",
]
