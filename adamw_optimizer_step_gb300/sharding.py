"""Owner partition of the Muon weights over data-parallel ranks, and the
all-gather that hands every rank the owners' updated weights.

Newton-Schulz needs a whole matrix, and its cost grows with a higher power
of the matrix's short side, so splitting the optimizer work evenly by
element count leaves the ranks badly unbalanced.  Two of the pages answer
this the same way:

* the NorMuon paper (zskr.cn), section 3.2: instead of every device
  orthogonalising every parameter, each parameter tensor gets one owner
  (tensors sorted by size, then dealt out), the owner runs the
  orthogonalisation, and the result is sent back to all devices;
* the Qwen3.8-Flash-Next optimizer notes, distributed Muon: a static
  partitioner assigns complete matrices by their estimated NS FLOPs, the
  owner runs a step equivalent to the single-device one, and the result is
  put back into the original layout.

Here the unit is a stored weight (all of its view's matrices go to one
owner), its cost is the Newton-Schulz FLOPs the library's kernels execute
for it (``gbo_muon_plan_desc_flops``), and the assignment is longest
processing time first (LPT): weights in decreasing cost, each to the rank
with the least load so far.  LPT's largest load is at most the mean load
plus (1 - 1/world) times the largest single cost, and at most 4/3 of the
best possible largest load.

A rank's Muon plan lists every weight but passes a gradient only for the
weights it owns (a weight without a gradient is skipped: its weight and
momentum stay untouched on that rank), so only the owner keeps that
weight's momentum current.  After the step, :meth:`MuonShards.gather`
all-gathers each owner's updated weights (one flat buffer per rank and
dtype, padded to the longest) and copies them into place on every rank.
Collectives go through ``torch.distributed``: NCCL for device tensors, gloo
for host tensors.
"""

import torch
import torch.distributed as dist

from . import _binding as B


def lpt_partition(costs, world):
    """Owner rank of every item and the load of every rank.

    Items are taken in decreasing cost (ties by index), each to the rank
    with the least load (ties: the lowest rank), so the result depends only
    on the costs and ``world``.
    """
    if world < 1:
        raise ValueError("world must be >= 1")
    owners = [0] * len(costs)
    loads = [0.0] * world
    for i in sorted(range(len(costs)), key=lambda k: (-float(costs[k]), k)):
        r = min(range(world), key=lambda q: (loads[q], q))
        owners[i] = r
        loads[r] += float(costs[i])
    return owners, loads


class MuonShards:
    """The owner partition of one Muon table (a list of plan entries, as
    ``gbo_muon_plan_create`` takes them) over ``world`` ranks.

    ``costs`` (per entry) default to the executed Newton-Schulz FLOPs of
    each weight under ``plan_opts``.  Entries without a gradient cost
    nothing and are owned by the rank LPT gives them (none of them is
    stepped anywhere).
    """

    def __init__(self, entries, world, rank, costs=None, **plan_opts):
        if not 0 <= rank < world:
            raise ValueError("rank %d outside 0..%d" % (rank, world - 1))
        self.world, self.rank = world, rank
        self.costs = list(costs) if costs is not None else B.muon_desc_flops(entries, **plan_opts)
        if len(self.costs) != len(entries):
            raise ValueError("one cost per entry")
        self.owners, self.loads = lpt_partition(self.costs, world)

    def owned(self, rank=None):
        """Indices of the entries ``rank`` (default: this rank) owns."""
        r = self.rank if rank is None else rank
        return [i for i, o in enumerate(self.owners) if o == r]

    def local_entries(self, entries):
        """The table this rank plans and steps: every entry, with the
        gradient dropped from the ones another rank owns."""
        return [e if self.owners[i] == self.rank else dict(e, g=None) for i, e in enumerate(entries)]

    def gather(self, weights, group=None):
        """All-gather the owners' updated weights into ``weights`` (one
        tensor per entry, in table order, on every rank) in place."""
        if len(weights) != len(self.owners):
            raise ValueError("one weight per entry")
        if not all(w.is_contiguous() for w in weights):
            raise ValueError("weights must be contiguous")
        for dtype in sorted({w.dtype for w in weights}, key=str):
            idx = [[i for i in self.owned(r) if weights[i].dtype == dtype] for r in range(self.world)]
            sizes = [sum(weights[i].numel() for i in ix) for ix in idx]
            n = max(sizes)
            if n == 0:
                continue
            dev = weights[idx[self.rank][0]].device if idx[self.rank] else weights[0].device
            send = torch.zeros(n, dtype=dtype, device=dev)
            off = 0
            for i in idx[self.rank]:
                k = weights[i].numel()
                send[off:off + k].copy_(weights[i].reshape(-1))
                off += k
            recv = [torch.empty(n, dtype=dtype, device=dev) for _ in range(self.world)]
            dist.all_gather(recv, send, group=group)
            for r in range(self.world):
                if r == self.rank:
                    continue
                off = 0
                for i in idx[r]:
                    k = weights[i].numel()
                    weights[i].reshape(-1).copy_(recv[r][off:off + k])
                    off += k
