"""The owner partition of the Muon weights (NorMuon paper, section 3.2;
Qwen3.8-Flash-Next optimizer notes, distributed Muon): LPT over executed
Newton-Schulz FLOPs, and the all-gather of the owners' updated weights, on
two gloo ranks on the CPU.  The per-rank step is the oracle's (test
infrastructure): what is under test is the partition and the exchange, which
must reproduce a single-rank step exactly."""

import itertools
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from adamw_optimizer_step_gb300 import build as build_mod
from adamw_optimizer_step_gb300.sharding import MuonShards, lpt_partition


def test_lpt_bounds_and_determinism():
    rng = np.random.default_rng(5)
    for world in (1, 2, 3, 8):
        for _ in range(30):
            costs = list(rng.integers(1, 1000, size=int(rng.integers(1, 40))).astype(float))
            owners, loads = lpt_partition(costs, world)
            # every item has exactly one owner, and the loads add up
            assert len(owners) == len(costs) and all(0 <= o < world for o in owners)
            for r in range(world):
                assert loads[r] == sum(c for c, o in zip(costs, owners) if o == r)
            # list scheduling's bound: mean load + (1 - 1/world) x the largest item
            assert max(loads) <= sum(costs) / world + (1 - 1 / world) * max(costs) + 1e-9
            assert lpt_partition(costs, world) == (owners, loads)


def test_lpt_within_four_thirds_of_optimal():
    """Brute force over every assignment of up to 9 items to 2 or 3 ranks."""
    rng = np.random.default_rng(6)
    for world in (2, 3):
        for _ in range(40):
            costs = list(rng.integers(1, 50, size=int(rng.integers(2, 9 if world == 2 else 7))).astype(float))
            best = min(max(sum(c for c, a in zip(costs, assign) if a == r) for r in range(world))
                       for assign in itertools.product(range(world), repeat=len(costs)))
            _, loads = lpt_partition(costs, world)
            assert max(loads) <= (4 / 3 - 1 / (3 * world)) * best + 1e-9


SHAPES = [(4 * 96, 1000, (4, 96, 1000), None), (2048, 512, None, None), (512, 2048, None, None),
          (640, 192, (2, 5, 64, 192), (20, 44)), (256, 256, None, None), (64, 64, None, None),
          (130, 600, None, None), (3 * 2 * 4, 8, (3, 2, 4, 8), None)]


def host_entries(seed):
    gen = torch.Generator().manual_seed(seed)
    out = []
    for rows, cols, view, split in SHAPES:
        out.append(dict(w=(torch.randn(rows, cols, generator=gen) * 0.02).to(torch.bfloat16),
                        g=(torch.randn(rows, cols, generator=gen) * 1e-3).to(torch.bfloat16),
                        mom=torch.randn(rows, cols, generator=gen) * 1e-3, view=view, split=split))
    return out


def test_costs_from_the_library():
    """Costs are the library's executed FLOPs per weight: a weight's cost is
    the sum over its view's matrices, a skipped weight costs nothing, and a
    longer matrix of the same short side costs more."""
    build_mod.build()
    entries = host_entries(1)
    sh = MuonShards(entries, 2, 0)
    assert len(sh.costs) == len(entries) and all(c > 0 for c in sh.costs)
    assert sh.costs[1] > sh.costs[5] and sh.costs[2] > sh.costs[5]
    skipped = [dict(e, g=None) if i == 0 else e for i, e in enumerate(entries)]
    assert MuonShards(skipped, 2, 0).costs[0] == 0.0
    assert sorted(sh.owned(0) + sh.owned(1)) == list(range(len(entries)))


def oracle_step(e):
    """One Muon step of one weight with the oracle: (W rounded to its dtype, B)."""
    import oracle
    W, B, _, _ = oracle.muon_step_tensor(e["w"].double().numpy(), e["g"].double().numpy(),
                                         e["mom"].double().numpy(), view=e["view"], split=e["split"], lr=0.02)
    return torch.from_numpy(W).to(e["w"].dtype), torch.from_numpy(B).float()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    entries = host_entries(2)
    shards = MuonShards(entries, world, rank)
    local = shards.local_entries(entries)
    for i, e in enumerate(local):
        if e["g"] is not None:  # this rank owns weight i: it steps it
            W, Bm = oracle_step(e)
            e["w"].copy_(W)
            e["mom"].copy_(Bm)
    shards.gather([e["w"] for e in entries])
    out[rank] = ([e["w"].clone() for e in entries], [e["mom"].clone() for e in entries], shards.owners,
                 shards.loads)
    dist.destroy_process_group()


def test_two_rank_owner_step_equals_single_rank_step():
    build_mod.build()
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    ref = host_entries(2)
    want = [oracle_step(e) for e in ref]
    owners = out[0][2]
    assert owners == out[1][2] and set(owners) == {0, 1}  # both ranks agree, both own weights
    loads = out[0][3]
    costs = MuonShards(ref, world, 0).costs
    assert max(loads) <= sum(costs) / world + (1 - 1 / world) * max(costs)
    for r in range(world):
        weights, moms, _, _ = out[r]
        for i, (W, Bm) in enumerate(want):
            # every rank holds every updated weight, bitwise the single-rank result
            assert torch.equal(weights[i], W), (r, i)
            # the momentum is kept current by the owner only
            if owners[i] == r:
                assert torch.equal(moms[i], Bm), (r, i)
            else:
                assert torch.equal(moms[i], ref[i]["mom"]), (r, i)
