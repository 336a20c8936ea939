"""Random-schedule model of the streamed momentum pass's shared-memory ring.

The kernel (momentum_stream_kernel) has one producer that arms a stage's
"full" mbarrier (one arrival with expected bytes) and issues its bulk copies,
and consumer groups that wait on "full" with a parity wait, read the stage and
arrive on its "empty" mbarrier, on which the producer waits before it arms the
stage again.  A parity wait only tells the phase it names from the one after
it, so a waiter must never be a whole phase ahead of its barrier.  This model
plays producer, copy completions (in any order) and consumer groups in random
interleavings with the mbarriers' parity semantics, and checks:

- the kernel's mapping (block tile i to group i % groups, into that group's
  own ring of `per` stages) never passes a wait on the wrong phase and never
  arms a full barrier twice in one phase, for the group and stage counts the
  kernel builds with (read from its source);
- a single ring shared by the groups, whose size is not a multiple of the
  group count, does fail: that layout ended in a GPU fault (Xid 43) on tables
  with tens of tiles per block before it was replaced.
"""

import os
import random
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "adamw_optimizer_step_gb300", "csrc", "muon_elementwise.cu")


def kernel_ring_shape():
    """(groups, stages per group for bf16 G, for fp32 G) from the kernel's constants."""
    src = open(SRC).read()
    groups = int(re.search(r"#define GBO_MS_GROUPS (\d+)", src).group(1))
    budget = int(re.search(r"constexpr int kMsBudget = (\d+) \* 1024;", src).group(1)) * 1024
    flat = 4096
    per = [budget // (groups * (flat * g + flat * 4)) for g in (2, 4)]
    return groups, per


def simulate(n_tiles, groups, stage_of, use_of, n_stages, seed):
    """None if every wait passed on its own phase, else a description of the first violation."""
    rng = random.Random(seed)
    full_ph = [0] * n_stages      # completed phases of each full barrier
    full_armed = [False] * n_stages
    full_tx = [0] * n_stages
    empty_ph = [0] * n_stages     # completed phases of each empty barrier (one group's arrivals each)
    landed = [None] * n_stages    # the tile whose bytes sit in the stage
    in_flight = []
    nxt = 0
    gnext = list(range(groups))
    done = 0
    for _ in range(200000):
        if done == n_tiles:
            return None
        r = rng.random()
        if r < 0.3 and nxt < n_tiles:  # producer: wait empty, arm full, issue
            i = nxt
            s, u = stage_of(i), use_of(i)
            if u > 0:
                if (empty_ph[s] & 1) == ((u - 1) & 1):
                    continue  # still waiting
                if empty_ph[s] != u:
                    return "producer passed an empty wait on the wrong phase at tile %d" % i
            if full_armed[s]:
                return "full barrier armed twice in one phase at tile %d" % i
            full_armed[s] = True
            full_tx[s] += 1
            in_flight.append((s, i))
            nxt += 1
        elif r < 0.6 and in_flight:  # a copy lands (any order)
            s, i = in_flight.pop(rng.randrange(len(in_flight)))
            landed[s] = i
            full_tx[s] -= 1
            if full_armed[s] and full_tx[s] == 0:
                full_ph[s] += 1
                full_armed[s] = False
        else:  # a consumer group: wait full, read, arrive empty
            g = rng.randrange(groups)
            i = gnext[g]
            if i >= n_tiles:
                continue
            s, u = stage_of(i), use_of(i)
            if (full_ph[s] & 1) == (u & 1):
                continue  # still waiting
            if full_ph[s] != u + 1 or landed[s] != i:
                return "group %d passed a full wait on the wrong phase at tile %d" % (g, i)
            empty_ph[s] += 1
            gnext[g] += groups
            done += 1
    return "no progress"


def per_group(groups, per):
    return (lambda i: (i % groups) * per + (i // groups) % per,
            lambda i: (i // groups) // per, groups * per)


def shared_ring(stages):
    return (lambda i: i % stages, lambda i: i // stages, stages)


def test_kernel_rings_never_pass_a_wrong_phase():
    groups, pers = kernel_ring_shape()
    assert groups >= 1 and all(p >= 2 for p in pers)
    for per in pers:
        stage_of, use_of, n = per_group(groups, per)
        for seed in range(1500):
            bad = simulate(5 + seed % 60, groups, stage_of, use_of, n, seed)
            assert bad is None, (groups, per, seed, bad)


def test_shared_ring_of_the_faulting_layout_fails():
    stage_of, use_of, n = shared_ring(8)
    failures = sum(simulate(5 + seed % 60, 3, stage_of, use_of, n, seed) is not None for seed in range(1500))
    assert failures > 0
    # a shared ring is safe when its size is a multiple of the group count:
    # each stage then always serves the same group
    stage_of, use_of, n = shared_ring(6)
    assert all(simulate(5 + seed % 60, 3, stage_of, use_of, n, seed) is None for seed in range(500))
