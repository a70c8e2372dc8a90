"""CPU model of the decode kernel's shared-memory pipeline protocol.

The kernel's producer warp fills a ring of S stages with one TMA copy per
page (mbarrier "full", armed with expect_tx, completed by the copy) and its
consumer warps release stages through mbarrier "empty".  Waits are parity
waits, which only tell the current phase from the previous one.  This model
replays that protocol with randomised scheduling and out-of-order copy
completion and checks, at every wait that passes, that the data it admits is
really there and has not been overwritten, and that nothing deadlocks.

It is a model of the synchronisation only (no GPU): it reproduces the phase
aliasing that a ring shared round-robin by several consumers suffers, and
shows that the kernel's assignment (page k -> stage k % S -> warp k % NW,
with NW dividing S) is free of it.
"""
import random

import pytest


class Barrier:
    def __init__(self):
        self.completed = 0          # phases completed so far

    def try_wait(self, parity):
        return (self.completed & 1) != parity


def simulate(seg_pages, S, NW, assign, seed, max_ticks=200000):
    rng = random.Random(seed)
    K = sum(seg_pages)
    starts = [sum(seg_pages[:i]) for i in range(len(seg_pages))]
    full = [Barrier() for _ in range(S)]
    empty = [Barrier() for _ in range(S)]
    issued, landed, consumed = [False] * K, [False] * K, [False] * K
    in_flight = []                      # (land_tick, k)
    errors = []

    # consumer programs: list of ("page", k) and ("bar", seg) steps
    progs = []
    for w in range(NW):
        steps = []
        for si, (kb, n) in enumerate(zip(starts, seg_pages)):
            for k in range(kb, kb + n):
                lp = k - kb
                owner = (k % NW) if assign == "global" else (lp % NW)
                if owner == w:
                    steps.append(("page", k))
            steps.append(("bar", si))
        progs.append(steps)
    pc = [0] * NW
    busy_until = [0] * NW
    at_bar = [None] * NW
    prod_k = 0
    tick = 0
    while tick < max_ticks:
        tick += 1
        # land copies (any order)
        still = []
        for t, k in in_flight:
            if t <= tick:
                s = k % S
                if full[s].completed != k // S:
                    errors.append(f"copy of page {k} completed phase {full[s].completed} of stage {s}")
                full[s].completed += 1
                landed[k] = True
            else:
                still.append((t, k))
        in_flight = still
        agents = list(range(NW + 1))
        rng.shuffle(agents)
        for a in agents:
            if a == NW:                                     # producer
                if prod_k < K:
                    k = prod_k
                    s = k % S
                    if empty[s].try_wait(((k // S) & 1) ^ 1):
                        if k >= S and not consumed[k - S]:
                            errors.append(f"producer reused stage {s} before page {k - S} was consumed")
                        issued[k] = True
                        in_flight.append((tick + rng.randint(1, 40), k))
                        prod_k += 1
                continue
            w = a
            if pc[w] >= len(progs[w]) or busy_until[w] > tick:
                continue
            kind, x = progs[w][pc[w]]
            if kind == "page":
                k = x
                s = k % S
                if full[s].try_wait((k // S) & 1):
                    if not landed[k]:
                        errors.append(f"warp {w} admitted page {k} before its copy landed")
                    if k + S < K and issued[k + S]:
                        errors.append(f"warp {w} admitted page {k} after the stage was refilled")
                    consumed[k] = True
                    empty[s].completed += 1
                    if empty[s].completed != k // S + 1:
                        errors.append(f"empty barrier of stage {s} out of order at page {k}")
                    busy_until[w] = tick + rng.randint(0, 6)
                    pc[w] += 1
            else:
                at_bar[w] = x
                if all(at_bar[v] == x or pc[v] > progs[v].index(("bar", x)) for v in range(NW)):
                    for v in range(NW):
                        if at_bar[v] == x:
                            at_bar[v] = None
                            pc[v] += 1
        if errors:
            return errors
        if prod_k == K and not in_flight and all(pc[w] == len(progs[w]) for w in range(NW)):
            return []
    return [f"no progress after {max_ticks} ticks (deadlock)"]


def random_segments(rng, n_max=12, pages_max=40):
    return [rng.randint(0, pages_max) for _ in range(rng.randint(1, n_max))]


@pytest.mark.parametrize("NW,spw", [(4, 1), (4, 2), (4, 4), (2, 3), (8, 2)])
def test_kernel_assignment_is_safe(NW, spw):
    rng = random.Random(NW * 10 + spw)
    for trial in range(60):
        segs = random_segments(rng)
        errs = simulate(segs, S=NW * spw, NW=NW, assign="global", seed=trial)
        assert not errs, (segs, errs[:3])


def test_shared_stage_round_robin_aliases():
    """The assignment the kernel no longer uses - pages dealt round-robin per
    segment over a ring whose stages several warps share - admits pages that
    have not landed (parity aliasing) under some schedules."""
    rng = random.Random(1)
    found = False
    for trial in range(200):
        segs = [rng.randint(20, 200)]
        if simulate(segs, S=6, NW=4, assign="local", seed=trial):
            found = True
            break
    assert found
