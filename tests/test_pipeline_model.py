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


def test_kernel_assignment_is_safe_with_tiny_segments():
    """Dozens of zero- to three-page segments per CTA (thousands of short
    requests): the stage hand-off stays safe with E4M3's ring (8 stages, 4
    consumer warps)."""
    rng = random.Random(11)
    for trial in range(100):
        segs = [rng.choice([0, 0, 1, 1, 1, 2, 3]) for _ in range(rng.randint(30, 50))]
        errs = simulate(segs, S=8, NW=4, assign="global", seed=trial)
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


def simulate_pool(static_pages, pool_pages, S, NW, R, seed, max_ticks=400000):
    """The kernel's protocol with a run-time pool: after its static segments
    the producer publishes each claimed pool segment (then an end marker)
    through a ring of R queue slots (mbarriers "qfull", one arrival, and
    "qempty", NW arrivals) and starts it on a stream position that is a
    multiple of NW, filling the gap with empty stages (arrive on "full"
    without a copy).  Each consumer warp reads the queue, releases the empty
    stages it owns and then takes the segment's pages k with k % NW == w.
    Checks every admitted page and queue entry, and that nothing deadlocks."""
    rng = random.Random(seed)
    full = [Barrier() for _ in range(S)]
    empty = [Barrier() for _ in range(S)]
    qfull = [Barrier() for _ in range(R)]
    qempty = [Barrier() for _ in range(R)]
    qempty_arrivals = [0] * R
    qval = [None] * R
    errors = []

    # stream layout: static segments back to back, pool segments aligned
    prod = []      # producer steps: ("page", k) | ("pad", k) | ("pub", j, value)
    cons = [[] for _ in range(NW)]   # ("page", k) | ("pad", k) | ("take", j, value) | ("bar", i)
    k = 0
    seg_no = 0
    for n in static_pages:
        for kk in range(k, k + n):
            prod.append(("page", kk))
            cons[kk % NW].append(("page", kk))
        for w in range(NW):
            cons[w].append(("bar", seg_no))
        k += n
        seg_no += 1
    for j, n in enumerate(list(pool_pages) + [None]):
        prod.append(("pub", j, n))
        for w in range(NW):
            cons[w].append(("take", j, n))
        if n is None:
            break
        ka = -(-k // NW) * NW
        for kk in range(k, ka):
            prod.append(("pad", kk))
            cons[kk % NW].append(("pad", kk))
        k = ka
        for kk in range(k, k + n):
            prod.append(("page", kk))
            cons[kk % NW].append(("page", kk))
        for w in range(NW):
            cons[w].append(("bar", seg_no))
        k += n
        seg_no += 1
    K = k
    issued, landed, consumed = [False] * K, [False] * K, [False] * K
    in_flight = []
    ppc = 0
    pc = [0] * NW
    at_bar = [None] * NW
    bar_pos = [{} for _ in range(NW)]
    for w in range(NW):
        for i, st in enumerate(cons[w]):
            if st[0] == "bar":
                bar_pos[w][st[1]] = i
    busy_until = [0] * NW
    tick = 0
    while tick < max_ticks:
        tick += 1
        still = []
        for t, kk in in_flight:
            if t <= tick:
                s = kk % S
                if full[s].completed != kk // S:
                    errors.append(f"copy of page {kk} completed the wrong phase of stage {s}")
                full[s].completed += 1
                landed[kk] = True
            else:
                still.append((t, kk))
        in_flight = still
        agents = list(range(NW + 1))
        rng.shuffle(agents)
        for a in agents:
            if a == NW:
                if ppc >= len(prod):
                    continue
                st = prod[ppc]
                if st[0] in ("page", "pad"):
                    kk = st[1]
                    s = kk % S
                    if empty[s].try_wait(((kk // S) & 1) ^ 1):
                        if kk >= S and not consumed[kk - S]:
                            errors.append(f"stage {s} reused before page {kk - S} was released")
                        issued[kk] = True
                        if st[0] == "page":
                            in_flight.append((tick + rng.randint(1, 40), kk))
                        else:
                            full[s].completed += 1
                            landed[kk] = True
                        ppc += 1
                else:
                    _, j, n = st
                    slot = j % R
                    if qempty[slot].try_wait(((j // R) & 1) ^ 1):
                        qval[slot] = (j, n)
                        qfull[slot].completed += 1
                        ppc += 1
                continue
            w = a
            if pc[w] >= len(cons[w]) or busy_until[w] > tick:
                continue
            st = cons[w][pc[w]]
            if st[0] in ("page", "pad"):
                kk = st[1]
                s = kk % S
                if full[s].try_wait((kk // S) & 1):
                    if not landed[kk]:
                        errors.append(f"warp {w} admitted stream position {kk} before it landed")
                    if kk + S < K and issued[kk + S]:
                        errors.append(f"warp {w} admitted position {kk} after its stage was refilled")
                    consumed[kk] = True
                    empty[s].completed += 1
                    busy_until[w] = tick + (rng.randint(0, 6) if st[0] == "page" else 0)
                    pc[w] += 1
            elif st[0] == "take":
                _, j, n = st
                slot = j % R
                if qfull[slot].try_wait((j // R) & 1):
                    if qval[slot] != (j, n):
                        errors.append(f"warp {w} read queue entry {qval[slot]} instead of {(j, n)}")
                    qempty_arrivals[slot] += 1
                    if qempty_arrivals[slot] == NW:
                        qempty_arrivals[slot] = 0
                        qempty[slot].completed += 1
                    pc[w] += 1
            else:
                x = st[1]
                at_bar[w] = x
                if all(at_bar[v] == x or pc[v] > bar_pos[v][x] for v in range(NW)):
                    for v in range(NW):
                        if at_bar[v] == x:
                            at_bar[v] = None
                            pc[v] += 1
        if errors:
            return errors
        if ppc == len(prod) and not in_flight and all(pc[w] == len(cons[w]) for w in range(NW)):
            return []
    return [f"no progress after {max_ticks} ticks (deadlock)"]


@pytest.mark.parametrize("NW,spw", [(4, 2), (4, 4), (2, 3), (8, 1)])
def test_pool_queue_and_alignment_are_safe(NW, spw):
    """Static segments, then pool segments of 0..9 pages (many shorter than
    NW, so most need padding), passed through a 4-slot queue."""
    rng = random.Random(100 + NW * 10 + spw)
    for trial in range(40):
        static = random_segments(rng, n_max=4, pages_max=30)
        pool = [rng.randint(0, 9) for _ in range(rng.randint(0, 25))]
        errs = simulate_pool(static, pool, S=NW * spw, NW=NW, R=4, seed=trial)
        assert not errs, (static, pool, errs[:3])
