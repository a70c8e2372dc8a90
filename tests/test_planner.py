"""Host planner (no GPU): the work list covers every (request, kv head, page)
and every (request, kv head, token) exactly once - bit-exact against the
oracle's coverage definitions - and balances pages across the persistent
grid."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_fa_gb300 import workloads as W


def expand(seg):
    """(request, kv head, page position) triples a work list covers, sorted."""
    if len(seg) == 0:
        return np.zeros((0, 3), np.int64)
    cnt = (seg[:, 3] - seg[:, 2]).astype(np.int64)
    r = np.repeat(seg[:, 0].astype(np.int64), cnt)
    h = np.repeat(seg[:, 1].astype(np.int64), cnt)
    starts = np.repeat(seg[:, 2].astype(np.int64), cnt)
    offs = np.arange(cnt.sum()) - np.repeat(np.cumsum(cnt) - cnt, cnt)
    out = np.stack([r, h, starts + offs], axis=1)
    order = np.lexsort((out[:, 2], out[:, 1], out[:, 0]))
    return out[order]


def segment_token_ranges(seg, indptr, P):
    """(request, kv head, first token, end token) of every non-empty segment,
    read the way the kernels read a segment: its pages are full except the
    last, which holds last_valid tokens."""
    seg = np.asarray(seg, np.int64).reshape(-1, 8)
    indptr = np.asarray(indptr, np.int64)
    s = seg[seg[:, 3] > seg[:, 2]]
    base = indptr[s[:, 0]]
    t0 = (s[:, 2] - base) * P
    t1 = (s[:, 3] - 1 - base) * P + s[:, 4]
    return np.stack([s[:, 0], s[:, 1], t0, t1], axis=1)


def expand_tokens(seg, indptr, P):
    """(request, kv head, token) triples a work list covers, sorted."""
    r = segment_token_ranges(seg, indptr, P)
    cnt = r[:, 3] - r[:, 2]
    assert np.all(cnt > 0), "a segment covers no token or a negative count"
    rep = lambda c: np.repeat(r[:, c], cnt)
    offs = np.arange(cnt.sum()) - np.repeat(np.cumsum(cnt) - cnt, cnt)
    out = np.stack([rep(0), rep(1), rep(2) + offs], axis=1)
    return out[np.lexsort((out[:, 2], out[:, 1], out[:, 0]))]


def token_runs(seg, indptr, P):
    """The same set as expand_tokens, as maximal runs (request, kv head,
    first, end) of consecutive tokens: pieces of a unit that abut merge into
    one run, a gap leaves two and an overlap or repeat leaves a run that
    starts inside the previous one - neither matches the oracle's one run
    [0, len) per unit."""
    r = segment_token_ranges(seg, indptr, P)
    r = r[np.lexsort((r[:, 2], r[:, 1], r[:, 0]))]
    runs = []
    for req, h, a, b in r.tolist():
        if runs and runs[-1][0] == req and runs[-1][1] == h and runs[-1][3] == a:
            runs[-1][3] = b
        else:
            runs.append([req, h, a, b])
    return np.array(runs, dtype=np.int64).reshape(-1, 4)


def assert_token_coverage(seg, indptr, last, Hkv, P=16, triples_limit=4_000_000):
    """Bit-exact token coverage against the oracle: as runs always, and as
    explicit triples when the batch is small enough to list them."""
    np.testing.assert_array_equal(token_runs(seg, indptr, P),
                                  oracle.expected_token_intervals(indptr, last, Hkv, P))
    if int(oracle.request_lengths(indptr, last, P).sum()) * Hkv <= triples_limit:
        np.testing.assert_array_equal(expand_tokens(seg, indptr, P),
                                      oracle.expected_token_coverage(indptr, last, Hkv, P))


POOL_TIERS, POOL_MIN = 4, 2   # the planner's pool schedule
SEG_COST = 2                  # fixed cost of a segment, in pages (no pool)


def expected_pages_per_cta(indptr, Hkv, max_ctas, min_pages, pool_pages, n_ctas):
    """Pages of the static part each CTA should hold: the stream of units
    (request-major, then kv head), each a fixed cost followed by its pages,
    cut into equal quotas of cost positions."""
    np_req = np.diff(np.asarray(indptr, np.int64))
    T = int(np_req.sum()) * Hkv
    n0 = max(1, min(max_ctas, -(-T // min_pages)))
    busy = int((np_req > 0).sum()) * Hkv
    c0 = SEG_COST if pool_pages == 0 else 0
    if c0 and -(-(T + c0 * busy) // n0) <= 2 * c0:
        c0 = 0
    C = T + c0 * busy
    S = C - pool_pages
    quota = -(-S // n0)
    units = np.repeat(np_req, Hkv)
    length = units + c0 * (units > 0)
    first = np.cumsum(length) - units          # position of each unit's first page
    pos = np.repeat(first, units) + (np.arange(int(units.sum())) - np.repeat(np.cumsum(units) - units, units))
    pos = pos[pos < S]
    owner = np.minimum(pos // quota, n_ctas - 1)
    return np.bincount(owner, minlength=n_ctas), C, quota


def check_work(lib, indptr, last, Hkv, max_ctas, min_pages=8, P=16, pool=0.0):
    cta, seg, mer, n_slots = lib.plan_work_host(indptr, last, Hkv, P, max_ctas, min_pages, pool)
    indptr = np.asarray(indptr, np.int64)
    B = len(indptr) - 1
    # coverage, bit-exact: pages, and tokens (last_valid of every segment)
    want = oracle.expected_coverage(indptr, Hkv)
    np.testing.assert_array_equal(expand(seg), want)
    assert_token_coverage(seg, indptr, last, Hkv, P)
    # every empty (request, head) still has exactly one empty segment
    for i in np.nonzero(np.diff(indptr) == 0)[0]:
        e = seg[(seg[:, 0] == i)]
        assert len(e) == Hkv and np.all(e[:, 2] == e[:, 3]) and np.all(e[:, 5] == -1)
    # CTA ranges partition the static segments, in order; the rest is the pool
    n_ctas = len(cta) - 1
    assert cta[0] == 0 and cta[-1] <= len(seg) and np.all(np.diff(cta) >= 0)
    assert 1 <= n_ctas <= max_ctas
    T = int(indptr[-1]) * Hkv
    pool_pages = int(pool * T)
    if pool_pages < n_ctas * POOL_MIN * 2:
        pool_pages = 0
    S = T - pool_pages
    pages = np.array([(seg[cta[c]:cta[c + 1], 3] - seg[cta[c]:cta[c + 1], 2]).sum()
                      for c in range(n_ctas)])
    pooled = seg[cta[-1]:]
    assert pages.sum() == S
    assert (pooled[:, 3] - pooled[:, 2]).sum() == pool_pages
    if pool_pages == 0:
        assert len(pooled) == 0
    if T:
        assert n_ctas <= -(-T // min_pages)
        # every CTA holds the pages of one quota of cost positions, the last
        # CTA the rest
        want, C, quota = expected_pages_per_cta(indptr, Hkv, max_ctas, min_pages, pool_pages,
                                                n_ctas)
        np.testing.assert_array_equal(pages, want)
        if pool_pages == 0:
            assert n_ctas == -(-C // quota)
            assert np.all(pages > 0)           # no CTA left without pages
    if pool_pages:
        # the pool is the end of the stream (request-major, then kv head, then
        # page) and its chunks are no longer than the first tier's
        key = lambda x: (x[:, 0].astype(np.int64) * Hkv + x[:, 1]) * (1 << 31) + x[:, 2]
        stat = seg[:cta[-1]]
        stat = stat[stat[:, 3] > stat[:, 2]]
        if len(stat):
            assert key(stat).max() < key(pooled[pooled[:, 3] > pooled[:, 2]]).min()
        first = -(-pool_pages // (2 * n_ctas))
        assert (pooled[:, 3] - pooled[:, 2]).max() <= max(first, POOL_MIN)
        units = len({(int(r), int(h)) for r, h in pooled[:, :2]})
        assert len(pooled) <= (POOL_TIERS + 1) * n_ctas + 1 + units
    # last_valid: the page that ends a request carries its last_page_len;
    # to_end: tokens from the segment's first token to the end of its request
    for s in seg:
        r, pe = s[0], s[3]
        if s[2] < pe:
            want_last = last[r] if pe == indptr[r + 1] else P
            assert s[4] == want_last
            length = (indptr[r + 1] - indptr[r] - 1) * P + last[r]
            assert s[7] == length - (s[2] - indptr[r]) * P
    # split units: slots are contiguous, cover the pieces in page order
    slots_seen = []
    for u, (r, h, s0, ns) in enumerate(mer):
        pieces = seg[(seg[:, 0] == r) & (seg[:, 1] == h)]
        assert len(pieces) == ns >= 2
        assert list(pieces[:, 5]) == list(range(s0, s0 + ns))
        assert np.all(pieces[:, 6] == u)
        assert np.all(pieces[1:, 2] == pieces[:-1, 3])
        slots_seen += list(range(s0, s0 + ns))
    assert sorted(slots_seen) == list(range(n_slots))
    unsplit = seg[seg[:, 5] < 0]
    assert np.all(unsplit[:, 6] == -1)
    for r, h in unsplit[:, :2]:
        assert ((seg[:, 0] == r) & (seg[:, 1] == h)).sum() == 1
    assert n_slots <= 2 * (n_ctas * (POOL_TIERS + 3) + 1)
    if pool_pages == 0:
        assert n_slots <= 2 * n_ctas
    return cta, seg, mer, n_slots


def _table(lengths, P=16):
    lengths = np.asarray(lengths, np.int64)
    indptr, _, last, _ = W.page_table(lengths, P, None, torch.Generator().manual_seed(0), False)
    return indptr.numpy(), last.numpy()


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_named_workloads_coverage(lib, name):
    cfg = W.CONFIGS[name]
    lengths = W.draw_lengths(cfg, torch.Generator().manual_seed(cfg.seed))
    indptr, last = _table(lengths)
    for max_ctas in (152 * 3, 152 * 2, 7):
        for pool in (0.0, 0.125, 0.3):
            check_work(lib, indptr, last, cfg.num_kv_heads, max_ctas, pool=pool)


def test_random_batches(lib):
    rng = np.random.default_rng(0)
    for _ in range(60):
        B = int(rng.integers(1, 40))
        lengths = rng.integers(0, 700, size=B)
        lengths[rng.random(B) < 0.15] = 0       # some empty requests
        Hkv = int(rng.choice([1, 2, 4, 8]))
        indptr, last = _table(lengths)
        check_work(lib, indptr, last, Hkv, int(rng.integers(1, 500)), int(rng.integers(1, 20)),
                   pool=float(rng.choice([0.0, 0.125, 0.4])))


def test_all_empty_and_single_page(lib):
    check_work(lib, *_table([0, 0, 0]), 2, 100)
    check_work(lib, *_table([1]), 1, 100)
    check_work(lib, *_table([16]), 4, 1)


def test_pool_chunks_shrink(lib):
    """gqa_uniform on 456 CTAs with 1/8 of the stream pooled: the chunks are
    claimed long ones first and end in short ones."""
    cfg = W.CONFIGS["gqa_uniform"]
    indptr, last = _table(W.draw_lengths(cfg, torch.Generator().manual_seed(cfg.seed)))
    cta, seg, mer, n_slots = check_work(lib, indptr, last, 8, 456, pool=0.125)
    pooled = seg[cta[-1]:]
    sizes = pooled[:, 3] - pooled[:, 2]
    assert sizes.sum() == 65536 // 8
    assert sizes[:100].mean() > 2 * sizes[-100:].mean()
    assert sizes[-100:].max() <= 3
    assert len(pooled) <= 5 * 456 + 64


def test_deterministic(lib):
    indptr, last = _table(np.random.default_rng(1).integers(1, 5000, size=50))
    a = lib.plan_work_host(indptr, last, 8, 16, 456)
    b = lib.plan_work_host(indptr, last, 8, 16, 456)
    for x, y in zip(a[:3], b[:3]):
        np.testing.assert_array_equal(x, y)


def test_host_array_forms(lib):
    """indptr and last_page_len taken as a list, numpy or torch CPU array of
    any integer type, contiguous or not, give the same work list (int32 CPU
    tensors are read in place, everything else is converted first)."""
    indptr, last = _table(np.random.default_rng(5).integers(1, 3000, size=37))
    ref = lib.plan_work_host(indptr, last, 4, 16, 120)
    ip32 = torch.tensor(indptr, dtype=torch.int32)
    strided = torch.stack([ip32, torch.zeros_like(ip32)], 1)[:, 0]   # stride 2
    assert not strided.is_contiguous()
    forms = [
        (list(map(int, indptr)), list(map(int, last))),
        (np.asarray(indptr, np.int64), np.asarray(last, np.int64)),
        (ip32, torch.tensor(last, dtype=torch.int32)),
        (ip32.to(torch.int64), torch.tensor(last, dtype=torch.int64)),
        (strided, torch.tensor(last, dtype=torch.int32)),
    ]
    for ip, ln in forms:
        got = lib.plan_work_host(ip, ln, 4, 16, 120)
        for x, y in zip(ref[:3], got[:3]):
            np.testing.assert_array_equal(x, y)
        assert ref[3] == got[3]
    with pytest.raises(ValueError):
        lib.plan_work_host(ip32, torch.tensor(last[:-1], dtype=torch.int32), 4, 16, 120)


def test_long_request_spread_over_grid(lib):
    """One 65536-token request with 32 kv heads fills every CTA (split-KV)."""
    indptr, last = _table([65536])
    cta, seg, mer, _ = check_work(lib, indptr, last, 32, 456)
    assert len(cta) - 1 == 456
    assert len(mer) == 32   # every (request, head) split


@pytest.mark.parametrize("indptr,last", [
    ([0, 2, 1], [16, 16]),      # decreasing
    ([1, 2], [16]),             # indptr[0] != 0
    ([0, 2], [0]),              # last_page_len below 1
    ([0, 2], [17]),             # last_page_len above page_size
])
def test_rejects_malformed(lib, indptr, last):
    with pytest.raises(lib.FaError) as e:
        lib.plan_work_host(np.array(indptr), np.array(last), 2, 16, 10)
    assert e.value.status == -1


def test_rejects_bad_sizes(lib):
    with pytest.raises(lib.FaError):
        lib.plan_work_host(np.array([0, 1]), np.array([3]), 0, 16, 10)
    with pytest.raises(lib.FaError):
        lib.plan_work_host(np.array([0, 1]), np.array([3]), 1, 16, 0)


def test_token_coverage_catches_planted_mistakes(lib):
    """The token-level check fails on the plausible planner mistakes that a
    page-level check cannot see: a full last page, a split piece that ends
    early, a piece that repeats a token, a dropped empty-request segment
    does not matter (no tokens) but a dropped page does."""
    indptr, last = _table([37, 0, 16, 250, 1, 1000])
    cta, seg, mer, n_slots = lib.plan_work_host(indptr, last, 2, 16, 9, 8, 0.0)
    assert_token_coverage(seg, indptr, last, 2)
    ends = np.nonzero((seg[:, 3] > seg[:, 2]) & (seg[:, 4] < 16))[0]
    assert len(ends)
    bad = seg.copy(); bad[ends[0], 4] = 16                       # last page taken as full
    with pytest.raises(AssertionError):
        assert_token_coverage(bad, indptr, last, 2)
    pieces = np.nonzero(seg[:, 5] >= 0)[0]
    assert len(pieces) >= 2
    first_piece = pieces[0]
    bad = seg.copy(); bad[first_piece, 4] = 15                   # a piece stops one token early
    with pytest.raises(AssertionError):
        assert_token_coverage(bad, indptr, last, 2)
    bad = seg.copy(); bad[first_piece, 3] += 1; bad[first_piece, 4] = 16   # overlaps the next piece
    with pytest.raises(AssertionError):
        assert_token_coverage(bad, indptr, last, 2)
    long_ = int(np.argmax(seg[:, 3] - seg[:, 2]))
    bad = seg.copy(); bad[long_, 2] += 1                         # a page dropped
    with pytest.raises(AssertionError):
        assert_token_coverage(bad, indptr, last, 2)


# ---------------------------------------------------------------- head-grouped plans

def expected_group_pages(indptr, Hkv, max_ctas, min_pages):
    """Pages each group of the head-grouped plan holds (for each kv head):
    the batch's pages in request order, a fixed cost before every non-empty
    request, cut into equal quotas of cost positions, one per group."""
    np_req = np.diff(np.asarray(indptr, np.int64))
    T = int(np_req.sum())
    groups = max(1, min(max_ctas // Hkv, -(-T // min_pages) if T else max_ctas // Hkv))
    busy = int((np_req > 0).sum())
    c0 = SEG_COST
    if -(-(T + c0 * busy) // groups) <= 2 * c0:
        c0 = 0
    C = T + c0 * busy
    quota = -(-C // groups) if C else 1
    if T:
        groups = (C - 1) // quota + 1
    length = np_req + c0 * (np_req > 0)
    first = np.cumsum(length) - np_req
    pos = np.repeat(first, np_req) + (np.arange(T) - np.repeat(np.cumsum(np_req) - np_req, np_req))
    return np.bincount(np.minimum(pos // quota, groups - 1), minlength=groups), groups


def check_heads_work(lib, indptr, last, Hkv, max_ctas, min_pages=8, P=16):
    cta, seg, mer, n_slots = lib.plan_work_host(indptr, last, Hkv, P, max_ctas, min_pages,
                                                heads=True)
    if max_ctas < Hkv:   # not one group: the stream plan
        ref = lib.plan_work_host(indptr, last, Hkv, P, max_ctas, min_pages)
        for x, y in zip(ref[:3], (cta, seg, mer)):
            np.testing.assert_array_equal(x, y)
        return cta, seg, mer, n_slots
    indptr = np.asarray(indptr, np.int64)
    n = len(cta) - 1
    # coverage, bit-exact, pages and tokens
    np.testing.assert_array_equal(expand(seg), oracle.expected_coverage(indptr, Hkv))
    assert_token_coverage(seg, indptr, last, Hkv, P)
    assert cta[0] == 0 and cta[-1] == len(seg) and np.all(np.diff(cta) >= 0)
    want, groups = expected_group_pages(indptr, Hkv, max_ctas, min_pages)
    assert n == groups * Hkv <= max_ctas
    for c in range(n):
        s = seg[cta[c]:cta[c + 1]]
        assert np.all(s[:, 1] == c % Hkv)                     # one kv head per CTA
        assert (s[:, 3] - s[:, 2]).sum() == want[c // Hkv]    # its group's share of pages
        if c % Hkv:                                           # the group's CTAs: same pieces
            first = seg[cta[c - c % Hkv]:cta[c - c % Hkv + 1]]
            np.testing.assert_array_equal(np.delete(s, [1, 5, 6], 1),
                                          np.delete(first, [1, 5, 6], 1))
    if int(indptr[-1]):
        assert np.all(want > 0)                               # every group holds pages
    # last_valid and to_end as the kernels read them
    for s in seg:
        r, pe = s[0], s[3]
        if s[2] < pe:
            assert s[4] == (last[r] if pe == indptr[r + 1] else P)
            length = (indptr[r + 1] - indptr[r] - 1) * P + last[r]
            assert s[7] == length - (s[2] - indptr[r]) * P
    # split units: contiguous slots in page order, every slot used once
    seen = []
    for u, (r, h, s0, ns) in enumerate(mer):
        pieces = seg[(seg[:, 0] == r) & (seg[:, 1] == h)]
        pieces = pieces[np.argsort(pieces[:, 2])]
        assert len(pieces) == ns >= 2
        assert list(pieces[:, 5]) == list(range(s0, s0 + ns)) and np.all(pieces[:, 6] == u)
        assert np.all(pieces[1:, 2] == pieces[:-1, 3])
        seen += list(range(s0, s0 + ns))
    assert sorted(seen) == list(range(n_slots))
    for r, h in seg[seg[:, 5] < 0][:, :2]:
        assert ((seg[:, 0] == r) & (seg[:, 1] == h)).sum() == 1
    assert n_slots <= 2 * n
    return cta, seg, mer, n_slots


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_heads_plan_named_workloads(lib, name):
    cfg = W.CONFIGS[name]
    indptr, last = _table(W.draw_lengths(cfg, torch.Generator().manual_seed(cfg.seed)))
    for max_ctas in (152 * 4, 152 * 3, 9, cfg.num_kv_heads):
        check_heads_work(lib, indptr, last, cfg.num_kv_heads, max_ctas)


def test_heads_plan_random_batches(lib):
    rng = np.random.default_rng(21)
    for _ in range(60):
        B = int(rng.integers(1, 40))
        lengths = rng.integers(0, 900, size=B)
        lengths[rng.random(B) < 0.15] = 0
        Hkv = int(rng.choice([1, 2, 3, 4, 5, 8]))
        indptr, last = _table(lengths)
        check_heads_work(lib, indptr, last, Hkv, int(rng.integers(Hkv, 500)),
                         int(rng.integers(1, 20)))


def test_heads_plan_edge_batches(lib):
    check_heads_work(lib, *_table([0, 0, 0]), 2, 100)
    check_heads_work(lib, *_table([0, 5, 0, 0]), 4, 100)
    check_heads_work(lib, *_table([1]), 1, 100)
    check_heads_work(lib, *_table([65536]), 32, 456)      # one long request over 14 groups
    check_heads_work(lib, *_table([100, 900]), 8, 4)       # fewer CTAs than kv heads
