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


# ------------------------------------------------------------------ buckets by 8-column tiles

def tiles_of(qo, G):
    """8-column tiles each request of a ragged batch needs (1 for no rows)."""
    return np.maximum(1, (G * np.diff(np.asarray(qo, np.int64)) + 7) // 8)


def expected_buckets(indptr, qo, G, Hkv, widest, one_tile_own, min_units, all_b):
    """The documented policy: every request to the widest tile count
    present, except the one-tile requests when they may and do hold enough
    (page, kv head) pairs, or every tile count with all_b.  Returns the
    buckets' tile counts (widest first; [] for one launch of the widest
    kernel) and each request's bucket tile count."""
    t = tiles_of(qo, G)
    if len(t) == 0:
        return [], t
    top = int(t.max())
    pages = np.diff(np.asarray(indptr, np.int64))
    one_units = Hkv * int(pages[t == 1].sum())
    own = {u: all_b or (u == 1 and one_tile_own and one_units >= min_units)
           for u in range(1, widest + 1)}
    dest = np.array([u if own[int(u)] else top for u in t])
    tiles = sorted(set(dest.tolist()), reverse=True)
    return ([] if tiles == [widest] else tiles), dest


def check_buckets(lib, indptr, last, qo, G, Hkv, widest, max_ctas, one_tile_own=False,
                  min_units=0, all_b=False, P=16):
    """The buckets' concatenated work list against its definition, rebuilt
    from independent pieces: per bucket, the head-grouped plan of its
    requests as a batch of their own (fa_plan_work_host_heads) with request
    ids, page positions, merge units and partial slots moved as documented;
    then coverage of the whole batch bit for bit, and partial slots of
    different buckets disjoint in columns."""
    res = lib.plan_work_host_buckets(indptr, last, qo, G, Hkv, P, widest, max_ctas,
                                     one_tile_own, min_units, all_b)
    tiles, dest = expected_buckets(indptr, qo, G, Hkv, widest, one_tile_own, min_units, all_b)
    if not tiles:
        assert res is None
        return None
    cta, seg, mer, btiles, first, cols = res
    assert list(btiles) == tiles
    indptr = np.asarray(indptr, np.int64)
    last = np.asarray(last, np.int64)
    np.testing.assert_array_equal(expand(seg), oracle.expected_coverage(indptr, Hkv))
    assert_token_coverage(seg, indptr, last, Hkv, P)
    bounds = list(first) + [len(cta) - 1]
    col_end, m0 = 0, 0
    spans = []
    for b, tb in enumerate(tiles):
        reqs = np.nonzero(dest == tb)[0]
        sub_ip = np.concatenate([[0], np.cumsum(np.diff(indptr)[reqs])]).astype(np.int32)
        ref_cta, ref_seg, ref_mer, ref_slots = lib.plan_work_host(
            sub_ip, last[reqs].astype(np.int32), Hkv, P, int(max_ctas[tb - 1]), 8, heads=True)
        c0, c1 = bounds[b], bounds[b + 1]
        assert c1 - c0 == len(ref_cta) - 1 <= max_ctas[tb - 1]
        np.testing.assert_array_equal(cta[c0:c1 + 1] - cta[c0], ref_cta)
        nc = 8 * tb
        slot_base = -(-col_end // nc)
        exp = ref_seg.astype(np.int64)
        exp[:, 2:4] += (indptr[reqs] - sub_ip[:-1])[exp[:, 0]][:, None]
        exp[:, 0] = reqs[exp[:, 0]]
        exp[:, 5] = np.where(exp[:, 5] >= 0, exp[:, 5] + slot_base, -1)
        exp[:, 6] = np.where(exp[:, 6] >= 0, exp[:, 6] + m0, -1)
        got = seg[cta[c0]:cta[c1]]
        np.testing.assert_array_equal(got, exp)
        expm = ref_mer.astype(np.int64)
        if len(expm):
            expm[:, 0] = reqs[expm[:, 0]]
            expm[:, 2] += slot_base
        np.testing.assert_array_equal(mer[m0:m0 + len(ref_mer)], expm)
        spans += [(int(s) * nc, (int(s) + 1) * nc) for s in got[:, 5] if s >= 0]
        m0 += len(ref_mer)
        col_end = (slot_base + ref_slots) * nc
    assert m0 == len(mer) and cols == col_end
    spans.sort()
    assert all(a[1] <= z[0] for a, z in zip(spans, spans[1:]))
    return res


def _ragged_rows(rng, lengths, G, widest):
    """Query rows per request for a random tile count 1..widest each (0
    rows for a request without tokens)."""
    rows = []
    for n in lengths:
        t = int(rng.integers(1, widest + 1))
        lo, hi = (8 * (t - 1)) // G + 1, (8 * t) // G
        rows.append(0 if n == 0 else min(int(n), int(rng.integers(lo, hi + 1))))
    return np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)


def test_buckets_random_batches(lib):
    rng = np.random.default_rng(41)
    for _ in range(80):
        G = int(rng.choice([1, 2, 4, 8]))
        widest = int(rng.integers(2, 5))
        B = int(rng.integers(1, 40))
        lengths = rng.integers(0, 900, size=B)
        lengths[rng.random(B) < 0.15] = 0
        Hkv = int(rng.choice([1, 2, 3, 8]))
        indptr, last = _table(lengths)
        qo = _ragged_rows(rng, lengths, G, widest)
        max_ctas = [int(x) for x in rng.integers(1, 200, size=4)]
        units = int(rng.integers(0, 2000))
        for own, all_b in ((False, False), (True, False), (False, True)):
            check_buckets(lib, indptr, last, qo, G, Hkv, widest, max_ctas, own, units, all_b)


def test_buckets_policy(lib):
    """Which launches the policy makes (group 8: tiles = query rows)."""
    indptr, last = _table([5000, 5000, 300, 900, 40])
    mc = [608, 760, 608, 456]
    qo = np.array([0, 1, 2, 5, 7, 11], np.int32)           # 1, 1, 3, 2, 4 rows
    one_units = 8 * 2 * 313                                  # the one-row requests' pairs
    r = check_buckets(lib, indptr, last, qo, 8, 8, 4, mc)    # 16-bit KV: one launch, widest
    assert r is None
    r = check_buckets(lib, indptr, last, qo, 8, 8, 4, mc, True, one_units)   # E4M3, enough
    assert list(r[3]) == [4, 1]
    r = check_buckets(lib, indptr, last, qo, 8, 8, 4, mc, True, one_units + 1)   # too little
    assert r is None
    r = check_buckets(lib, indptr, last, qo, 8, 8, 4, mc, all_b=True)
    assert list(r[3]) == [4, 3, 2, 1]
    qo3 = np.array([0, 1, 2, 5, 7, 10], np.int32)          # widest request: 3 rows
    r = check_buckets(lib, indptr, last, qo3, 8, 8, 4, mc)   # one launch on three warps
    assert list(r[3]) == [3] and r[4][0] == 0
    r = check_buckets(lib, indptr, last, qo3, 8, 8, 4, mc, True, one_units)
    assert list(r[3]) == [3, 1]
    qo2 = np.array([0, 2, 4, 6, 8, 10], np.int32)          # uniform 2 rows
    r = check_buckets(lib, indptr, last, qo2, 8, 8, 4, mc, True, 0)
    assert list(r[3]) == [2]


def test_buckets_rejects(lib):
    indptr, last = _table([100, 200])
    with pytest.raises(lib.FaError):                        # 5 rows at group 8 > 4 tiles
        lib.plan_work_host_buckets(indptr, last, [0, 5, 6], 8, 2, 16, 4, [8, 8, 8, 8])
    with pytest.raises(lib.FaError):                        # qo_indptr must start at 0
        lib.plan_work_host_buckets(indptr, last, [1, 2, 3], 8, 2, 16, 4, [8, 8, 8, 8])
    with pytest.raises(lib.FaError):                        # no grid for a used bucket
        lib.plan_work_host_buckets(indptr, last, [0, 1, 3], 8, 2, 16, 4, [8, 0, 8, 8],
                                   all_buckets=True)
