"""CUDA path vs the float64 oracle, through the C ABI, on seeded inputs.

Tolerances (absolute, on o and lse): fp32 1e-5, bf16 2e-2, E4M3 KV 3e-2
against the dequantised oracle.  Small cases are compared element by
element; the full-size workloads run in the launch configuration bench.py
times and are checked on sampled requests that the oracle computes one by
one (their pages copied out into a compact batch).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_fa_gb300 import workloads as W
from tests.helpers import oracle_decode, sub_batch

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2, torch.float16: 2e-2,
       torch.float8_e4m3fn: 3e-2}


def tol_for(b):
    return TOL[b.paged_kv.dtype] if b.paged_kv.dtype == torch.float8_e4m3fn else TOL[b.q.dtype]


def run_lib(fa, b, workspace=None, **kw):
    p = fa.plan(b.indptr, b.indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                b.head_dim, b.page_size, q_data_type=b.q.dtype, kv_data_type=b.paged_kv.dtype,
                workspace=workspace)
    o, lse = p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale, **kw)
    torch.cuda.synchronize()
    return p, o, lse


def compare(o, lse, ref_o, ref_lse, tol, rows=None, rel=0.0):
    """Max-abs check of o and lse; rel adds rel * |oracle o| to the o bound
    (for outputs whose magnitude makes the output dtype's own rounding
    exceed tol)."""
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o, lse = o[rows], lse[rows]
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), empty), "empty requests must give lse = -inf"
    if rel and o.size:
        excess = (np.abs(o - ref_o) - rel * np.abs(ref_o)).max()
        assert excess <= tol, f"max |o - oracle| - {rel}|oracle| = {excess:.3g} > {tol}"
        o = ref_o  # checked
    err_o = np.abs(o - ref_o).max() if o.size else 0.0
    err_l = np.abs(lse[~empty] - ref_lse[~empty]).max() if (~empty).any() else 0.0
    assert err_o <= tol, f"max |o - oracle| = {err_o:.3g} > {tol}"
    assert err_l <= tol, f"max |lse - oracle| = {err_l:.3g} > {tol}"
    return err_o, err_l


def check_coverage(p, b):
    """The plan's work list against the oracle's coverage definitions, bit
    for bit: every (request, kv head, page) and every (request, kv head,
    token) exactly once."""
    _, seg, _ = p.work()
    from tests.test_planner import assert_token_coverage, expand
    np.testing.assert_array_equal(expand(seg), oracle.expected_coverage(b.indptr.numpy(),
                                                                        b.num_kv_heads))
    assert_token_coverage(seg, b.indptr.numpy(), b.last_page_len.numpy(), b.num_kv_heads,
                          b.page_size)


# ------------------------------------------------------------------ small, element by element

def test_tiny_workload(lib, cuda):
    b = W.make_config_batch("tiny", device=cuda)
    p, o, lse = run_lib(lib, b)
    check_coverage(p, b)
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, TOL[torch.float32])


COMBOS = [(torch.float32, torch.float32), (torch.bfloat16, torch.bfloat16),
          (torch.float16, torch.float16), (torch.bfloat16, torch.float8_e4m3fn),
          (torch.float16, torch.float8_e4m3fn)]


@pytest.mark.parametrize("kernel", ["default", "simt"])
@pytest.mark.parametrize("q_dtype,kv_dtype", COMBOS, ids=lambda d: str(d).split(".")[-1])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_small_shapes(lib, cuda, monkeypatch, q_dtype, kv_dtype, head_dim, group, kernel):
    """Ragged lengths over several pages with partial tails, a 1-token and an
    empty request, spanning several CTAs and split units; on the default
    consumer (tensor cores where they apply) and on the CUDA-core one."""
    if kernel == "simt":
        monkeypatch.setenv("FADECODE_KERNEL", "simt")
    else:
        monkeypatch.delenv("FADECODE_KERNEL", raising=False)
    Hkv = 2
    lengths = [1, 0, 16, 17, 250, 1000, 33, 611]
    b = W.make_batch(batch_lengths=lengths, num_qo_heads=Hkv * group, num_kv_heads=Hkv,
                     head_dim=head_dim, q_dtype=q_dtype, kv_dtype=kv_dtype,
                     seed=7 + head_dim + group, device=cuda, pool_pages=200)
    p, o, lse = run_lib(lib, b)
    check_coverage(p, b)
    assert p.check() == 0
    mma_applies = (kernel == "default" and group >= 2 and kv_dtype != torch.float32
                   and head_dim * b.paged_kv.element_size() % 128 == 0)
    assert p.info["tensor_cores"] == int(mma_applies)
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, tol_for(b))


@pytest.mark.parametrize("merge", ["fused", "kernel"])
def test_many_splits_and_merge(lib, cuda, monkeypatch, merge):
    """One long request split over the whole grid plus short ones: exercises
    the split merge across many partial slots, done by the last CTA of each
    split request (default) or by the separate merge kernel."""
    if merge == "kernel":
        monkeypatch.setenv("FADECODE_MERGE", "kernel")
    else:
        monkeypatch.delenv("FADECODE_MERGE", raising=False)
    b = W.make_batch(batch_lengths=[9000, 3, 40], num_qo_heads=8, num_kv_heads=2, head_dim=128,
                     q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=3, device=cuda)
    p, o, lse = run_lib(lib, b)
    info = p.info
    assert info["num_merge_units"] >= 2 and info["num_partial_slots"] > 10
    assert info["fused_merge"] == int(merge == "fused")
    # the same plan again: the arrival counters must have been re-armed
    o2, lse2 = p.run(b.q, b.paged_kv)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, TOL[torch.bfloat16])


def test_shared_prefix_pages(lib, cuda):
    """Requests that point at the same pages (prefix sharing) read them in place."""
    b = W.make_batch(batch_lengths=[160, 160, 100], num_qo_heads=4, num_kv_heads=4, head_dim=64,
                     q_dtype=torch.float32, kv_dtype=torch.float32, seed=5, device=cuda)
    idx = b.indices.clone()
    idx[10:16] = idx[0:6]          # request 1 reuses request 0's first 6 pages
    b.indices = idx
    p, o, lse = run_lib(lib, b)
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, TOL[torch.float32])


def test_all_requests_empty(lib, cuda):
    b = W.make_batch(batch_lengths=[0, 0, 0], num_qo_heads=4, num_kv_heads=2, head_dim=64,
                     q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=1, device=cuda,
                     pool_pages=2)
    p, o, lse = run_lib(lib, b)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


POOL_CASES = [  # (q dtype, kv dtype, qo heads, kv heads, q_len, path)
    (torch.bfloat16, torch.bfloat16, 8, 2, 1, "run"),
    (torch.bfloat16, torch.float8_e4m3fn, 16, 2, 1, "run"),
    (torch.float32, torch.float32, 2, 2, 1, "run"),            # CUDA-core consumer
    (torch.bfloat16, torch.bfloat16, 4, 2, 2, "multi"),
    (torch.bfloat16, torch.float8_e4m3fn, 8, 2, 1, "token_scales"),
    (torch.bfloat16, torch.bfloat16, 8, 2, 1, "unified_max"),
]


@pytest.mark.parametrize("case", POOL_CASES, ids=lambda c: f"{c[5]}-{str(c[1]).split('.')[-1]}-g{c[2] // c[3]}")
def test_run_time_pool(lib, cuda, monkeypatch, case):
    """A batch large enough for the run-time pool (40 % of the page stream
    here): every output against the oracle, twice in a row (the claim
    counters re-arm), bitwise equal between the runs (a pool segment is
    computed the same way whichever CTA claims it)."""
    q_dt, kv_dt, hq, hkv, q_len, path = case
    monkeypatch.setenv("FADECODE_POOL", "0.4")
    # 3715 pages x 2 kv heads: enough for a pool on 4 CTAs per SM
    lengths = [9000, 7, 0, 5000, 16, 12000, 33, 8191, 640, 3000, 20000, 1500]
    lengths = [max(n, q_len) if q_len > 1 else n for n in lengths]  # room for the drafts
    b = W.make_batch(batch_lengths=lengths, num_qo_heads=hq, num_kv_heads=hkv, head_dim=128,
                     q_dtype=q_dt, kv_dtype=kv_dt, seed=120 + hq + q_len, device=cuda,
                     token_scales=(path == "token_scales"), q_len=q_len)
    if path == "multi":
        p = lib.plan_multi_token(b.indptr, b.indices, b.last_page_len, q_len, hq, hkv, 128, 16,
                                 q_data_type=q_dt, kv_data_type=kv_dt)
    else:
        p = lib.plan(b.indptr, b.indices, b.last_page_len, hq, hkv, 128, 16, q_data_type=q_dt,
                     kv_data_type=kv_dt)
    assert p.info["num_pool_segments"] > 0 and p.info["pool_pages"] > 0
    check_coverage(p, b)

    def once():
        if path == "token_scales":
            r = p.run_token_scales(b.q, b.paged_kv, b.extra["k_scales"], b.extra["v_scales"])
        elif path == "unified_max":
            r = p.run_unified_max(b.q, b.paged_kv, W.cauchy_schwarz_bound(b))
        else:
            r = p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale)
        torch.cuda.synchronize()
        return r

    o1, lse1 = once()
    o2, lse2 = once()
    assert p.check() == 0
    assert torch.equal(o1, o2) and torch.equal(lse1, lse2)
    ref_o, ref_lse = oracle_decode(b)
    compare(o2, lse2, ref_o, ref_lse, tol_for(b),
            rel=TOKEN_SCALE_REL if path == "token_scales" else 0.0)


@pytest.mark.parametrize("hq,hkv,kv_dtype", [(12, 3, torch.bfloat16), (40, 5, torch.float8_e4m3fn),
                                          (6, 3, torch.bfloat16)],
                         ids=["3-kv-heads", "5-kv-heads-e4m3", "3-kv-heads-g2"])
def test_head_groups_of_odd_size(lib, cuda, hq, hkv, kv_dtype):
    """Head-grouped plans whose groups do not divide the grid evenly (3 or 5
    kv heads): every row against the oracle, exact coverage."""
    b = W.make_batch(batch_lengths=[5000, 33, 0, 1200, 16, 777, 2], num_qo_heads=hq,
                     num_kv_heads=hkv, head_dim=128, q_dtype=torch.bfloat16, kv_dtype=kv_dtype,
                     seed=hq + hkv, device=cuda)
    p, o, lse = run_lib(lib, b)
    assert p.check() == 0 and p.info["num_ctas"] % hkv == 0
    check_coverage(p, b)
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, tol_for(b))


@pytest.mark.parametrize("kind", ["bf16-g4", "e4m3-g8", "ragged-q", "mha"])
def test_both_plan_kinds(lib, cuda, monkeypatch, kind):
    """The head-grouped plan (default) and the stream plan
    (FADECODE_PLAN=stream) over the same batch: both against the oracle,
    both with exact coverage, and within the output dtype's rounding of
    each other (their split pieces differ, so their sums run in other
    orders)."""
    lengths = [3000, 17, 0, 900, 1, 12000, 260, 48]
    if kind == "ragged-q":
        b = W.make_ragged_q_batch(batch_lengths=lengths, q_counts=[2, 1, 0, 4, 1, 3, 4, 2],
                                  num_qo_heads=32, num_kv_heads=8, head_dim=128,
                                  q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn,
                                  seed=61, device=cuda)
    else:
        hq, hkv, kv_dt = {"bf16-g4": (32, 8, torch.bfloat16), "e4m3-g8": (64, 8,
                          torch.float8_e4m3fn), "mha": (16, 16, torch.bfloat16)}[kind]
        b = W.make_batch(batch_lengths=lengths, num_qo_heads=hq, num_kv_heads=hkv,
                         head_dim=128, q_dtype=torch.bfloat16, kv_dtype=kv_dt, seed=62,
                         device=cuda)
    runner = run_ragged if kind == "ragged-q" else run_lib
    outs = {}
    for mode in ("heads", "stream"):
        if mode == "stream":
            monkeypatch.setenv("FADECODE_PLAN", "stream")
        else:
            monkeypatch.delenv("FADECODE_PLAN", raising=False)
        p, o, lse = runner(lib, b)
        assert p.check() == 0 and p.info["num_merge_units"] > 0
        check_coverage(p, b)
        outs[mode] = (o, lse)
        if mode == "heads":
            _, seg, _ = p.work()
            cta = p.work()[0]
            H = b.num_kv_heads
            for c in range(len(cta) - 1):   # CTA c serves kv head c % num_kv_heads
                assert np.all(seg[cta[c]:cta[c + 1], 1] == c % H)
    ref_o, ref_lse = oracle_decode(b)
    for o, lse in outs.values():
        compare(o, lse, ref_o, ref_lse, tol_for(b))
    diff = (outs["heads"][0].float() - outs["stream"][0].float()).abs().max().item()
    assert diff <= 2 ** -6


def _short_lengths(seed):
    rng = np.random.default_rng(seed)
    lengths = rng.integers(0, 49, size=2500)
    lengths[rng.random(lengths.size) < 0.3] = 0
    lengths[rng.random(lengths.size) < 0.1] = 1
    return lengths.tolist()


@pytest.mark.parametrize("q_dtype,kv_dtype,hq,hkv,token_scales", [
    (torch.bfloat16, torch.bfloat16, 32, 8, False),
    (torch.bfloat16, torch.float8_e4m3fn, 64, 8, False),
    (torch.bfloat16, torch.float8_e4m3fn, 64, 8, True),
], ids=["bf16", "e4m3", "e4m3-token-scales"])
def test_many_short_requests(lib, cuda, q_dtype, kv_dtype, hq, hkv, token_scales):
    """Thousands of short requests (a third empty, many of one token or one
    page): tens of thousands of units over one grid, so every CTA runs dozens
    of segments back to back; every output against the oracle."""
    b = W.make_batch(batch_lengths=_short_lengths(77), num_qo_heads=hq, num_kv_heads=hkv,
                     head_dim=128, q_dtype=q_dtype, kv_dtype=kv_dtype, seed=78, device=cuda,
                     token_scales=token_scales)
    p, o, lse = run_token_scales(lib, b) if token_scales else run_lib(lib, b)
    assert p.info["num_segments"] > 10 * p.info["num_ctas"]
    check_coverage(p, b)
    assert p.check() == 0
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, tol_for(b), rel=TOKEN_SCALE_REL if token_scales else 0.0)


@pytest.mark.parametrize("token_scales", [False, True], ids=["e4m3", "e4m3-token-scales"])
def test_many_short_requests_fresh_plans(lib, cuda, token_scales):
    """The shape that once exposed a missing cross-proxy fence (a stage
    released to its TMA refill before the warp's generic reads of its V rows
    were performed): 20 fresh E4M3 batches and plans of 2,500 short
    requests, each decoded once (its first launch) right after a bf16 launch
    of the same shape, every output against the oracle."""
    hot = W.make_batch(batch_lengths=_short_lengths(5), num_qo_heads=32, num_kv_heads=8,
                       head_dim=128, q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=6,
                       device=cuda)
    hot_plan = lib.plan(hot.indptr, hot.indices, hot.last_page_len, 32, 8, 128, 16,
                        q_data_type=torch.bfloat16, kv_data_type=torch.bfloat16)
    for it in range(20):
        hot_plan.run(hot.q, hot.paged_kv)
        b = W.make_batch(batch_lengths=_short_lengths(200 + it), num_qo_heads=64,
                         num_kv_heads=8, head_dim=128, q_dtype=torch.bfloat16,
                         kv_dtype=torch.float8_e4m3fn, seed=300 + it, device=cuda,
                         token_scales=token_scales)
        p, o, lse = run_token_scales(lib, b) if token_scales else run_lib(lib, b)
        assert p.check() == 0
        ref_o, ref_lse = oracle_decode(b)
        compare(o, lse, ref_o, ref_lse, tol_for(b), rel=TOKEN_SCALE_REL if token_scales else 0.0)
        del b, p, o, lse


def test_page_locked_host_buffers(lib, cuda):
    """q, the page ids, o and lse in page-locked host memory, read and written
    by the kernels directly: bitwise the same as with device buffers."""
    b = W.make_batch(batch_lengths=[3000, 17, 0, 900, 16, 5000], num_qo_heads=16,
                     num_kv_heads=4, head_dim=128, q_dtype=torch.bfloat16,
                     kv_dtype=torch.bfloat16, seed=141, device=cuda)
    p = lib.plan(b.indptr, b.indices, b.last_page_len, 16, 4, 128, 16,
                 q_data_type=torch.bfloat16, kv_data_type=torch.bfloat16)
    o_d, lse_d = p.run(b.q, b.paged_kv)
    idx_h = b.indices.cpu().pin_memory()
    ph = lib.plan(b.indptr, idx_h, b.last_page_len, 16, 4, 128, 16,
                  q_data_type=torch.bfloat16, kv_data_type=torch.bfloat16)
    q_h = b.q.cpu().pin_memory()
    o_h, lse_h = ph.run(q_h, b.paged_kv)
    torch.cuda.synchronize()
    assert o_h.is_pinned() and lse_h.is_pinned()
    assert ph.check() == 0
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    with pytest.raises(ValueError):       # pageable host memory is refused
        ph.run(b.q.cpu(), b.paged_kv)


def test_cuda_graph_capture(lib, cuda):
    """fa_decode_run only enqueues kernels (no allocation, no host sync), so a
    run can be captured into a CUDA graph and replayed; every replay equals
    the eager run bit for bit (split units re-arm their counters inside the
    kernel, so replays need no reset)."""
    b = W.make_batch(batch_lengths=[3000, 17, 0, 900, 16, 5000], num_qo_heads=16,
                     num_kv_heads=4, head_dim=128, q_dtype=torch.bfloat16,
                     kv_dtype=torch.bfloat16, seed=131, device=cuda)
    p = lib.plan(b.indptr, b.indices, b.last_page_len, 16, 4, 128, 16,
                 q_data_type=torch.bfloat16, kv_data_type=torch.bfloat16)
    assert p.info["num_merge_units"] > 0
    o = torch.empty_like(b.q)
    lse = torch.empty((b.batch, 16), dtype=torch.float32, device=cuda)
    p.run(b.q, b.paged_kv, out=o, lse=lse)
    torch.cuda.synchronize()
    ref_o, ref_lse = o.clone(), lse.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        p.run(b.q, b.paged_kv, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        p.run(b.q, b.paged_kv, out=o, lse=lse)
    for _ in range(3):
        o.zero_()
        lse.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    assert p.check() == 0


def test_cuda_graph_capture_buckets(lib, cuda, monkeypatch):
    """A ragged plan in four buckets (four launches a run) captured into a
    CUDA graph: every replay equals the eager run bit for bit."""
    monkeypatch.setenv("FADECODE_BUCKETS", "all")
    b = W.make_ragged_q_batch(batch_lengths=[3000, 40, 2500, 17, 5000], q_counts=[1, 4, 2, 0, 3],
                              num_qo_heads=16, num_kv_heads=2, head_dim=128,
                              q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn, seed=137,
                              device=cuda)
    p, ref_o, ref_lse = run_ragged(lib, b)
    assert p.info["num_buckets"] == 4 and p.info["num_merge_units"] > 0
    o, lse = torch.empty_like(ref_o), torch.empty_like(ref_lse)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale, out=o, lse=lse)
    for _ in range(3):
        o.zero_()
        lse.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    assert p.check() == 0


def test_ragged_q_buckets_fall_back_to_one_launch(lib, cuda, monkeypatch):
    """A workspace that holds the one-launch plan but not the plan in
    buckets: the plan falls back to one launch, with the same rows."""
    b = W.make_ragged_q_batch(batch_lengths=[3000, 40, 2500, 17, 5000], q_counts=[1, 4, 2, 0, 3],
                              num_qo_heads=16, num_kv_heads=2, head_dim=128,
                              q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn, seed=139,
                              device=cuda)
    monkeypatch.setenv("FADECODE_BUCKETS", "0")
    p1, o1, lse1 = run_ragged(lib, b)
    one = p1.info["workspace_bytes_used"]
    monkeypatch.setenv("FADECODE_BUCKETS", "all")
    p4, o4, lse4 = run_ragged(lib, b)
    four = p4.info["workspace_bytes_used"]
    assert p4.info["num_buckets"] == 4
    ws = torch.empty(one, dtype=torch.uint8, device=cuda)
    p, o, lse = run_ragged(lib, b, workspace=ws)
    assert p.check() == 0
    assert p.info["num_buckets"] == (1 if four > one else 4)
    ref_o, ref_lse = oracle_decode(b)
    for x, y in ((o, lse), (o1, lse1), (o4, lse4)):
        compare(x, y, ref_o, ref_lse, tol_for(b))


def test_stream_handle_is_current_stream(lib, cuda):
    """Without an explicit stream, calls go to torch's current stream of the
    current device, inside a stream context too; an explicit stream or raw
    handle is passed through."""
    assert lib._stream_handle(None) == torch.cuda.current_stream().cuda_stream
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert lib._stream_handle(None) == side.cuda_stream
        assert lib._stream_handle(None) == torch.cuda.current_stream().cuda_stream
    assert lib._stream_handle(side) == side.cuda_stream
    assert lib._stream_handle(side.cuda_stream) == side.cuda_stream


def test_dependent_launch_chain(lib, cuda):
    """Back-to-back decode launches in one stream, each second one decoding
    with q = the output of the launch just before it (nothing in between,
    fresh q for the first launch every round): it must read that q only
    once the first launch has completed, so its result equals the oracle on
    the first launch's actual output, round after round."""
    import dataclasses
    b = W.make_batch(batch_lengths=[3000, 17, 900, 5000, 64, 2048], num_qo_heads=16,
                     num_kv_heads=4, head_dim=128, q_dtype=torch.bfloat16,
                     kv_dtype=torch.bfloat16, seed=181, device=cuda)
    p = lib.plan(b.indptr, b.indices, b.last_page_len, 16, 4, 128, 16,
                 q_data_type=torch.bfloat16, kv_data_type=torch.bfloat16)
    gen = torch.Generator(device=cuda).manual_seed(182)
    rounds = 3
    qs = [torch.randn(b.q.shape, generator=gen, device=cuda).to(torch.bfloat16) * 4
          for _ in range(rounds)]
    o1s = [torch.zeros_like(b.q) for _ in range(rounds)]
    o2s = [torch.zeros_like(b.q) for _ in range(rounds)]
    l1s = [torch.zeros(b.q.shape[:-1], device=cuda) for _ in range(rounds)]
    l2s = [torch.zeros(b.q.shape[:-1], device=cuda) for _ in range(rounds)]
    torch.cuda.synchronize()
    for k in range(rounds):
        p.run(qs[k], b.paged_kv, out=o1s[k], lse=l1s[k])
        p.run(o1s[k], b.paged_kv, out=o2s[k], lse=l2s[k])
    torch.cuda.synchronize()
    assert p.check() == 0
    for k in range(rounds):
        ref1 = oracle_decode(dataclasses.replace(b, q=qs[k]))
        ref2 = oracle_decode(dataclasses.replace(b, q=o1s[k]))
        compare(o1s[k], l1s[k], ref1[0], ref1[1], TOL[torch.bfloat16])
        compare(o2s[k], l2s[k], ref2[0], ref2[1], TOL[torch.bfloat16])


def test_alternating_kernels_in_one_stream(lib, cuda):
    """Plans of different decode kernels launched in turn on one stream (a
    16-bit and an E4M3 page split, a ragged plan in two buckets; the
    library chains only launches of the same kernel as dependents): every
    run bitwise equal to the same plan run on its own, and the second plan
    reading q from the first's output sees it complete."""
    import dataclasses
    ba = W.make_batch(batch_lengths=[3000, 17, 900, 5000], num_qo_heads=16, num_kv_heads=2,
                      head_dim=128, q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=191,
                      device=cuda)
    bb = W.make_batch(batch_lengths=[700, 4000, 1, 2500], num_qo_heads=16, num_kv_heads=2,
                      head_dim=128, q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn,
                      seed=192, device=cuda)
    br = W.make_ragged_q_batch(batch_lengths=[3000, 40, 2500, 5000], q_counts=[1, 4, 2, 1],
                               num_qo_heads=16, num_kv_heads=2, head_dim=128,
                               q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn, seed=193,
                               device=cuda)
    pa, oa, la = run_lib(lib, ba)
    pb, ob, lb = run_lib(lib, bb)
    import os
    os.environ["FADECODE_BUCKETS"] = "all"
    try:
        pr, orr, lr = run_ragged(lib, br)
    finally:
        del os.environ["FADECODE_BUCKETS"]
    assert pr.info["num_buckets"] == 3
    ob2 = torch.empty_like(ob)
    lb2 = torch.empty_like(lb)
    for _ in range(3):
        xa, ya = pa.run(ba.q, ba.paged_kv)
        xb, yb = pb.run(oa, bb.paged_kv, k_scale=bb.k_scale, v_scale=bb.v_scale, out=ob2,
                        lse=lb2)
        xr, yr = pr.run(br.q, br.paged_kv, k_scale=br.k_scale, v_scale=br.v_scale)
        torch.cuda.synchronize()
        assert torch.equal(xa, oa) and torch.equal(ya, la)
        assert torch.equal(xr, orr) and torch.equal(yr, lr)
    ref = oracle_decode(dataclasses.replace(bb, q=oa))
    compare(ob2, lb2, ref[0], ref[1], tol_for(bb))
    assert pa.check() == 0 and pb.check() == 0 and pr.check() == 0


@pytest.mark.parametrize("merge", ["fused", "kernel"])
def test_deterministic_and_no_lse(lib, cuda, monkeypatch, merge):
    if merge == "kernel":
        monkeypatch.setenv("FADECODE_MERGE", "kernel")
    else:
        monkeypatch.delenv("FADECODE_MERGE", raising=False)
    b = W.make_batch(batch_lengths=[700, 5000, 64], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                     q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=11, device=cuda)
    p, o1, l1 = run_lib(lib, b)
    o2, l2 = p.run(b.q, b.paged_kv)
    o3, l3 = p.run(b.q, b.paged_kv, return_lse=False)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3) and l3 is None


def test_wrapper_api(lib, cuda):
    """The plan/run wrapper in the shape the pages use it."""
    b = W.make_batch(batch_lengths=[64] * 8, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                     q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=2, device=cuda)
    ws = torch.zeros(128 * 1024 * 1024, dtype=torch.uint8, device=cuda)
    w = lib.BatchDecodeWithPagedKVCacheWrapper(ws, "NHD")
    w.plan(b.indptr.to(cuda), b.indices, b.last_page_len.to(cuda), 32, 8, 128, 16,
           q_data_type=torch.bfloat16, kv_data_type=torch.bfloat16)
    out = w.run(b.q, b.paged_kv)
    torch.cuda.synchronize()
    ref_o, _ = oracle_decode(b)
    assert np.abs(out.float().cpu().numpy() - ref_o).max() <= TOL[torch.bfloat16]


def test_workspace_too_small_rejected(lib, cuda):
    b = W.make_batch(batch_lengths=[100] * 4, num_qo_heads=8, num_kv_heads=8, head_dim=64,
                     q_dtype=torch.float32, kv_dtype=torch.float32, seed=1, device=cuda)
    ws = torch.zeros(256, dtype=torch.uint8, device=cuda)
    with pytest.raises(lib.FaError) as e:
        run_lib(lib, b, workspace=ws)
    assert e.value.status == -3


def test_unsupported_rejected(lib, cuda):
    idx = torch.zeros(1, dtype=torch.int32, device=cuda)
    with pytest.raises(lib.FaError) as e:
        lib.plan([0, 1], idx, [1], 12, 4, 128, 16)      # group 3
    assert e.value.status == -2
    with pytest.raises(lib.FaError) as e:
        lib.plan([0, 1], idx, [1], 8, 8, 96, 16)        # head_dim 96
    assert e.value.status == -2
    with pytest.raises(lib.FaError) as e:
        lib.plan([0, 1], idx, [1], 8, 8, 128, 32)       # page_size 32
    assert e.value.status == -2


# ------------------------------------------------------------------ per-token FP8 scales

# Per-token magnitudes up to 2^3 make |o| reach tens, where a bf16 output's
# own rounding (half an ulp: 2^-9 relative) exceeds the absolute bound, so
# this workload is checked against abs 3e-2 + 2^-8 * |oracle o|.
TOKEN_SCALE_REL = 2.0 ** -8


def run_token_scales(lib, b):
    p = lib.plan(b.indptr, b.indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                 b.head_dim, b.page_size, q_data_type=b.q.dtype, kv_data_type=b.paged_kv.dtype)
    o, lse = p.run_token_scales(b.q, b.paged_kv, b.extra["k_scales"], b.extra["v_scales"])
    torch.cuda.synchronize()
    return p, o, lse


@pytest.mark.parametrize("q_dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("group", [2, 4, 8])
def test_token_scales_small(lib, cuda, q_dtype, group):
    b = W.make_batch(batch_lengths=[1, 0, 16, 17, 250, 1000, 33, 611], num_qo_heads=2 * group,
                     num_kv_heads=2, head_dim=128, q_dtype=q_dtype,
                     kv_dtype=torch.float8_e4m3fn, seed=40 + group, device=cuda, pool_pages=200,
                     token_scales=True)
    p, o, lse = run_token_scales(lib, b)
    assert p.check() == 0
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, TOL[torch.float8_e4m3fn], rel=TOKEN_SCALE_REL)


@pytest.mark.parametrize("q_dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("group", [2, 4, 8])
def test_token_scales_unit_magnitude(lib, cuda, q_dtype, group):
    """Per-token scales over N(0,1) values (no per-token magnitude spread),
    against the oracle at the plain FP8-KV bound, abs 3e-2, with no relative
    term: several CTAs, split units, empty and one-token requests."""
    b = W.make_batch(batch_lengths=[1, 0, 16, 17, 250, 1000, 33, 611, 3000, 4500],
                     num_qo_heads=4 * group, num_kv_heads=4, head_dim=128, q_dtype=q_dtype,
                     kv_dtype=torch.float8_e4m3fn, seed=50 + group, device=cuda,
                     token_scales=True, token_spread=0.0)
    p, o, lse = run_token_scales(lib, b)
    assert p.check() == 0
    assert p.info["num_merge_units"] > 0
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, TOL[torch.float8_e4m3fn])


def test_token_scales_uniform_scales_against_oracle(lib, cuda):
    """Every per-token scale set to one constant per tensor: the per-token
    kernel against the per-token oracle, and the per-tensor kernel against
    the per-tensor oracle with those constants, both at abs 3e-2 (scales of
    2^-6 keep |o| near 1, where a bf16 output's rounding is far below the
    bound)."""
    import dataclasses
    b = W.make_batch(batch_lengths=[300, 2000, 7], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                     q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn, seed=44, device=cuda,
                     token_scales=True, token_spread=0.0)
    ks = torch.full_like(b.extra["k_scales"], 0.015625)
    vs = torch.full_like(b.extra["v_scales"], 0.015625)
    bt = dataclasses.replace(b, extra={"k_scales": ks, "v_scales": vs})
    p = lib.plan(b.indptr, b.indices, b.last_page_len, 32, 8, 128, 16,
                 q_data_type=torch.bfloat16, kv_data_type=torch.float8_e4m3fn)
    o1, l1 = p.run_token_scales(b.q, b.paged_kv, ks, vs)
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle_decode(bt)
    compare(o1, l1, ref_o, ref_lse, TOL[torch.float8_e4m3fn])
    bp = dataclasses.replace(b, extra={}, k_scale=0.015625, v_scale=0.015625)
    o2, l2 = p.run(b.q, b.paged_kv, k_scale=0.015625, v_scale=0.015625)
    torch.cuda.synchronize()
    ref_o2, ref_lse2 = oracle_decode(bp)
    compare(o2, l2, ref_o2, ref_lse2, TOL[torch.float8_e4m3fn])


def test_token_scales_unsupported(lib, cuda):
    idx = torch.zeros(1, dtype=torch.int32, device=cuda)
    kv = torch.zeros((1, 2, 16, 8, 128), dtype=torch.float8_e4m3fn, device=cuda)
    sc = torch.ones((1, 8, 16), dtype=torch.float32, device=cuda)
    q = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device=cuda)
    p = lib.plan([0, 1], idx, [1], 8, 8, 128, 16, q_data_type=torch.bfloat16,
                 kv_data_type=torch.float8_e4m3fn)          # group 1: CUDA-core consumer only
    with pytest.raises(lib.FaError) as e:
        p.run_token_scales(q, kv, sc, sc)
    assert e.value.status == -2
    kvb = torch.zeros((1, 2, 16, 8, 128), dtype=torch.bfloat16, device=cuda)
    pb = lib.plan([0, 1], idx, [1], 8, 8, 128, 16, q_data_type=torch.bfloat16)
    rc = lib.library().fa_decode_run_token_scales(pb._h, q.data_ptr(), kvb.data_ptr(), 1, 0.0,
                                                  sc.data_ptr(), sc.data_ptr(),
                                                  torch.empty_like(q).data_ptr(), None,
                                                  torch.cuda.current_stream().cuda_stream)
    assert rc == -2   # bf16 KV has no per-token scales


# ------------------------------------------------------------------ per-head FP8 scales

def quantise_per_head(b, spread, seed):
    """Redraw b's E4M3 cache with K and V of kv head h at magnitude
    2^(u_h * spread) and one scale per head and half (amax / 448), as a
    cache quantised head by head would hold; returns the two scale tensors."""
    gen = torch.Generator(device=b.paged_kv.device).manual_seed(seed)
    pool, _, P, Hkv, D = b.paged_kv.shape
    scales = []
    for half in range(2):
        mag = torch.exp2((torch.rand(Hkv, generator=gen, device=b.paged_kv.device) * 2 - 1)
                         * spread)
        x = torch.randn((pool, P, Hkv, D), generator=gen, device=b.paged_kv.device) * mag[:, None]
        s = (x.abs().amax(dim=(0, 1, 3)) / 448.0).clamp_min(1e-12)
        b.paged_kv[:, half] = (x / s[:, None]).to(torch.float8_e4m3fn)
        scales.append(s.to(torch.float32).contiguous())
    return scales


def oracle_head_scales(b, ks, vs):
    from tests.helpers import as_bits
    q, qc = as_bits(b.q)
    kv, kc = as_bits(b.paged_kv)
    return oracle.batch_decode_head_scales(q, qc, kv, kc, b.indptr.numpy(),
                                           b.indices.cpu().numpy(), b.last_page_len.numpy(),
                                           b.num_qo_heads, b.num_kv_heads, b.head_dim,
                                           b.page_size, ks.cpu().numpy(), vs.cpu().numpy())


@pytest.mark.parametrize("q_dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv,d", [(16, 8, 128), (32, 4, 128), (64, 8, 128), (8, 8, 128),
                                      (16, 4, 64)],
                         ids=["g2", "g8", "g8-fp8kv", "g1-cuda-cores", "d64-cuda-cores"])
def test_head_scales_against_oracle(lib, cuda, q_dtype, hq, hkv, d):
    """One scale per kv head (fa_decode_run_head_scales) on a cache whose
    heads differ in magnitude by up to 2^2 either way: every row against the
    per-head oracle, on the tensor-core and the CUDA-core consumers, with
    split units.  |o| reaches about 16 on the largest heads, where the bf16
    output's own rounding (half an ulp, 2^-9 relative) passes an absolute
    3e-2, so the bound is abs 3e-2 + 2^-8 |oracle o|, as for the per-token
    spread workload."""
    b = W.make_batch(batch_lengths=[1, 16, 17, 300, 2900, 45], num_qo_heads=hq,
                     num_kv_heads=hkv, head_dim=d, q_dtype=q_dtype,
                     kv_dtype=torch.float8_e4m3fn, seed=hq + hkv + d, device=cuda)
    ks, vs = quantise_per_head(b, 2.0, seed=7 + hq)
    p = lib.plan(b.indptr, b.indices, b.last_page_len, hq, hkv, d, 16, q_data_type=q_dtype,
                 kv_data_type=torch.float8_e4m3fn)
    o, lse = p.run_head_scales(b.q, b.paged_kv, ks, vs)
    torch.cuda.synchronize()
    assert p.check() == 0 and p.info["num_merge_units"] > 0
    ref_o, ref_lse = oracle_head_scales(b, ks, vs)
    compare(o, lse, ref_o, ref_lse, TOL[torch.float8_e4m3fn], rel=2 ** -8)


def test_head_scales_equal_heads_is_per_tensor(lib, cuda):
    """Every head with the same two scales gives the per-tensor run (within
    the fp32 rounding of where the scale is folded in)."""
    b = W.make_batch(batch_lengths=[33, 700, 5000], num_qo_heads=32, num_kv_heads=8,
                     head_dim=128, q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn,
                     seed=31, device=cuda)
    p = lib.plan(b.indptr, b.indices, b.last_page_len, 32, 8, 128, 16,
                 q_data_type=torch.bfloat16, kv_data_type=torch.float8_e4m3fn)
    ref, ref_lse = p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale)
    ks = torch.full((8,), b.k_scale, dtype=torch.float32, device=cuda)
    vs = torch.full((8,), b.v_scale, dtype=torch.float32, device=cuda)
    o, lse = p.run_head_scales(b.q, b.paged_kv, ks, vs)
    torch.cuda.synchronize()
    assert (o.float() - ref.float()).abs().max().item() <= 2 ** -7
    assert (lse - ref_lse).abs().max().item() <= 1e-4


@pytest.mark.parametrize("buckets", ["default", "all"])
def test_head_scales_ragged_q(lib, cuda, monkeypatch, buckets):
    """Per-head scales on a ragged multi-token plan (group 8, 1..4 drafts:
    the column split; with FADECODE_BUCKETS=all one launch per tile count,
    every bucket kernel) against the ragged oracle run head by head."""
    if buckets == "all":
        monkeypatch.setenv("FADECODE_BUCKETS", "all")
    else:
        monkeypatch.delenv("FADECODE_BUCKETS", raising=False)
    lengths = [20, 400, 3000, 64, 9]
    counts = [1, 4, 2, 3, 4]
    b = W.make_ragged_q_batch(batch_lengths=lengths, q_counts=counts, num_qo_heads=16,
                              num_kv_heads=2, head_dim=128, q_dtype=torch.bfloat16,
                              kv_dtype=torch.float8_e4m3fn, seed=41, device=cuda)
    ks, vs = quantise_per_head(b, 1.0, seed=42)
    p = lib.plan_ragged_q(b.indptr, b.indices, b.last_page_len, b.extra["qo_indptr"], 16, 2,
                          128, 16, q_data_type=torch.bfloat16, kv_data_type=torch.float8_e4m3fn)
    o, lse = p.run_head_scales(b.q, b.paged_kv, ks, vs)
    torch.cuda.synchronize()
    assert p.check() == 0
    assert p.info["num_buckets"] == (4 if buckets == "all" else 1)
    # the heads do not interact: kv head h's rows are the per-tensor oracle
    # with head h's scales
    import dataclasses
    g = 8
    for h in range(2):
        bh = dataclasses.replace(b, k_scale=float(ks[h]), v_scale=float(vs[h]))
        ref_o, ref_lse = oracle_decode(bh)
        rows = slice(h * g, (h + 1) * g)
        compare(o[:, rows], lse[:, rows], ref_o[:, rows], ref_lse[:, rows],
                TOL[torch.float8_e4m3fn], rel=2 ** -8)


def test_head_scales_rejects(lib, cuda):
    idx = torch.zeros(1, dtype=torch.int32, device=cuda)
    q = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device=cuda)
    sc = torch.ones(8, dtype=torch.float32, device=cuda)
    kvb = torch.zeros((1, 2, 16, 8, 128), dtype=torch.bfloat16, device=cuda)
    pb = lib.plan([0, 1], idx, [1], 8, 8, 128, 16, q_data_type=torch.bfloat16)
    with pytest.raises(lib.FaError) as e:     # a 16-bit cache has no per-head scales
        pb.run_head_scales(q, kvb, sc, sc)
    assert e.value.status == -2
    kv = torch.zeros((1, 2, 16, 8, 128), dtype=torch.float8_e4m3fn, device=cuda)
    p = lib.plan([0, 1], idx, [1], 8, 8, 128, 16, q_data_type=torch.bfloat16,
                 kv_data_type=torch.float8_e4m3fn)
    rc = lib.library().fa_decode_run_head_scales(p._h, q.data_ptr(), kv.data_ptr(), 1, 0.0,
                                                 None, sc.data_ptr(),
                                                 torch.empty_like(q).data_ptr(), None,
                                                 torch.cuda.current_stream().cuda_stream)
    assert rc == -1
    with pytest.raises(ValueError):
        p.run_head_scales(q, kv, sc[:4], sc)


# ------------------------------------------------------------------ multi-token decode

def run_ragged(lib, b, workspace=None):
    p = lib.plan_ragged_q(b.indptr, b.indices, b.last_page_len, b.extra["qo_indptr"],
                          b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size,
                          q_data_type=b.q.dtype, kv_data_type=b.paged_kv.dtype,
                          workspace=workspace)
    o, lse = p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    return p, o, lse


# (group, most query tokens a request has): up to 8 columns the warps split
# the pages, beyond that each warp owns 8 of up to 32 columns
RAGGED_CASES = [(1, 8), (1, 20), (2, 3), (2, 12), (4, 2), (4, 5), (8, 1), (8, 2), (8, 4)]


@pytest.mark.parametrize("kv_dtype", [torch.bfloat16, torch.float8_e4m3fn], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("group,max_q", RAGGED_CASES)
def test_ragged_q_small(lib, cuda, kv_dtype, group, max_q):
    """A different number of query tokens per request (qo_indptr), 0 to
    max_q, drafts straddling page boundaries, requests split over CTAs, a
    request with no query rows: every row against the ragged-q oracle."""
    lengths = [8, 9, 16, 17, 250, 1000, 33, 611, 3000, 1, 40]
    rng = np.random.default_rng(100 * group + max_q)
    counts = [min(int(rng.integers(0, max_q + 1)), n) for n in lengths]
    counts[0] = min(max_q, lengths[0])      # the widest request
    counts[8] = max_q                        # and a long, split one
    counts[3] = 0                            # a request with no query rows
    b = W.make_ragged_q_batch(batch_lengths=lengths, q_counts=counts, num_qo_heads=2 * group,
                              num_kv_heads=2, head_dim=128, q_dtype=torch.bfloat16,
                              kv_dtype=kv_dtype, seed=70 + group + max_q, device=cuda)
    p, o, lse = run_ragged(lib, b)
    assert p.info["ragged_q"] == 1 and p.info["total_q_rows"] == sum(counts)
    assert p.info["num_merge_units"] > 0 and p.check() == 0
    check_coverage(p, b)
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, tol_for(b))
    # the same plan again: bitwise the same (counters re-armed)
    o2, lse2 = p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def bucket_of_segments(info, cta, seg):
    """Bucket index of every segment of a plan's work list."""
    nb = info["num_buckets"]
    first = list(info["bucket_first_cta"][:nb]) + [info["num_ctas"]]
    out = np.zeros(len(seg), np.int64)
    for b in range(nb):
        out[cta[first[b]]:cta[first[b + 1]]] = b
    return out


# (group, query rows per request): requests of 1 to 4 (or 3) 8-column tiles
BUCKET_CASES = [(8, [1, 4, 2, 0, 3, 4, 1, 1, 2, 3]), (4, [2, 8, 1, 0, 3, 6, 2, 1, 5, 4]),
                (2, [4, 12, 2, 0, 5, 16, 4, 1, 9, 8]), (1, [8, 20, 4, 0, 9, 32, 8, 1, 17, 24])]


@pytest.mark.parametrize("merge", ["fused", "kernel"])
@pytest.mark.parametrize("kv_dtype", [torch.bfloat16, torch.float8_e4m3fn], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("group,counts", BUCKET_CASES, ids=[f"g{g}" for g, _ in BUCKET_CASES])
def test_ragged_q_buckets(lib, cuda, monkeypatch, kv_dtype, group, counts, merge):
    """A ragged batch planned in buckets by the 8-column tiles its requests
    need (FADECODE_BUCKETS=all: a launch for every tile count present,
    however small): one launch each on the 8-column kernel, the two- and
    three-warp column splits and the four-warp one, their partial states
    sharing the workspace.  Every row against the oracle; the work list
    covers every page once; each bucket holds exactly the requests of its
    tile count; the buckets' partial states do not overlap; a one-launch
    plan (FADECODE_BUCKETS=0) gives the same rows within the bound; a rerun
    is bitwise the same; the plan's timing events bracket every launch."""
    if merge == "kernel":
        monkeypatch.setenv("FADECODE_MERGE", "kernel")
    else:
        monkeypatch.delenv("FADECODE_MERGE", raising=False)
    monkeypatch.setenv("FADECODE_BUCKETS", "all")
    lengths = [3000, 40, 2500, 17, 1000, 611, 5000, 9, 250, 4100]
    b = W.make_ragged_q_batch(batch_lengths=lengths, q_counts=counts, num_qo_heads=2 * group,
                              num_kv_heads=2, head_dim=128, q_dtype=torch.bfloat16,
                              kv_dtype=kv_dtype, seed=300 + group, device=cuda)
    p, o, lse = run_ragged(lib, b)
    info = p.info
    tiles = np.maximum(1, (group * np.asarray(counts) + 7) // 8)
    nb = info["num_buckets"]
    assert nb == len(set(tiles.tolist())) and p.check() == 0
    bq = np.asarray(info["bucket_q_len"][:nb])
    assert list(group * bq // 8) == sorted(set(tiles.tolist()), reverse=True)
    check_coverage(p, b)
    cta, seg, _ = p.work()
    bucket = bucket_of_segments(info, cta, seg)
    assert np.array_equal(tiles[seg[:, 0]], group * bq[bucket] // 8)
    assert (seg[:, 6] >= 0).any()
    # partial states in floats per row: slot x columns of the bucket's kernel
    cols = group * bq[bucket]
    spans = sorted((int(s[5]) * c, (int(s[5]) + 1) * c) for s, c in zip(seg, cols) if s[5] >= 0)
    assert all(a[1] <= z[0] for a, z in zip(spans, spans[1:]))
    assert spans[-1][1] <= info["num_partial_slots"] * group * info["q_len"]
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, tol_for(b))
    o2, lse2 = p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    ev1.record()
    p.set_timing_events(ev0, ev1)
    p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale, out=o2, lse=lse2)
    p.set_timing_events(None, None)
    torch.cuda.synchronize()
    assert ev0.elapsed_time(ev1) > 0 and torch.equal(o, o2)
    monkeypatch.setenv("FADECODE_BUCKETS", "0")
    p1, o1, lse1 = run_ragged(lib, b)
    assert p1.info["num_buckets"] == 1 and p1.check() == 0
    compare(o1, lse1, ref_o, ref_lse, tol_for(b))
    monkeypatch.delenv("FADECODE_BUCKETS")
    pd, od, lsed = run_ragged(lib, b)   # default: small buckets join wider ones
    assert pd.check() == 0 and pd.info["num_buckets"] <= nb
    compare(od, lsed, ref_o, ref_lse, tol_for(b))


@pytest.mark.parametrize("case", ["e4m3", "e4m3_little", "bf16"])
def test_ragged_q_bucket_policy(lib, cuda, monkeypatch, case):
    """The default plan of a ragged batch at group 8 whose widest request has
    3 tiles: one launch on the three-warp column split, plus, with E4M3 KV
    and enough work in the one-tile requests (here 1,252 pages x 8 kv heads,
    above 64 per SM), a second launch of those on the 8-column kernel.
    Every row against the oracle."""
    monkeypatch.delenv("FADECODE_BUCKETS", raising=False)
    kv = torch.bfloat16 if case == "bf16" else torch.float8_e4m3fn
    one = [40] * 4 if case == "e4m3_little" else [5000] * 4
    lengths = one + [3000, 2000, 700]
    counts = [1, 1, 1, 1, 3, 2, 3]
    b = W.make_ragged_q_batch(batch_lengths=lengths, q_counts=counts, num_qo_heads=64,
                              num_kv_heads=8, head_dim=128, q_dtype=torch.bfloat16, kv_dtype=kv,
                              seed=331, device=cuda)
    p, o, lse = run_ragged(lib, b)
    info = p.info
    assert p.check() == 0
    if case == "e4m3":
        assert info["num_buckets"] == 2 and info["bucket_q_len"][:2] == [3, 1]
        cta, seg, _ = p.work()
        bucket = bucket_of_segments(info, cta, seg)
        assert set(seg[bucket == 1, 0].tolist()) == {0, 1, 2, 3}
    else:
        assert info["num_buckets"] == 1 and info["bucket_q_len"][0] == 3
    check_coverage(p, b)
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, tol_for(b))


def test_ragged_q_one_token_each_is_decode(lib, cuda):
    """qo_indptr = 0, 1, 2, ...: the same rows as plain decode, within the
    bf16 bound of the oracle and of each other."""
    lengths = [300, 17, 4000, 1, 90]
    b = W.make_ragged_q_batch(batch_lengths=lengths, q_counts=[1] * 5, num_qo_heads=32,
                              num_kv_heads=8, head_dim=128, q_dtype=torch.bfloat16,
                              kv_dtype=torch.bfloat16, seed=91, device=cuda)
    _, o, lse = run_ragged(lib, b)
    import dataclasses
    bd = dataclasses.replace(b, extra={})
    _, o1, lse1 = run_lib(lib, bd)
    ref_o, ref_lse = oracle_decode(bd)
    compare(o, lse, ref_o, ref_lse, TOL[torch.bfloat16])
    assert (o.float() - o1.float()).abs().max().item() <= TOL[torch.bfloat16]


@pytest.mark.parametrize("kv_dtype", [torch.bfloat16, torch.float8_e4m3fn], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("group,q_len", [(8, 2), (8, 3), (8, 4), (4, 4), (4, 6), (2, 8),
                                         (2, 12), (1, 16), (1, 24)])
def test_multi_token_wide(lib, cuda, kv_dtype, group, q_len):
    """Uniform multi-token plans with more than 8 columns (group x q_len, up
    to 32): the group-8 shape verifying 2, 3 or 4 draft tokens; 16 and 24
    columns run on the column split of two and three warps (one bucket)."""
    lengths = [max(n, q_len) for n in (8, 9, 16, 17, 250, 1000, 33, 611, 2500)]
    b = W.make_batch(batch_lengths=lengths, num_qo_heads=2 * group, num_kv_heads=2,
                     head_dim=128, q_dtype=torch.bfloat16, kv_dtype=kv_dtype,
                     seed=80 + group + q_len, device=cuda, q_len=q_len)
    p, o, lse = run_multi(lib, b)
    assert p.info["q_len"] >= q_len and p.check() == 0
    tiles = group * q_len // 8
    assert p.info["num_buckets"] == 1
    assert group * p.info["bucket_q_len"][0] == 8 * tiles or tiles == 4
    check_coverage(p, b)
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, tol_for(b))


def run_multi(lib, b, workspace=None):
    p = lib.plan_multi_token(b.indptr, b.indices, b.last_page_len, b.q_len, b.num_qo_heads,
                             b.num_kv_heads, b.head_dim, b.page_size, q_data_type=b.q.dtype,
                             kv_data_type=b.paged_kv.dtype, workspace=workspace)
    o, lse = p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    return p, o, lse


@pytest.mark.parametrize("kv_dtype", [torch.bfloat16, torch.float8_e4m3fn], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("group,q_len", [(1, 2), (1, 4), (1, 8), (2, 2), (2, 4), (4, 2)])
def test_multi_token_small(lib, cuda, kv_dtype, group, q_len):
    """Draft tokens straddling page boundaries (lengths 8, 9, 17, 33, ...),
    requests split over CTAs, causal mask among the draft tokens."""
    b = W.make_batch(batch_lengths=[8, 9, 16, 17, 250, 1000, 33, 611], num_qo_heads=2 * group,
                     num_kv_heads=2, head_dim=128, q_dtype=torch.bfloat16, kv_dtype=kv_dtype,
                     seed=60 + group + q_len, device=cuda, pool_pages=200, q_len=q_len)
    p, o, lse = run_multi(lib, b)
    assert p.info["q_len"] == q_len and p.check() == 0
    check_coverage(p, b)
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, tol_for(b))


def test_multi_token_rejects(lib, cuda):
    b = W.make_batch(batch_lengths=[40, 3], num_qo_heads=8, num_kv_heads=2, head_dim=128,
                     q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=1, device=cuda,
                     q_len=4)
    with pytest.raises(lib.FaError) as e:      # request of 3 tokens cannot hold 4 queries
        run_multi(lib, b)
    assert e.value.status == -1
    idx = torch.zeros(1, dtype=torch.int32, device=cuda)
    with pytest.raises(lib.FaError) as e:      # group 8 x q_len 8 > 32 columns
        lib.plan_multi_token([0, 1], idx, [16], 8, 64, 8, 128, 16)
    assert e.value.status == -2


# ------------------------------------------------------------------ cascade (shared prefix)

def run_cascade(lib, b):
    pre, ip, idx, last = W.cascade_parts(b)
    p = lib.cascade_plan(pre, ip, idx, last, b.num_qo_heads, b.num_kv_heads, b.head_dim,
                         b.page_size, q_data_type=b.q.dtype, kv_data_type=b.paged_kv.dtype)
    o, lse = p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    return p, o, lse


@pytest.mark.parametrize("kernel", ["tcgen05", "mma"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("batch,hq,hkv,prefix_pages", [
    (6, 8, 2, 5),       # 24 rows: one partial row block, a partial last tile
    (40, 16, 4, 9),     # 160 rows per kv head: two row blocks
    (3, 16, 2, 1),      # group 8, a one-page prefix
    (20, 32, 4, 70),    # many tiles per chunk: TMEM score buffers and ring reused
    (80, 16, 4, 9),     # 320 rows per kv head: a block pair and a lone third block
])
def test_cascade_small(lib, cuda, monkeypatch, kernel, dtype, batch, hq, hkv, prefix_pages):
    """Cascade output equals attention over each request's full page list
    (shared prefix pages, then its own), checked against the oracle, with the
    prefix pass on tcgen05 (default) and on mma.sync."""
    if kernel == "mma":
        monkeypatch.setenv("FADECODE_CASCADE", "mma")
    else:
        monkeypatch.delenv("FADECODE_CASCADE", raising=False)
    rng = np.random.default_rng(batch + prefix_pages)
    sfx = rng.integers(0, 200, size=batch)
    sfx[0] = 0          # a request with no pages of its own
    sfx[-1] = 16        # one full page of its own
    b = W.make_cascade_batch(prefix_pages=prefix_pages, suffix_lengths=sfx, num_qo_heads=hq,
                             num_kv_heads=hkv, head_dim=128, dtype=dtype,
                             seed=70 + batch, device=cuda)
    p, o, lse = run_cascade(lib, b)
    assert p.check() == 0
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, TOL[dtype])


@pytest.mark.parametrize("kernel", ["tcgen05", "mma"])
@pytest.mark.parametrize("q_dtype,kv_dtype,head_dim", [
    (torch.bfloat16, torch.float8_e4m3fn, 128),
    (torch.float16, torch.float8_e4m3fn, 128),
    (torch.bfloat16, torch.bfloat16, 64),
    (torch.float16, torch.float16, 64),
], ids=["bf16-e4m3-d128", "f16-e4m3-d128", "bf16-d64", "f16-d64"])
@pytest.mark.parametrize("batch,hq,hkv,prefix_pages", [
    (6, 8, 2, 5),
    (40, 16, 4, 9),
    (20, 32, 4, 70),
])
def test_cascade_kv_dtypes(lib, cuda, monkeypatch, kernel, q_dtype, kv_dtype, head_dim, batch,
                           hq, hkv, prefix_pages):
    """Cascade over an E4M3 cache (per-tensor k/v scales) and at head_dim 64.
    The prefix pass of these runs on the mma.sync kernel whichever kernel is
    asked for (the tcgen05 one takes 16-bit D=128 only), so both settings
    must give the same bits; each is checked against the oracle's attention
    over the full page lists."""
    if kernel == "mma":
        monkeypatch.setenv("FADECODE_CASCADE", "mma")
    else:
        monkeypatch.delenv("FADECODE_CASCADE", raising=False)
    rng = np.random.default_rng(batch * 3 + prefix_pages)
    sfx = rng.integers(0, 200, size=batch)
    sfx[0] = 0
    sfx[-1] = 16
    b = W.make_cascade_batch(prefix_pages=prefix_pages, suffix_lengths=sfx, num_qo_heads=hq,
                             num_kv_heads=hkv, head_dim=head_dim, dtype=q_dtype,
                             kv_dtype=kv_dtype, seed=90 + batch, device=cuda)
    p, o, lse = run_cascade(lib, b)
    assert p.check() == 0
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, tol_for(b))
    with pytest.raises(TypeError):      # the plan's KV dtype is checked on every run
        other = torch.float16 if kv_dtype != torch.float16 else torch.bfloat16
        p.run(b.q, b.paged_kv.view(torch.uint8).to(other))


def test_cascade_overlap_graph_and_timing(lib, cuda, monkeypatch):
    """The prefix kernel on the plan's side stream (default), on the caller's
    stream (FADECODE_CASCADE_OVERLAP=0), with timing events set (the kernel
    alone) and replayed from a captured CUDA graph: the same kernels in every
    arrangement, so the outputs agree bit for bit."""
    rng = np.random.default_rng(5)
    b = W.make_cascade_batch(prefix_pages=40, suffix_lengths=rng.integers(0, 300, size=24),
                             num_qo_heads=16, num_kv_heads=4, head_dim=128,
                             dtype=torch.bfloat16, seed=171, device=cuda)
    pre, ip, idx, last = W.cascade_parts(b)
    def make():
        return lib.cascade_plan(pre, ip, idx, last, 16, 4, 128, 16, q_data_type=torch.bfloat16)
    monkeypatch.setenv("FADECODE_CASCADE_OVERLAP", "0")
    ref_o, ref_lse = make().run(b.q, b.paged_kv)
    monkeypatch.delenv("FADECODE_CASCADE_OVERLAP")
    p = make()
    o = torch.empty_like(b.q)
    lse = torch.empty((b.batch, 16), dtype=torch.float32, device=cuda)
    p.run(b.q, b.paged_kv, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    ev1.record()
    p.set_timing_events(ev0, ev1)
    o.zero_()
    p.run(b.q, b.paged_kv, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and ev0.elapsed_time(ev1) > 0
    p.set_timing_events(None, None)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        p.run(b.q, b.paged_kv, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        p.run(b.q, b.paged_kv, out=o, lse=lse)
    for _ in range(3):
        o.zero_()
        lse.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    assert p.check() == 0
    ref = oracle_decode(b)
    compare(o, lse, ref[0], ref[1], TOL[torch.bfloat16])


def test_cascade_many_plans(lib, cuda):
    """Cascade plans take their fork/join events from a per-device free list
    and give them back when destroyed: several plans alive at once, run
    interleaved, then destroyed and planned again, all give the same
    results bit for bit."""
    import gc
    rng = np.random.default_rng(9)
    b = W.make_cascade_batch(prefix_pages=24, suffix_lengths=rng.integers(0, 120, size=12),
                             num_qo_heads=16, num_kv_heads=4, head_dim=128,
                             dtype=torch.bfloat16, seed=191, device=cuda)
    pre, ip, idx, last = W.cascade_parts(b)
    def make():
        return lib.cascade_plan(pre, ip, idx, last, 16, 4, 128, 16, q_data_type=torch.bfloat16)
    ref_o, ref_lse = make().run(b.q, b.paged_kv)
    torch.cuda.synchronize()
    for _ in range(3):
        plans = [make() for _ in range(4)]
        outs = [p.run(b.q, b.paged_kv) for p in plans for _ in range(2)]
        torch.cuda.synchronize()
        for o, lse in outs:
            assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
        assert all(p.check() == 0 for p in plans)
        del plans, outs
        gc.collect()
    ref = oracle_decode(b)
    compare(ref_o, ref_lse, ref[0], ref[1], TOL[torch.bfloat16])


def test_cascade_rejects(lib, cuda):
    idx = torch.zeros(1, dtype=torch.int32, device=cuda)
    with pytest.raises(lib.FaError) as e:
        lib.cascade_plan(idx, [0, 0], idx, [16], 8, 8, 256, 16, q_data_type=torch.bfloat16)
    assert e.value.status == -2          # head_dim 256 not built
    with pytest.raises(lib.FaError) as e:
        lib.cascade_plan(idx, [0, 0], idx, [16], 8, 8, 64, 16, q_data_type=torch.bfloat16,
                         kv_data_type=torch.float8_e4m3fn)
    assert e.value.status == -2          # E4M3 at head_dim 64 not built
    with pytest.raises(lib.FaError) as e:
        lib.cascade_plan(idx, [0, 0], idx, [16], 8, 8, 128, 16, q_data_type=torch.float32)
    assert e.value.status == -2


# ------------------------------------------------------------------ unified max

# The window of the unified-max reference, natural-log units: the kernel
# re-centres a head whose maximum logit lies more than UM_ABOVE above the
# bound or more than UM_BELOW below it (16 and 64 in log2 units).
UM_ABOVE = 16 / math.log2(math.e)
UM_BELOW = 64 / math.log2(math.e)


def run_um(lib, b, bound):
    p = lib.plan(b.indptr, b.indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                 b.head_dim, b.page_size, q_data_type=b.q.dtype, kv_data_type=b.paged_kv.dtype)
    p.unified_max_fallbacks()          # start the count from zero
    o, lse = p.run_unified_max(b.q, b.paged_kv, bound, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    return p, o, lse, p.unified_max_fallbacks()


def max_logits(b):
    """Per (request, qo head) maximum of sm_scale * q . k, in float64 on the
    host (for choosing bounds in the tests; empty requests give -inf)."""
    q = b.q.double().cpu()
    kv = b.paged_kv.double().cpu()
    G = b.num_qo_heads // b.num_kv_heads
    ip, idx = b.indptr.numpy(), b.indices.cpu().numpy()
    out = np.full((b.batch, b.num_qo_heads), -np.inf)
    for r in range(b.batch):
        n = int(b.lengths[r])
        if n == 0:
            continue
        k = kv[idx[ip[r]:ip[r + 1]], 0].reshape(-1, b.num_kv_heads, b.head_dim)[:n]
        for h in range(b.num_qo_heads):
            s = k[:, h // G] @ q[r, h] / math.sqrt(b.head_dim)
            out[r, h] = s.max().item()
    return out


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [2, 4, 8])
@pytest.mark.parametrize("where", ["cauchy_schwarz", "inside_above", "inside_below",
                                   "far_above", "far_below"])
def test_unified_max_small(lib, cuda, head_dim, group, where):
    """Softmax referenced to a static bound: the same result as the oracle
    for any bound.  Inside the window no head is re-centred (weights down to
    2^-43 or up to 2^11 relative to the bound still give the oracle's
    answer); far outside it the re-centring fallback runs and still does."""
    Hkv = 2
    lengths = [1, 0, 16, 17, 250, 1000, 33, 611]
    b = W.make_batch(batch_lengths=lengths, num_qo_heads=Hkv * group, num_kv_heads=Hkv,
                     head_dim=head_dim, q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16,
                     seed=90 + head_dim + group, device=cuda, pool_pages=200)
    top = np.max(max_logits(b))
    bound = {"cauchy_schwarz": W.cauchy_schwarz_bound(b),
             "inside_above": top + 30.0,
             "inside_below": top - 8.0,
             "far_above": top + UM_BELOW + 40.0,
             "far_below": top - UM_ABOVE - 20.0}[where]
    p, o, lse, n = run_um(lib, b, bound)
    assert p.info["unified_max"] == 1 and p.check() == 0
    if where.startswith("far"):
        assert n > 0, "a bound outside the window must take the fallback"
    else:
        assert n == 0, f"{n} fallbacks for a bound inside the window"
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, TOL[torch.bfloat16])


@pytest.mark.parametrize("q_dtype,kv_dtype", [(torch.float16, torch.float16),
                                              (torch.bfloat16, torch.float8_e4m3fn),
                                              (torch.float16, torch.float8_e4m3fn)],
                         ids=["f16", "bf16-e4m3", "f16-e4m3"])
@pytest.mark.parametrize("group", [2, 4, 8])
@pytest.mark.parametrize("where", ["cauchy_schwarz", "top", "far_above", "far_below"])
def test_unified_max_f16_weights(lib, cuda, q_dtype, kv_dtype, group, where):
    """Unified max with f16 weights (f16 or E4M3 KV): window [bound - 8,
    bound + 15] in log2 units.  The oracle's result for any bound; far from
    the logits the exact re-centring runs."""
    Hkv = 2
    lengths = [1, 0, 16, 17, 250, 1000, 33, 611]
    b = W.make_batch(batch_lengths=lengths, num_qo_heads=Hkv * group, num_kv_heads=Hkv,
                     head_dim=128, q_dtype=q_dtype, kv_dtype=kv_dtype, seed=110 + group,
                     device=cuda, pool_pages=200)
    top = np.max(max_logits(b)) * b.k_scale
    bound = {"cauchy_schwarz": W.cauchy_schwarz_bound(b), "top": top,
             "far_above": top + 30.0, "far_below": top - 30.0}[where]
    p, o, lse, n = run_um(lib, b, bound)
    assert p.info["unified_max"] == 1 and p.check() == 0
    if where.startswith("far"):
        assert n > 0, "a bound outside the window must take the fallback"
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, tol_for(b))


def test_unified_max_many_splits(lib, cuda):
    """A long request split over the grid: partial states of one head carry
    different references (some pieces re-centred, some not) and still merge
    to the oracle's result."""
    b = W.make_batch(batch_lengths=[60000, 5, 300], num_qo_heads=16, num_kv_heads=4,
                     head_dim=128, q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=97,
                     device=cuda)
    top = np.max(max_logits(b))
    # the window's upper edge 1 below the top logit: pieces holding the top
    # logits re-centre, the others keep the bound
    p, o, lse, n = run_um(lib, b, top - UM_ABOVE - 1.0)
    assert p.info["num_merge_units"] > 0 and p.check() == 0
    assert 0 < n < p.info["num_segments"] * 4
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, TOL[torch.bfloat16])
    # same plan, regular softmax: results agree to rounding
    o2, lse2 = p.run(b.q, b.paged_kv)
    torch.cuda.synchronize()
    assert (o.float() - o2.float()).abs().max().item() <= TOL[torch.bfloat16]


def test_unified_max_rejects(lib, cuda):
    b = W.make_batch(batch_lengths=[40, 3], num_qo_heads=8, num_kv_heads=2, head_dim=128,
                     q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=1, device=cuda)
    p = lib.plan(b.indptr, b.indices, b.last_page_len, 8, 2, 128, 16,
                 q_data_type=torch.bfloat16, kv_data_type=torch.bfloat16)
    for bad in (math.inf, -math.inf, math.nan):
        with pytest.raises(lib.FaError) as e:
            p.run_unified_max(b.q, b.paged_kv, bad)
        assert e.value.status == -1
    # group 1, fp32 and multi-token plans have no unified-max kernel
    for q_dt, kv_dt, hq in [(torch.bfloat16, torch.bfloat16, 2),
                            (torch.float16, torch.float8_e4m3fn, 2),
                            (torch.float32, torch.float32, 8)]:
        bb = W.make_batch(batch_lengths=[40, 3], num_qo_heads=hq, num_kv_heads=2,
                          head_dim=128, q_dtype=q_dt, kv_dtype=kv_dt, seed=2, device=cuda)
        pp = lib.plan(bb.indptr, bb.indices, bb.last_page_len, hq, 2, 128, 16,
                      q_data_type=q_dt, kv_data_type=kv_dt)
        assert pp.info["unified_max"] == 0
        with pytest.raises(lib.FaError) as e:
            pp.run_unified_max(bb.q, bb.paged_kv, 10.0)
        assert e.value.status == -2
    bm = W.make_batch(batch_lengths=[40, 30], num_qo_heads=8, num_kv_heads=2, head_dim=128,
                      q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=3, device=cuda,
                      q_len=2)
    pm = lib.plan_multi_token(bm.indptr, bm.indices, bm.last_page_len, 2, 8, 2, 128, 16)
    assert pm.info["unified_max"] == 0


# ------------------------------------------------------------------ merge_states

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_merge_states(lib, cuda, dtype):
    g = torch.Generator(device=cuda).manual_seed(4)
    n, H, D = 37, 8, 128
    oa = torch.randn((n, H, D), generator=g, device=cuda).to(dtype)
    ob = torch.randn((n, H, D), generator=g, device=cuda).to(dtype)
    la = torch.randn((n, H), generator=g, device=cuda) * 4
    lb = torch.randn((n, H), generator=g, device=cuda) * 4
    la[0, :3] = -math.inf
    lb[0, 1:4] = -math.inf
    o, l = lib.merge_states(oa, la, ob, lb)
    torch.cuda.synchronize()
    ro, rl = oracle.merge_states(oa.double().cpu().numpy(), la.double().cpu().numpy(),
                                 ob.double().cpu().numpy(), lb.double().cpu().numpy())
    tol = TOL[dtype]
    assert np.abs(o.double().cpu().numpy() - ro).max() <= tol
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(l.cpu().numpy()), ~fin)
    assert np.abs(l.double().cpu().numpy()[fin] - rl[fin]).max() <= 1e-5
    # in place (outputs alias the a inputs)
    lib.merge_states(oa, la, ob, lb, out=oa, lse_out=la)
    torch.cuda.synchronize()
    assert torch.equal(oa, o) and torch.equal(la, l)


# ------------------------------------------------------------------ full-size workloads

def _row_chunks(b, max_kv_bytes=2 << 30):
    """Consecutive request ranges of b whose pages hold at most about
    max_kv_bytes of KV each (a request larger than that is a chunk of its
    own), so that the oracle's host copy of a chunk stays bounded."""
    per_page = b.paged_kv[0].numel() * b.paged_kv.element_size()
    npg = np.diff(b.indptr.numpy().astype(np.int64))
    chunks, cur, acc = [], [], 0
    for r in range(b.batch):
        cost = int(npg[r]) * per_page
        if cur and acc + cost > max_kv_bytes:
            chunks.append(cur)
            cur, acc = [], 0
        cur.append(r)
        acc += cost
    if cur:
        chunks.append(cur)
    return chunks


def compare_all_rows(b, o, lse, tol, rel=0.0):
    """Every output row of a full-size batch against the oracle, element by
    element, one bounded chunk of requests at a time (ragged q: the chunk's
    requests' query rows)."""
    for reqs in _row_chunks(b):
        rows = reqs
        if "qo_indptr" in b.extra:
            qo = np.asarray(b.extra["qo_indptr"], np.int64)
            rows = np.concatenate([np.arange(qo[r], qo[r + 1]) for r in reqs])
        ref_o, ref_lse = oracle_decode(sub_batch(b, reqs))
        compare(o, lse, ref_o, ref_lse, tol, rows=rows, rel=rel)


@pytest.mark.parametrize("name", ["gqa_uniform", "ragged", "long_split", "fp8_kv",
                                  "fp8_kv_token_scales", "spec_decode", "cascade",
                                  "gqa_unified_max", "spec_decode_ragged"])
def test_full_size_workloads(lib, cuda, name):
    """The full-size workloads in the launch configuration bench.py times:
    every output row of every request against the oracle (ragged: all 450
    requests, the ones the plan splits over several CTAs included)."""
    b = W.make_config_batch(name, device=cuda)
    if "k_scales" in b.extra:
        p, o, lse = run_token_scales(lib, b)
    elif "qo_indptr" in b.extra:
        p, o, lse = run_ragged(lib, b)
    elif b.q_len > 1:
        p, o, lse = run_multi(lib, b)
    elif name == "gqa_unified_max":
        p, o, lse, n = run_um(lib, b, W.cauchy_schwarz_bound(b))
        assert n == 0
    elif "prefix_pages" in b.extra:
        p, o, lse = run_cascade(lib, b)
        # and the same batch through plain decode
        _, o2, lse2 = run_lib(lib, b)
        assert (o.float() - o2.float()).abs().max().item() <= 2 * TOL[torch.bfloat16]
    else:
        p, o, lse = run_lib(lib, b)
    assert p.check() == 0
    if "prefix_pages" not in b.extra:
        check_coverage(p, b)
        if name == "ragged":
            assert p.info["num_merge_units"] > 0      # some requests are split
    assert torch.isfinite(lse).all() and torch.isfinite(o.float()).all()
    compare_all_rows(b, o, lse, tol_for(b), rel=TOKEN_SCALE_REL if "k_scales" in b.extra else 0.0)
    del b, o, lse
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ randomised sweep

@pytest.mark.parametrize("seed", range(24))
def test_random_batches_against_oracle(lib, cuda, seed):
    """Random shapes, dtypes and length mixes (empty requests, one-token
    requests, partial last pages, requests long enough to be split),
    element by element against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    q_dt, kv_dt = COMBOS[seed % len(COMBOS)]
    D = int(rng.choice([64, 128]))
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 24))
    lengths = rng.integers(1, 2500, size=B)
    lengths[rng.random(B) < 0.15] = 0
    lengths[rng.random(B) < 0.1] = 1
    b = W.make_batch(batch_lengths=lengths.tolist(), num_qo_heads=Hkv * G, num_kv_heads=Hkv,
                     head_dim=D, q_dtype=q_dt, kv_dtype=kv_dt, seed=2000 + seed, device=cuda)
    p, o, lse = run_lib(lib, b)
    check_coverage(p, b)
    assert p.check() == 0
    ref_o, ref_lse = oracle_decode(b)
    compare(o, lse, ref_o, ref_lse, tol_for(b))
