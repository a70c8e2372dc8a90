"""fa_decode_static - decoding without allocating anything.

Some callers cannot allocate: they are handed only input and output
pointers by a framework that owns every device buffer, or they run where a
cudaMalloc (which can synchronise the device) or a page-locked host
allocation is not allowed.  For them the library offers one entry point that
keeps its work list and partial states in a fixed array of its own.  These
tests call it through the C ABI and check that

- its o and lse equal the regular plan/run path bit for bit (same kernels,
  same grid, same work list), on calls in a row whose split units differ, so
  a call cannot lean on anything an earlier call left in the shared array;
- repeated calls leave the device's free memory and the library's
  page-locked staging counters unchanged;
- its device-check word is readable (fa_decode_static_check) and flags a
  page id outside the cache;
- a batch too large for the array, or a call during a stream capture, is
  refused before anything is enqueued.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_decode_fa_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CODES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2, torch.float8_e4m3fn: 3}


def call_static(fa, b, o=None, lse=None, indices=None, stream=None):
    indptr = np.ascontiguousarray(b.indptr.numpy(), dtype=np.int32)
    last = np.ascontiguousarray(b.last_page_len.numpy(), dtype=np.int32)
    o = torch.empty_like(b.q) if o is None else o
    lse = (torch.empty((b.batch, b.num_qo_heads), dtype=torch.float32, device=b.q.device)
           if lse is None else lse)
    idx = b.indices if indices is None else indices
    st = torch.cuda.current_stream().cuda_stream if stream is None else stream
    rc = fa.library().fa_decode_static(
        indptr.ctypes.data, idx.data_ptr(), last.ctypes.data, b.batch, b.num_qo_heads,
        b.num_kv_heads, b.head_dim, b.page_size, CODES[b.q.dtype], CODES[b.paged_kv.dtype],
        b.q.data_ptr(), b.paged_kv.data_ptr(), b.num_pages, 0.0, b.k_scale, b.v_scale,
        o.data_ptr(), lse.data_ptr(), st)
    return rc, o, lse


def static_check(fa):
    flags = ctypes.c_int(0)
    rc = fa.library().fa_decode_static_check(torch.cuda.current_stream().cuda_stream,
                                             ctypes.byref(flags))
    assert rc in (0, -5)
    return flags.value


def call_regular(fa, b):
    p = fa.plan(b.indptr, b.indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                b.head_dim, b.page_size, q_data_type=b.q.dtype, kv_data_type=b.paged_kv.dtype)
    o, lse = p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    return p, o, lse


def batches(cuda):
    return [
        # a long request split over many CTAs plus short ones
        W.make_batch(batch_lengths=[60000, 9000, 3, 0, 611, 17, 2048], num_qo_heads=32,
                     num_kv_heads=8, head_dim=128, q_dtype=torch.bfloat16,
                     kv_dtype=torch.bfloat16, seed=21, device=cuda),
        # a smaller batch with other split units, over an E4M3 cache
        W.make_batch(batch_lengths=[700, 1, 4000, 64], num_qo_heads=64, num_kv_heads=8,
                     head_dim=128, q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn,
                     seed=22, device=cuda),
        # fp32 over the CUDA-core consumer, group 1
        W.make_batch(batch_lengths=[33, 5000, 250], num_qo_heads=4, num_kv_heads=4,
                     head_dim=64, q_dtype=torch.float32, kv_dtype=torch.float32, seed=23,
                     device=cuda),
    ]


def test_static_equals_regular_bitwise(lib, cuda):
    bs = batches(cuda)
    refs = [call_regular(lib, b) for b in bs]
    splits = [p.info["num_merge_units"] for p, _, _ in refs]
    assert splits[0] > 0 and splits[0] != splits[1]
    for _ in range(2):          # the batches in a row, twice, on the one shared array
        for b, (p, ref_o, ref_lse) in zip(bs, refs):
            rc, o, lse = call_static(lib, b)
            assert rc == 0, lib.library().fa_status_string(rc)
            torch.cuda.synchronize()
            assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
            assert static_check(lib) == 0


def test_static_allocates_nothing(lib, cuda):
    """After one warm-up call (which loads the kernels and caches the array's
    address), twenty calls leave the device's free memory and the library's
    page-locked staging counters exactly where they were."""
    bs = batches(cuda)
    outs = [(torch.empty_like(b.q),
             torch.empty((b.batch, b.num_qo_heads), dtype=torch.float32, device=cuda))
            for b in bs]
    for b, (o, lse) in zip(bs, outs):
        assert call_static(lib, b, o, lse)[0] == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = lib.library_stats()
    for i in range(20):
        b = bs[i % len(bs)]
        o, lse = outs[i % len(bs)]
        assert call_static(lib, b, o, lse)[0] == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert lib.library_stats() == stats0


def test_static_check_flags_bad_page_id(lib, cuda):
    """A page id outside the cache reads zeros through the copy bounds and
    sets bit 0 of the static path's check word; the next clean call clears it."""
    b = W.make_batch(batch_lengths=[40, 70], num_qo_heads=8, num_kv_heads=2, head_dim=128,
                     q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=24, device=cuda)
    bad = b.indices.clone()
    bad[1] = b.num_pages + 5
    rc, _, _ = call_static(lib, b, indices=bad)
    assert rc == 0
    assert static_check(lib) & 1
    rc, _, _ = call_static(lib, b)
    assert rc == 0 and static_check(lib) == 0


def test_static_refuses_batches_beyond_its_array(lib, cuda):
    """A work list larger than FA_STATIC_SCRATCH_BYTES is refused before any
    launch (here 600,000 empty requests: 32 bytes of work list each)."""
    B = 600_000
    indptr = np.zeros(B + 1, np.int32)
    last = np.ones(B, np.int32)
    q = torch.zeros((1, 1, 64), dtype=torch.float32, device=cuda)
    kv = torch.zeros((1, 2, 16, 1, 64), dtype=torch.float32, device=cuda)
    o = torch.zeros_like(q)
    rc = lib.library().fa_decode_static(indptr.ctypes.data, None, last.ctypes.data, B, 1, 1, 64,
                                        16, 0, 0, q.data_ptr(), kv.data_ptr(), 1, 0.0, 1.0, 1.0,
                                        o.data_ptr(), None,
                                        torch.cuda.current_stream().cuda_stream)
    assert rc == -3, lib.library().fa_status_string(rc)
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0


def test_static_refused_during_capture(lib, cuda):
    """A call on a stream that is being captured returns FA_ERR_UNSUPPORTED
    and enqueues nothing (its upload is a copy from pageable memory)."""
    b = batches(cuda)[1]
    o = torch.zeros_like(b.q)
    lse = torch.zeros((b.batch, b.num_qo_heads), dtype=torch.float32, device=cuda)
    assert call_static(lib, b, o, lse)[0] == 0     # set-up happens outside the capture
    torch.cuda.synchronize()
    o.zero_()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
            rc, _, _ = call_static(lib, b, o, lse, stream=side.cuda_stream)
    assert rc == -2
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0
