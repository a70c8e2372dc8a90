"""fa_decode_static - decoding without allocating device memory.

Some callers cannot allocate: they are handed only input and output
pointers by a framework that owns every device buffer, or they run where a
cudaMalloc (which can synchronise the device) is not allowed.  For them the
library offers one entry point that keeps its work list and partial states
in a fixed array of its own.  These tests call it through the C ABI and
check its output against the regular plan/run path, on two calls in a row
(the second call must not see anything the first one left in the shared
array), and check that a batch too large for the array is refused.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_decode_fa_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2, torch.float16: 2e-2,
       torch.float8_e4m3fn: 3e-2}
CODES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2, torch.float8_e4m3fn: 3}


def static_fn(fa):
    f = fa.library().fa_decode_static
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    f.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, P, P, i64, f32, f32, f32,
                  P, P, P]
    f.restype = i32
    return f


def call_static(fa, b):
    indptr = np.ascontiguousarray(b.indptr.numpy(), dtype=np.int32)
    last = np.ascontiguousarray(b.last_page_len.numpy(), dtype=np.int32)
    o = torch.empty_like(b.q)
    lse = torch.empty((b.batch, b.num_qo_heads), dtype=torch.float32, device=b.q.device)
    rc = static_fn(fa)(indptr.ctypes.data, b.indices.data_ptr(), last.ctypes.data, b.batch,
                       b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size,
                       CODES[b.q.dtype], CODES[b.paged_kv.dtype], b.q.data_ptr(),
                       b.paged_kv.data_ptr(), b.num_pages, 0.0, b.k_scale, b.v_scale,
                       o.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return rc, o, lse


def call_regular(fa, b):
    p = fa.plan(b.indptr, b.indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                b.head_dim, b.page_size, q_data_type=b.q.dtype, kv_data_type=b.paged_kv.dtype)
    o, lse = p.run(b.q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    return o, lse


def test_static_matches_regular_two_calls(lib, cuda):
    batches = [
        W.make_batch(batch_lengths=[9000, 3, 0, 611, 17, 2048], num_qo_heads=32, num_kv_heads=8,
                     head_dim=128, q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=21,
                     device=cuda),
        W.make_batch(batch_lengths=[700, 1, 4000, 64], num_qo_heads=64, num_kv_heads=8,
                     head_dim=128, q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn,
                     seed=22, device=cuda),
    ]
    for b in batches:   # two calls in a row on the same shared array
        ref_o, ref_lse = call_regular(lib, b)
        rc, o, lse = call_static(lib, b)
        torch.cuda.synchronize()
        assert rc == 0, lib.library().fa_status_string(rc)
        tol = TOL[b.paged_kv.dtype] if b.paged_kv.dtype == torch.float8_e4m3fn else TOL[b.q.dtype]
        assert torch.equal(torch.isneginf(lse), torch.isneginf(ref_lse))
        fin = torch.isfinite(ref_lse)
        assert (o.float() - ref_o.float()).abs().max().item() <= tol
        assert (lse[fin] - ref_lse[fin]).abs().max().item() <= tol


def test_static_refuses_batches_beyond_its_array(lib, cuda):
    """A work list larger than FA_STATIC_SCRATCH_BYTES is refused before any
    launch (here 600,000 empty requests: 32 bytes of work list each)."""
    B = 600_000
    indptr = np.zeros(B + 1, np.int32)
    last = np.ones(B, np.int32)
    q = torch.zeros((1, 1, 64), dtype=torch.float32, device=cuda)
    kv = torch.zeros((1, 2, 16, 1, 64), dtype=torch.float32, device=cuda)
    o = torch.zeros_like(q)
    rc = static_fn(lib)(indptr.ctypes.data, None, last.ctypes.data, B, 1, 1, 64, 16, 0, 0,
                        q.data_ptr(), kv.data_ptr(), 1, 0.0, 1.0, 1.0, o.data_ptr(), None,
                        torch.cuda.current_stream().cuda_stream)
    assert rc == -3, lib.library().fa_status_string(rc)
    assert torch.count_nonzero(o) == 0
