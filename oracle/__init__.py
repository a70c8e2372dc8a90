"""Float64 CPU oracle for paged-KV decode attention (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The CUDA library never loads it
and it shares no code with that library.

The arithmetic lives in ``oracle.c`` (plain float64 loops, compiled with gcc);
this module compiles it on first use, loads it with ctypes and marshals numpy
arrays in and out.  ``expected_coverage`` states, as a plain set, which
(request, kv head, page) triples a decode plan has to cover, and
``expected_token_coverage`` which (request, kv head, token) triples.

Every function here is pinned by ``tests/test_oracle.py`` against closed forms,
brute force and library routines; nothing is marked "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# element-type codes understood by oracle.c
F32, BF16, F16, E4M3 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP) if it is missing or stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", _SRC,
           "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_batch_decode.argtypes = [
        P, i32, P, i32, i64, P, P, P, i32, i32, i32, i32, i32,
        dbl, dbl, dbl, P, P, i32]
    lib.oracle_batch_decode.restype = i32
    lib.oracle_batch_decode_token_scales.argtypes = [
        P, i32, P, i32, i64, P, P, P, i32, i32, i32, i32, i32, dbl, P, P, P, P, i32]
    lib.oracle_batch_decode_token_scales.restype = i32
    lib.oracle_batch_decode_multi.argtypes = [
        P, i32, P, i32, i64, P, P, P, i32, i32, i32, i32, i32, i32, dbl, dbl, dbl, P, P, i32]
    lib.oracle_batch_decode_multi.restype = i32
    lib.oracle_batch_decode_ragged_q.argtypes = [
        P, i32, P, i32, i64, P, P, P, P, i32, i32, i32, i32, i32, dbl, dbl, dbl, P, P, i32]
    lib.oracle_batch_decode_ragged_q.restype = i32
    lib.oracle_merge_states.argtypes = [P, P, P, P, P, P, i64, i32]
    lib.oracle_merge_states.restype = None
    lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_decode_e4m3.restype = dbl
    lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_bf16.restype = dbl
    lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_f16.restype = dbl
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i32
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """ctypes front end of one compiled copy of oracle.c."""

    def __init__(self, so_path: str):
        self.lib = _bind(ctypes.CDLL(so_path))

    def max_threads(self) -> int:
        """Threads the OpenMP runtime uses by default (OMP_NUM_THREADS or cores)."""
        return int(self.lib.oracle_max_threads())

    def batch_decode(self, q, q_dtype, paged_kv, kv_dtype, indptr, indices, last_page_len,
                     num_qo_heads, num_kv_heads, head_dim, page_size,
                     sm_scale=None, k_scale=1.0, v_scale=1.0, num_threads=0):
        """Decode attention for one query token per request, in float64.

        ``q`` is [B, Hq, D] and ``paged_kv`` is [num_pages, 2, page_size, Hkv, D],
        each a C-contiguous numpy array holding the stored bits (float32 for
        F32, uint16 for BF16/F16, uint8 for E4M3) with its element-type code.
        Returns (o [B, Hq, D] float64, lse [B, Hq] float64), lse being the
        natural-log log-sum-exp of the scaled logits.
        """
        q = np.ascontiguousarray(q)
        paged_kv = np.ascontiguousarray(paged_kv)
        indptr = np.ascontiguousarray(indptr, dtype=np.int32)
        indices = np.ascontiguousarray(indices, dtype=np.int32)
        last_page_len = np.ascontiguousarray(last_page_len, dtype=np.int32)
        B = indptr.shape[0] - 1
        if last_page_len.shape[0] < B:
            raise ValueError("last_page_len shorter than the batch")
        if sm_scale is None:
            sm_scale = 1.0 / float(np.sqrt(head_dim))
        per_page = 2 * page_size * num_kv_heads * head_dim
        if paged_kv.size % per_page:
            raise ValueError("paged_kv size is not a whole number of pages")
        num_pages = paged_kv.size // per_page
        if q.size != B * num_qo_heads * head_dim:
            raise ValueError("q has the wrong number of elements")
        o = np.zeros((B, num_qo_heads, head_dim), dtype=np.float64)
        lse = np.zeros((B, num_qo_heads), dtype=np.float64)
        if indices.size == 0:
            indices = np.zeros(1, dtype=np.int32)
        if last_page_len.size == 0:
            last_page_len = np.zeros(1, dtype=np.int32)
        rc = self.lib.oracle_batch_decode(
            _ptr(q), int(q_dtype), _ptr(paged_kv), int(kv_dtype), int(num_pages),
            _ptr(indptr), _ptr(indices), _ptr(last_page_len), int(B),
            int(num_qo_heads), int(num_kv_heads), int(head_dim), int(page_size),
            float(sm_scale), float(k_scale), float(v_scale), _ptr(o), _ptr(lse),
            int(num_threads))
        if rc != 0:
            raise ValueError("oracle_batch_decode rejected its arguments")
        return o, lse

    def batch_decode_token_scales(self, q, q_dtype, paged_kv, kv_dtype, indptr, indices,
                                  last_page_len, num_qo_heads, num_kv_heads, head_dim,
                                  page_size, k_scales, v_scales, sm_scale=None, num_threads=0):
        """Decode attention with per-token, per-kv-head dequantisation scales:
        k_scales / v_scales are float32 [num_pages, num_kv_heads, page_size]
        and multiply the stored K / V elements of that page, head and slot."""
        q = np.ascontiguousarray(q)
        paged_kv = np.ascontiguousarray(paged_kv)
        indptr = np.ascontiguousarray(indptr, dtype=np.int32)
        indices = np.ascontiguousarray(indices, dtype=np.int32)
        last_page_len = np.ascontiguousarray(last_page_len, dtype=np.int32)
        k_scales = np.ascontiguousarray(k_scales, dtype=np.float32)
        v_scales = np.ascontiguousarray(v_scales, dtype=np.float32)
        B = indptr.shape[0] - 1
        if sm_scale is None:
            sm_scale = 1.0 / float(np.sqrt(head_dim))
        per_page = 2 * page_size * num_kv_heads * head_dim
        num_pages = paged_kv.size // per_page
        if paged_kv.size % per_page or q.size != B * num_qo_heads * head_dim:
            raise ValueError("bad q / paged_kv size")
        if k_scales.size != num_pages * num_kv_heads * page_size or k_scales.shape != v_scales.shape:
            raise ValueError("scales must be [num_pages, num_kv_heads, page_size]")
        o = np.zeros((B, num_qo_heads, head_dim), dtype=np.float64)
        lse = np.zeros((B, num_qo_heads), dtype=np.float64)
        if indices.size == 0:
            indices = np.zeros(1, dtype=np.int32)
        if last_page_len.size == 0:
            last_page_len = np.zeros(1, dtype=np.int32)
        rc = self.lib.oracle_batch_decode_token_scales(
            _ptr(q), int(q_dtype), _ptr(paged_kv), int(kv_dtype), int(num_pages),
            _ptr(indptr), _ptr(indices), _ptr(last_page_len), int(B), int(num_qo_heads),
            int(num_kv_heads), int(head_dim), int(page_size), float(sm_scale),
            _ptr(k_scales), _ptr(v_scales), _ptr(o), _ptr(lse), int(num_threads))
        if rc != 0:
            raise ValueError("oracle_batch_decode_token_scales rejected its arguments")
        return o, lse

    def batch_decode_head_scales(self, q, q_dtype, paged_kv, kv_dtype, indptr, indices,
                                 last_page_len, num_qo_heads, num_kv_heads, head_dim, page_size,
                                 k_head_scales, v_head_scales, sm_scale=None, num_threads=0):
        """Decode attention with one dequantisation scale per kv head
        ("FlashInfer vs FlashAttention-3", "Production War Story: The FP8
        Precision Underflow Failure": scales finer than one per tensor):
        k_head_scales / v_head_scales are float32 [num_kv_heads] and multiply
        every stored K / V element of that head.  By definition this is the
        per-token form with every token of kv head h scaled by its head's
        scale, which is how it is computed here."""
        k_head_scales = np.asarray(k_head_scales, dtype=np.float32).reshape(-1)
        v_head_scales = np.asarray(v_head_scales, dtype=np.float32).reshape(-1)
        if k_head_scales.size != num_kv_heads or v_head_scales.size != num_kv_heads:
            raise ValueError("head scales must be [num_kv_heads]")
        per_page = 2 * page_size * num_kv_heads * head_dim
        num_pages = np.asarray(paged_kv).size // per_page
        shape = (num_pages, num_kv_heads, page_size)
        ks = np.broadcast_to(k_head_scales[None, :, None], shape)
        vs = np.broadcast_to(v_head_scales[None, :, None], shape)
        return self.batch_decode_token_scales(q, q_dtype, paged_kv, kv_dtype, indptr, indices,
                                              last_page_len, num_qo_heads, num_kv_heads,
                                              head_dim, page_size, ks, vs, sm_scale=sm_scale,
                                              num_threads=num_threads)

    def batch_decode_multi(self, q, q_dtype, paged_kv, kv_dtype, indptr, indices, last_page_len,
                           q_len, num_qo_heads, num_kv_heads, head_dim, page_size,
                           sm_scale=None, k_scale=1.0, v_scale=1.0, num_threads=0):
        """Multi-token decode: q [B, q_len, Hq, D]; query token i of a request
        attends to its positions 0 .. len - q_len + i.  Returns float64
        o [B, q_len, Hq, D] and lse [B, q_len, Hq]."""
        q = np.ascontiguousarray(q)
        paged_kv = np.ascontiguousarray(paged_kv)
        indptr = np.ascontiguousarray(indptr, dtype=np.int32)
        indices = np.ascontiguousarray(indices, dtype=np.int32)
        last_page_len = np.ascontiguousarray(last_page_len, dtype=np.int32)
        B = indptr.shape[0] - 1
        if sm_scale is None:
            sm_scale = 1.0 / float(np.sqrt(head_dim))
        per_page = 2 * page_size * num_kv_heads * head_dim
        num_pages = paged_kv.size // per_page
        if paged_kv.size % per_page or q.size != B * q_len * num_qo_heads * head_dim:
            raise ValueError("bad q / paged_kv size")
        o = np.zeros((B, q_len, num_qo_heads, head_dim), dtype=np.float64)
        lse = np.zeros((B, q_len, num_qo_heads), dtype=np.float64)
        if indices.size == 0:
            indices = np.zeros(1, dtype=np.int32)
        if last_page_len.size == 0:
            last_page_len = np.zeros(1, dtype=np.int32)
        rc = self.lib.oracle_batch_decode_multi(
            _ptr(q), int(q_dtype), _ptr(paged_kv), int(kv_dtype), int(num_pages), _ptr(indptr),
            _ptr(indices), _ptr(last_page_len), int(B), int(q_len), int(num_qo_heads),
            int(num_kv_heads), int(head_dim), int(page_size), float(sm_scale), float(k_scale),
            float(v_scale), _ptr(o), _ptr(lse), int(num_threads))
        if rc != 0:
            raise ValueError("oracle_batch_decode_multi rejected its arguments")
        return o, lse

    def batch_decode_ragged_q(self, q, q_dtype, paged_kv, kv_dtype, indptr, indices,
                              last_page_len, qo_indptr, num_qo_heads, num_kv_heads, head_dim,
                              page_size, sm_scale=None, k_scale=1.0, v_scale=1.0,
                              num_threads=0):
        """Decode with n_i = qo_indptr[i+1] - qo_indptr[i] query tokens for
        request i, q ragged [total_q, Hq, D]; query token j of request i
        attends to its positions 0 .. len_i - n_i + j.  Returns float64
        o [total_q, Hq, D] and lse [total_q, Hq]."""
        q = np.ascontiguousarray(q)
        paged_kv = np.ascontiguousarray(paged_kv)
        indptr = np.ascontiguousarray(indptr, dtype=np.int32)
        indices = np.ascontiguousarray(indices, dtype=np.int32)
        last_page_len = np.ascontiguousarray(last_page_len, dtype=np.int32)
        qo_indptr = np.ascontiguousarray(qo_indptr, dtype=np.int32)
        B = indptr.shape[0] - 1
        if qo_indptr.shape[0] != B + 1:
            raise ValueError("qo_indptr must have batch + 1 entries")
        if sm_scale is None:
            sm_scale = 1.0 / float(np.sqrt(head_dim))
        total_q = int(qo_indptr[-1])
        per_page = 2 * page_size * num_kv_heads * head_dim
        num_pages = paged_kv.size // per_page
        if paged_kv.size % per_page or q.size != total_q * num_qo_heads * head_dim:
            raise ValueError("bad q / paged_kv size")
        o = np.zeros((total_q, num_qo_heads, head_dim), dtype=np.float64)
        lse = np.zeros((total_q, num_qo_heads), dtype=np.float64)
        if indices.size == 0:
            indices = np.zeros(1, dtype=np.int32)
        if last_page_len.size == 0:
            last_page_len = np.zeros(1, dtype=np.int32)
        if total_q == 0:
            return o, lse
        rc = self.lib.oracle_batch_decode_ragged_q(
            _ptr(q), int(q_dtype), _ptr(paged_kv), int(kv_dtype), int(num_pages), _ptr(indptr),
            _ptr(indices), _ptr(last_page_len), _ptr(qo_indptr), B, num_qo_heads,
            num_kv_heads, head_dim, page_size, float(sm_scale), float(k_scale), float(v_scale),
            _ptr(o), _ptr(lse), int(num_threads))
        if rc != 0:
            raise ValueError("oracle rejected the arguments")
        return o, lse

    def merge_states(self, o_a, lse_a, o_b, lse_b):
        """Merge two arrays of normalised states (o [..., D], lse [...]) in float64."""
        o_a = np.ascontiguousarray(o_a, dtype=np.float64)
        o_b = np.ascontiguousarray(o_b, dtype=np.float64)
        lse_a = np.ascontiguousarray(lse_a, dtype=np.float64)
        lse_b = np.ascontiguousarray(lse_b, dtype=np.float64)
        if o_a.shape != o_b.shape or lse_a.shape != lse_b.shape:
            raise ValueError("shape mismatch")
        D = o_a.shape[-1]
        n = lse_a.size
        if o_a.size != n * D:
            raise ValueError("o and lse disagree on the number of states")
        o = np.empty_like(o_a)
        lse = np.empty_like(lse_a)
        self.lib.oracle_merge_states(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b),
                                     _ptr(o), _ptr(lse), int(n), int(D))
        return o, lse

    def merge_many(self, os_, lses):
        """Fold a list of states with the two-state merge, first to last."""
        o, lse = os_[0], lses[0]
        for o_b, lse_b in zip(os_[1:], lses[1:]):
            o, lse = self.merge_states(o, lse, o_b, lse_b)
        return o, lse

    def decode_e4m3(self, code: int) -> float:
        return float(self.lib.oracle_decode_e4m3(int(code)))

    def decode_bf16(self, bits: int) -> float:
        return float(self.lib.oracle_decode_bf16(int(bits)))

    def decode_f16(self, bits: int) -> float:
        return float(self.lib.oracle_decode_f16(int(bits)))


def compile_variant(source_text: str, so_path: str) -> str:
    """Compile a (possibly edited) copy of oracle.c to so_path; used by tests
    that plant a mistake in the oracle to show that its pins catch it."""
    src_path = so_path + ".c"
    with open(src_path, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", src_path,
                    "-o", so_path, "-lm"], check=True)
    return so_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def max_threads() -> int:
    return _default().max_threads()


def batch_decode(*args, **kw):
    return _default().batch_decode(*args, **kw)


def batch_decode_token_scales(*args, **kw):
    return _default().batch_decode_token_scales(*args, **kw)


def batch_decode_head_scales(*args, **kw):
    return _default().batch_decode_head_scales(*args, **kw)


def batch_decode_multi(*args, **kw):
    return _default().batch_decode_multi(*args, **kw)


def batch_decode_ragged_q(*args, **kw):
    return _default().batch_decode_ragged_q(*args, **kw)


def merge_states(*args, **kw):
    return _default().merge_states(*args, **kw)


def merge_many(*args, **kw):
    return _default().merge_many(*args, **kw)


def decode_e4m3(code: int) -> float:
    return _default().decode_e4m3(code)


def decode_bf16(bits: int) -> float:
    return _default().decode_bf16(bits)


def decode_f16(bits: int) -> float:
    return _default().decode_f16(bits)


def expected_coverage(indptr, num_kv_heads):
    """Every (request, kv head, page position) a decode plan must cover once.

    Request i owns page positions indptr[i] .. indptr[i+1]-1 of the index
    array, and each of its kv heads attends over all of them.  Returned as an
    int64 array of shape [n, 3] sorted by (request, kv head, position).
    """
    indptr = np.asarray(indptr, dtype=np.int64)
    B = indptr.shape[0] - 1
    blocks = []
    for i in range(B):
        sel = np.arange(indptr[i], indptr[i + 1], dtype=np.int64)
        for h in range(num_kv_heads):
            blocks.append(np.stack([np.full_like(sel, i), np.full_like(sel, h), sel], axis=1))
    if not blocks:
        return np.zeros((0, 3), dtype=np.int64)
    return np.concatenate(blocks, axis=0)


def request_lengths(indptr, last_page_len, page_size):
    """Context length of every request: (pages - 1) * page_size + last_page_len,
    0 for a request with no pages (its last_page_len is ignored).

    Follows plan()'s arguments in section "The API you actually use" of the
    page "FlashDecoding + FlashInfer - the decode-time attention story":
    request i owns pages indptr[i] .. indptr[i+1]-1, the last one holding
    last_page_len[i] valid slots."""
    indptr = np.asarray(indptr, dtype=np.int64)
    last = np.asarray(last_page_len, dtype=np.int64)
    pages = np.diff(indptr)
    return np.where(pages > 0, (pages - 1) * int(page_size) + last[:len(pages)], 0)


def expected_token_coverage(indptr, last_page_len, num_kv_heads, page_size):
    """Every (request, kv head, token) a decode plan must cover once: token t
    of request i for t in [0, len_i), for each kv head.  int64 [n, 3] sorted
    by (request, kv head, token)."""
    lens = request_lengths(indptr, last_page_len, page_size)
    blocks = []
    for i, n in enumerate(lens):
        t = np.arange(int(n), dtype=np.int64)
        for h in range(num_kv_heads):
            blocks.append(np.stack([np.full_like(t, i), np.full_like(t, h), t], axis=1))
    if not blocks:
        return np.zeros((0, 3), dtype=np.int64)
    return np.concatenate(blocks, axis=0)


def expected_token_intervals(indptr, last_page_len, num_kv_heads, page_size):
    """The same set as expected_token_coverage, as one half-open token range
    per non-empty (request, kv head): int64 [n, 4] rows (request, kv head,
    0, len), sorted.  For batches whose triples would not fit in memory."""
    lens = request_lengths(indptr, last_page_len, page_size)
    rows = [(i, h, 0, int(n)) for i, n in enumerate(lens) if n > 0
            for h in range(num_kv_heads)]
    return np.array(rows, dtype=np.int64).reshape(-1, 4)
