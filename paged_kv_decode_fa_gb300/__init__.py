"""Batched decode attention over a paged KV cache, for one GB300 (sm_103a).

Thin Python binding of ``libfadecode.so`` (C ABI in ``include/fa_decode.h``):
argument marshalling only.  Every step of the decode path runs in the
library's CUDA kernels; PyTorch supplies device memory and streams.  If the
library has not been built, the first call into it raises RuntimeError -
there is no fallback implementation.

The calls follow the plan/run split of the page "FlashDecoding + FlashInfer -
the decode-time attention story" (section "The API you actually use"):
``plan`` once per batch shape, ``run`` on the hot path, plus ``merge_states``
for the merge rule of section "FlashDecoding - the split-KV trick".
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

__all__ = [
    "FA_OK", "FaError", "DecodePlan", "plan", "plan_multi_token", "plan_ragged_q", "run",
    "merge_states",
    "CascadePlan", "cascade_plan",
    "workspace_size", "plan_work_host", "plan_work_host_buckets",
    "BatchDecodeWithPagedKVCacheWrapper",
    "LIB_PATH", "EXPORTED_SYMBOLS", "library", "library_stats",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfadecode.so")

# Entry points declared in include/fa_decode.h.
EXPORTED_SYMBOLS = (
    "fa_status_string", "fa_decode_workspace_size", "fa_decode_plan",
    "fa_decode_run", "fa_merge_states", "fa_decode_plan_destroy",
    "fa_decode_plan_get_info", "fa_decode_plan_get_work", "fa_plan_work_host",
    "fa_decode_check", "fa_decode_set_timing_events", "fa_decode_static",
    "fa_decode_run_token_scales", "fa_decode_plan_multi_token",
    "fa_cascade_workspace_size", "fa_cascade_plan", "fa_cascade_run", "fa_cascade_plan_destroy",
    "fa_cascade_check", "fa_decode_run_unified_max", "fa_decode_unified_max_fallbacks",
    "fa_cascade_set_timing_events", "fa_decode_static_check", "fa_library_get_stats",
    "fa_decode_plan_ragged_q", "fa_decode_workspace_size_ragged_q", "fa_cascade_run_scaled",
    "fa_plan_work_host_buckets",
    "fa_decode_run_head_scales", "fa_plan_work_host_heads",
)

FA_OK = 0
SEGMENT_INTS = 8
MERGE_INTS = 4
DTYPE_CODES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2,
               torch.float8_e4m3fn: 3}

class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_L().fa_status_string(status).decode()} ({status})")


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "batch", "num_qo_heads", "num_kv_heads", "head_dim", "page_size",
        "num_ctas", "ctas_per_sm", "num_sms", "num_segments", "num_merge_units",
        "num_partial_slots", "threads_per_cta", "smem_bytes_per_cta", "stages")] + [
        ("total_pages", ctypes.c_int64), ("total_tokens", ctypes.c_int64),
        ("workspace_bytes_used", ctypes.c_size_t), ("plan_upload_bytes", ctypes.c_size_t),
        ("tensor_cores", ctypes.c_int), ("fused_merge", ctypes.c_int), ("q_len", ctypes.c_int),
        ("unified_max", ctypes.c_int), ("num_pool_segments", ctypes.c_int),
        ("pool_pages", ctypes.c_int64), ("ragged_q", ctypes.c_int),
        ("total_q_rows", ctypes.c_int64), ("num_buckets", ctypes.c_int),
        ("bucket_first_cta", ctypes.c_int * 4), ("bucket_q_len", ctypes.c_int * 4)]

    def as_dict(self) -> dict:
        out = {}
        for n, _ in self._fields_:
            v = getattr(self, n)
            out[n] = list(v) if isinstance(v, ctypes.Array) else v
        return out


class LibraryStats(ctypes.Structure):
    _fields_ = [("pinned_host_allocations", ctypes.c_int64), ("pinned_host_bytes", ctypes.c_int64),
                ("staged_uploads", ctypes.c_int64)]


def library_stats() -> dict:
    """The library's own host-side resource counters (fa_library_get_stats)."""
    s = LibraryStats()
    _check(_L().fa_library_get_stats(ctypes.byref(s)), "fa_library_get_stats")
    return {n: int(getattr(s, n)) for n, _ in s._fields_}


def _load() -> ctypes.CDLL:
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                            ctypes.c_float, ctypes.c_size_t)
    lib.fa_status_string.argtypes = [i32]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_decode_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.fa_decode_workspace_size.restype = sz
    lib.fa_decode_plan.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                   P, sz, P, ctypes.POINTER(P)]
    lib.fa_decode_plan.restype = i32
    lib.fa_decode_plan_multi_token.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                               P, sz, P, ctypes.POINTER(P)]
    lib.fa_decode_plan_multi_token.restype = i32
    lib.fa_decode_plan_ragged_q.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                            P, sz, P, ctypes.POINTER(P)]
    lib.fa_decode_plan_ragged_q.restype = i32
    lib.fa_decode_workspace_size_ragged_q.argtypes = [i32, i32, i32, i32]
    lib.fa_decode_workspace_size_ragged_q.restype = sz
    lib.fa_decode_run.argtypes = [P, P, P, i64, f32, f32, f32, P, P, P]
    lib.fa_decode_run.restype = i32
    lib.fa_decode_run_token_scales.argtypes = [P, P, P, i64, f32, P, P, P, P, P]
    lib.fa_decode_run_token_scales.restype = i32
    lib.fa_decode_run_head_scales.argtypes = [P, P, P, i64, f32, P, P, P, P, P]
    lib.fa_decode_run_head_scales.restype = i32
    lib.fa_decode_run_unified_max.argtypes = [P, P, P, i64, f32, f32, f32, f32, P, P, P]
    lib.fa_decode_run_unified_max.restype = i32
    lib.fa_decode_unified_max_fallbacks.argtypes = [P, P, ctypes.POINTER(i32)]
    lib.fa_decode_unified_max_fallbacks.restype = i32
    lib.fa_cascade_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.fa_cascade_workspace_size.restype = sz
    lib.fa_cascade_plan.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, i32, i32, i32, P, sz, P,
                                    ctypes.POINTER(P)]
    lib.fa_cascade_plan.restype = i32
    lib.fa_cascade_run.argtypes = [P, P, P, i64, f32, P, P, P]
    lib.fa_cascade_run.restype = i32
    lib.fa_cascade_run_scaled.argtypes = [P, P, P, i64, f32, f32, f32, P, P, P]
    lib.fa_cascade_run_scaled.restype = i32
    lib.fa_cascade_plan_destroy.argtypes = [P]
    lib.fa_cascade_plan_destroy.restype = i32
    lib.fa_cascade_check.argtypes = [P, P, ctypes.POINTER(i32)]
    lib.fa_cascade_check.restype = i32
    lib.fa_merge_states.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, P]
    lib.fa_merge_states.restype = i32
    lib.fa_decode_plan_destroy.argtypes = [P]
    lib.fa_decode_plan_destroy.restype = i32
    lib.fa_decode_plan_get_info.argtypes = [P, ctypes.POINTER(PlanInfo)]
    lib.fa_decode_plan_get_info.restype = i32
    pp = ctypes.POINTER(ctypes.POINTER(ctypes.c_int32))
    lib.fa_decode_plan_get_work.argtypes = [P, pp, pp, pp]
    lib.fa_decode_plan_get_work.restype = i32
    lib.fa_plan_work_host.argtypes = [P, P, i32, i32, i32, i32, i32, ctypes.c_double, P, P, P,
                                      ctypes.POINTER(i32), ctypes.POINTER(i32),
                                      ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.fa_plan_work_host.restype = i32
    lib.fa_plan_work_host_heads.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P]
    lib.fa_plan_work_host_heads.restype = i32
    lib.fa_plan_work_host_buckets.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, i32,
                                              ctypes.c_int64, P, P, P, P, P, P, P, P, P, P]
    lib.fa_plan_work_host_buckets.restype = i32
    lib.fa_decode_check.argtypes = [P, P, ctypes.POINTER(i32)]
    lib.fa_decode_check.restype = i32
    lib.fa_decode_set_timing_events.argtypes = [P, P, P]
    lib.fa_decode_set_timing_events.restype = i32
    lib.fa_cascade_set_timing_events.argtypes = [P, P, P]
    lib.fa_cascade_set_timing_events.restype = i32
    lib.fa_decode_static.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, P, P, i64,
                                     f32, f32, f32, P, P, P]
    lib.fa_decode_static.restype = i32
    lib.fa_decode_static_check.argtypes = [P, ctypes.POINTER(i32)]
    lib.fa_decode_static_check.restype = i32
    lib.fa_library_get_stats.argtypes = [ctypes.POINTER(LibraryStats)]
    lib.fa_library_get_stats.restype = i32
    return lib


_lib_handle: ctypes.CDLL | None = None


def _L() -> ctypes.CDLL:
    """The loaded library.  Raises if it was never built: there is no fallback."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
        _lib_handle = _load()
    return _lib_handle


def library() -> ctypes.CDLL:
    """Load (once) and return the ctypes handle of libfadecode.so."""
    return _L()


def _check(status: int, what: str) -> None:
    if status != FA_OK:
        raise FaError(status, what)


# torch's current stream of a device as a raw handle, without building a
# Stream object (a few microseconds a call on the plan and run paths)
_current_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream) -> int | None:
    if stream is None:
        if _current_raw_stream is not None:
            return _current_raw_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _host_i32(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        if t.device.type == "cpu" and t.dtype == torch.int32 and t.is_contiguous():
            return t.detach().numpy()  # no copy
        t = t.detach().to("cpu")
        return np.ascontiguousarray(t.numpy(), dtype=np.int32)
    if isinstance(t, np.ndarray) and t.dtype == np.int32 and t.flags.c_contiguous:
        return t
    return np.ascontiguousarray(np.asarray(t), dtype=np.int32)


def _host_i32_ptr(t):
    """(owner, address, length) of a host int32 array: a contiguous CPU int32
    tensor is passed as it is, anything else goes through _host_i32."""
    if (isinstance(t, torch.Tensor) and t.device.type == "cpu" and t.dtype == torch.int32
            and t.dim() == 1 and t.is_contiguous()):
        return t, t.data_ptr(), t.shape[0]
    a = _host_i32(t)
    return a, a.ctypes.data, a.shape[0]


def _reachable(t: torch.Tensor) -> bool:
    """Device memory, or page-locked host memory that the kernels read and
    write directly over the CPU-GPU link (on a GB300 node, NVLink-C2C)."""
    return t.is_cuda or t.is_pinned()


def _cuda_device(t: torch.Tensor) -> torch.device:
    """The device a tensor lives on, or the current CUDA device for host memory."""
    return t.device if t.is_cuda else torch.device("cuda", torch.cuda.current_device())


def _dtype_code(dt) -> int:
    if dt not in DTYPE_CODES:
        raise ValueError(f"unsupported dtype {dt}")
    return DTYPE_CODES[dt]


def workspace_size(batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int) -> int:
    """Bytes of device workspace a plan of this batch may need (current device)."""
    n = _L().fa_decode_workspace_size(batch, num_qo_heads, num_kv_heads, head_dim)
    if n == 0:
        raise ValueError("invalid shape or no CUDA device")
    return int(n)


class DecodePlan:
    """A planned decode batch.  Holds the library's plan handle and keeps the
    tensors it refers to (indices, workspace) alive."""

    def __init__(self, handle, indices, workspace, q_dtype, kv_dtype, shape, q_len=1,
                 total_q_rows=None):
        self._h = handle
        self._indices = indices
        self._workspace = workspace
        self.q_dtype = q_dtype
        self.kv_dtype = kv_dtype
        self.q_len = q_len
        self.total_q_rows = total_q_rows  # ragged plans: rows of q / o
        self.batch, self.num_qo_heads, self.num_kv_heads, self.head_dim, self.page_size = shape

    def _q_shape(self):
        B, Hq, D = self.batch, self.num_qo_heads, self.head_dim
        if self.total_q_rows is not None:
            return (self.total_q_rows, Hq, D)
        return (B, Hq, D) if self.q_len == 1 else (B, self.q_len, Hq, D)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _L().fa_decode_plan_destroy(h)
            self._h = None

    @property
    def info(self) -> dict:
        i = PlanInfo()
        _check(_L().fa_decode_plan_get_info(self._h, ctypes.byref(i)), "fa_decode_plan_get_info")
        return i.as_dict()

    def work(self):
        """(cta_offsets [num_ctas+1], segments [n, 8], merge [m, 4]) as numpy int32."""
        info = self.info
        co = ctypes.POINTER(ctypes.c_int32)()
        sg = ctypes.POINTER(ctypes.c_int32)()
        mg = ctypes.POINTER(ctypes.c_int32)()
        _check(_L().fa_decode_plan_get_work(self._h, ctypes.byref(co), ctypes.byref(sg),
                                            ctypes.byref(mg)), "fa_decode_plan_get_work")
        n_c, n_s, n_m = info["num_ctas"], info["num_segments"], info["num_merge_units"]
        cta = np.ctypeslib.as_array(co, shape=(n_c + 1,)).copy()
        seg = (np.ctypeslib.as_array(sg, shape=(n_s * SEGMENT_INTS,)).reshape(n_s, SEGMENT_INTS).copy()
               if n_s else np.zeros((0, SEGMENT_INTS), np.int32))
        mer = (np.ctypeslib.as_array(mg, shape=(n_m * MERGE_INTS,)).reshape(n_m, MERGE_INTS).copy()
               if n_m else np.zeros((0, MERGE_INTS), np.int32))
        return cta, seg, mer

    def run(self, q: torch.Tensor, paged_kv: torch.Tensor, *, sm_scale: float | None = None,
            k_scale: float = 1.0, v_scale: float = 1.0, out: torch.Tensor | None = None,
            lse: torch.Tensor | None = None, return_lse: bool = True, stream=None):
        """Decode attention; returns (o, lse) (lse None if return_lse is False)."""
        out, lse = self._outputs(q, paged_kv, out, lse, return_lse)
        _check(_L().fa_decode_run(
            self._h, q.data_ptr(), paged_kv.data_ptr(), paged_kv.shape[0],
            0.0 if sm_scale is None else float(sm_scale), float(k_scale), float(v_scale),
            out.data_ptr(), lse.data_ptr() if lse is not None else None,
            _stream_handle(stream)), "fa_decode_run")
        return out, lse

    def run_unified_max(self, q: torch.Tensor, paged_kv: torch.Tensor, max_bound: float, *,
                        sm_scale: float | None = None, k_scale: float = 1.0,
                        v_scale: float = 1.0, out: torch.Tensor | None = None,
                        lse: torch.Tensor | None = None, return_lse: bool = True, stream=None):
        """Decode attention with the softmax referenced to a static bound
        `max_bound` on the logits sm_scale * k_scale * (q . k) instead of a
        running maximum (bf16 plans, groups 2/4/8); returns (o, lse)."""
        out, lse = self._outputs(q, paged_kv, out, lse, return_lse)
        _check(_L().fa_decode_run_unified_max(
            self._h, q.data_ptr(), paged_kv.data_ptr(), paged_kv.shape[0],
            0.0 if sm_scale is None else float(sm_scale), float(k_scale), float(v_scale),
            float(max_bound), out.data_ptr(), lse.data_ptr() if lse is not None else None,
            _stream_handle(stream)), "fa_decode_run_unified_max")
        return out, lse

    def run_head_scales(self, q: torch.Tensor, paged_kv: torch.Tensor, k_scales: torch.Tensor,
                        v_scales: torch.Tensor, *, sm_scale: float | None = None,
                        out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                        return_lse: bool = True, stream=None):
        """Decode over an E4M3 cache with one scale per kv head: k_scales /
        v_scales [num_kv_heads] float32 CUDA tensors; returns (o, lse)."""
        for s in (k_scales, v_scales):
            if (s.dtype != torch.float32 or tuple(s.shape) != (self.num_kv_heads,)
                    or not s.is_contiguous() or not s.is_cuda):
                raise ValueError(f"scales must be contiguous float32 CUDA tensors "
                                 f"[{self.num_kv_heads}]")
        out, lse = self._outputs(q, paged_kv, out, lse, return_lse)
        _check(_L().fa_decode_run_head_scales(
            self._h, q.data_ptr(), paged_kv.data_ptr(), paged_kv.shape[0],
            0.0 if sm_scale is None else float(sm_scale), k_scales.data_ptr(),
            v_scales.data_ptr(), out.data_ptr(), lse.data_ptr() if lse is not None else None,
            _stream_handle(stream)), "fa_decode_run_head_scales")
        return out, lse

    def unified_max_fallbacks(self, stream=None) -> int:
        """Synchronise; return and clear the count of unified-max re-centrings."""
        n = ctypes.c_int(0)
        _check(_L().fa_decode_unified_max_fallbacks(self._h, _stream_handle(stream),
                                                    ctypes.byref(n)),
               "fa_decode_unified_max_fallbacks")
        return int(n.value)

    def _outputs(self, q, paged_kv, out, lse, return_lse):
        """Check q / paged_kv against the plan; allocate missing outputs."""
        D = self.head_dim
        if q.dtype != self.q_dtype or paged_kv.dtype != self.kv_dtype:
            raise TypeError("q / paged_kv dtype differs from the plan")
        if tuple(q.shape) != self._q_shape() or not q.is_contiguous() or not _reachable(q):
            raise ValueError(f"q must be a contiguous CUDA or page-locked tensor "
                             f"{list(self._q_shape())}")
        if (paged_kv.dim() != 5 or paged_kv.shape[1] != 2 or paged_kv.shape[2] != self.page_size
                or paged_kv.shape[3] != self.num_kv_heads or paged_kv.shape[4] != D
                or not paged_kv.is_contiguous() or not paged_kv.is_cuda):
            raise ValueError("paged_kv must be a contiguous CUDA tensor "
                             "[num_pages, 2, page_size, num_kv_heads, head_dim]")
        pinned = not q.is_cuda  # outputs follow q: device, or page-locked host memory
        if out is None:
            out = torch.empty(self._q_shape(), dtype=q.dtype, device=q.device,
                              pin_memory=pinned)
        if return_lse and lse is None:
            lse = torch.empty(self._q_shape()[:-1], dtype=torch.float32, device=q.device,
                              pin_memory=pinned)
        for t in (out, lse):
            if t is not None and (not _reachable(t) or not t.is_contiguous()):
                raise ValueError("out / lse must be contiguous CUDA or page-locked tensors")
        return out, lse

    def run_token_scales(self, q: torch.Tensor, paged_kv: torch.Tensor, k_scales: torch.Tensor,
                         v_scales: torch.Tensor, *, sm_scale: float | None = None,
                         out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                         return_lse: bool = True, stream=None):
        """Decode over an E4M3 cache with per-token, per-kv-head scales
        k_scales / v_scales [num_pages, num_kv_heads, page_size] float32."""
        B, Hq, D = self.batch, self.num_qo_heads, self.head_dim
        if q.dtype != self.q_dtype or paged_kv.dtype != self.kv_dtype:
            raise TypeError("q / paged_kv dtype differs from the plan")
        want = (paged_kv.shape[0], self.num_kv_heads, self.page_size)
        for t in (k_scales, v_scales):
            if (t.dtype != torch.float32 or tuple(t.shape) != want or not t.is_contiguous()
                    or not t.is_cuda):
                raise ValueError(f"scales must be contiguous float32 CUDA tensors {want}")
        if tuple(q.shape) != (B, Hq, D) or not q.is_contiguous():
            raise ValueError(f"q must be a contiguous CUDA tensor [{B}, {Hq}, {D}]")
        if out is None:
            out = torch.empty((B, Hq, D), dtype=q.dtype, device=q.device)
        if return_lse and lse is None:
            lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
        _check(_L().fa_decode_run_token_scales(
            self._h, q.data_ptr(), paged_kv.data_ptr(), paged_kv.shape[0],
            0.0 if sm_scale is None else float(sm_scale), k_scales.data_ptr(),
            v_scales.data_ptr(), out.data_ptr(), lse.data_ptr() if lse is not None else None,
            _stream_handle(stream)), "fa_decode_run_token_scales")
        return out, lse

    def check(self, stream=None) -> int:
        """Synchronise and return the device-check flags (0 = clean)."""
        flags = ctypes.c_int(0)
        st = _L().fa_decode_check(self._h, _stream_handle(stream), ctypes.byref(flags))
        if st not in (FA_OK, -5):
            _check(st, "fa_decode_check")
        return int(flags.value)

    def set_timing_events(self, before, after) -> None:
        """Record torch.cuda.Events around the decode kernel of later runs (both
        launches of a ragged plan in two buckets; None = off).

        torch creates an event lazily at its first record, so record each
        event once from torch before handing it over."""
        _check(_L().fa_decode_set_timing_events(self._h, *_event_handles(before, after)),
               "fa_decode_set_timing_events")


def _event_handles(before, after):
    """CUDA event handles of two recorded torch.cuda.Events (None = off).
    torch creates an event lazily at its first record, so record each event
    once from torch before handing it over."""
    for ev in (before, after):
        if ev is not None and not ev.cuda_event:
            raise ValueError("record the torch.cuda.Event once before passing it")
    return (ctypes.c_void_p(before.cuda_event) if before is not None else None,
            ctypes.c_void_p(after.cuda_event) if after is not None else None)


def plan(indptr, indices: torch.Tensor, last_page_len, num_qo_heads: int, num_kv_heads: int,
         head_dim: int, page_size: int, *, q_data_type=torch.bfloat16,
         kv_data_type=None, workspace: torch.Tensor | None = None, stream=None) -> DecodePlan:
    """Plan a decode batch.  indptr/last_page_len may live on the host or the
    device (they are read on the host); indices must be an int32 CUDA tensor."""
    kv_data_type = q_data_type if kv_data_type is None else kv_data_type
    indptr_h, indptr_p, n_indptr = _host_i32_ptr(indptr)
    last_h, last_p, n_last = _host_i32_ptr(last_page_len)
    B = n_indptr - 1
    if n_last < B:
        raise ValueError("last_page_len shorter than the batch")
    if indices.dtype != torch.int32 or not _reachable(indices) or not indices.is_contiguous():
        raise ValueError("indices must be a contiguous int32 CUDA or page-locked tensor")
    if workspace is None:
        workspace = torch.empty(workspace_size(B, num_qo_heads, num_kv_heads, head_dim),
                                dtype=torch.uint8, device=_cuda_device(indices))
    handle = ctypes.c_void_p()
    _check(_L().fa_decode_plan(
        indptr_p, indices.data_ptr() if indices.numel() else None,
        last_p if B else None, B, num_qo_heads, num_kv_heads, head_dim, page_size,
        _dtype_code(q_data_type), _dtype_code(kv_data_type), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_handle(stream),
        ctypes.byref(handle)), "fa_decode_plan")
    return DecodePlan(handle.value, indices, workspace, q_data_type, kv_data_type,
                      (B, num_qo_heads, num_kv_heads, head_dim, page_size))


def plan_multi_token(indptr, indices: torch.Tensor, last_page_len, q_len: int, num_qo_heads: int,
                     num_kv_heads: int, head_dim: int, page_size: int, *,
                     q_data_type=torch.bfloat16, kv_data_type=None,
                     workspace: torch.Tensor | None = None, stream=None) -> DecodePlan:
    """Plan multi-token decode: q_len query tokens per request (the last q_len
    cache positions), query token i attending to positions <= len - q_len + i.
    run() then takes q [B, q_len, Hq, D] and returns o of that shape and lse
    [B, q_len, Hq]."""
    kv_data_type = q_data_type if kv_data_type is None else kv_data_type
    indptr_h, indptr_p, n_indptr = _host_i32_ptr(indptr)
    last_h, last_p, n_last = _host_i32_ptr(last_page_len)
    B = n_indptr - 1
    if n_last < B:
        raise ValueError("last_page_len shorter than the batch")
    if indices.dtype != torch.int32 or not _reachable(indices) or not indices.is_contiguous():
        raise ValueError("indices must be a contiguous int32 CUDA or page-locked tensor")
    if workspace is None:
        if (num_qo_heads // max(1, num_kv_heads)) * q_len > 8:   # the ragged-q kernels
            n = _L().fa_decode_workspace_size_ragged_q(B, num_qo_heads, num_kv_heads, head_dim)
        else:
            n = workspace_size(B, num_qo_heads * q_len, num_kv_heads, head_dim)
        if n == 0:
            raise ValueError("invalid shape or no CUDA device")
        workspace = torch.empty(int(n), dtype=torch.uint8, device=_cuda_device(indices))
    handle = ctypes.c_void_p()
    _check(_L().fa_decode_plan_multi_token(
        indptr_p, indices.data_ptr() if indices.numel() else None,
        last_p if B else None, B, q_len, num_qo_heads, num_kv_heads, head_dim,
        page_size, _dtype_code(q_data_type), _dtype_code(kv_data_type), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_handle(stream),
        ctypes.byref(handle)), "fa_decode_plan_multi_token")
    return DecodePlan(handle.value, indices, workspace, q_data_type, kv_data_type,
                      (B, num_qo_heads, num_kv_heads, head_dim, page_size), q_len=q_len)


def plan_ragged_q(indptr, indices: torch.Tensor, last_page_len, qo_indptr, num_qo_heads: int,
                  num_kv_heads: int, head_dim: int, page_size: int, *,
                  q_data_type=torch.bfloat16, kv_data_type=None,
                  workspace: torch.Tensor | None = None, stream=None) -> DecodePlan:
    """Plan decode with qo_indptr[i+1] - qo_indptr[i] query tokens for request
    i (the last positions of its cache, causal among themselves).  run() then
    takes q [qo_indptr[-1], Hq, D] and returns o of that shape and lse
    [qo_indptr[-1], Hq]."""
    kv_data_type = q_data_type if kv_data_type is None else kv_data_type
    indptr_h, indptr_p, n_indptr = _host_i32_ptr(indptr)
    last_h, last_p, n_last = _host_i32_ptr(last_page_len)
    qo_h, qo_p, n_qo = _host_i32_ptr(qo_indptr)
    B = n_indptr - 1
    if n_last < B or n_qo != B + 1:
        raise ValueError("last_page_len shorter than the batch, or qo_indptr not batch + 1 long")
    if indices.dtype != torch.int32 or not _reachable(indices) or not indices.is_contiguous():
        raise ValueError("indices must be a contiguous int32 CUDA or page-locked tensor")
    if workspace is None:
        n = _L().fa_decode_workspace_size_ragged_q(B, num_qo_heads, num_kv_heads, head_dim)
        if n == 0:
            raise ValueError("invalid shape or no CUDA device")
        workspace = torch.empty(int(n), dtype=torch.uint8, device=_cuda_device(indices))
    handle = ctypes.c_void_p()
    _check(_L().fa_decode_plan_ragged_q(
        indptr_p, indices.data_ptr() if indices.numel() else None,
        last_p if B else None, qo_p, B, num_qo_heads, num_kv_heads, head_dim,
        page_size, _dtype_code(q_data_type), _dtype_code(kv_data_type), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_handle(stream),
        ctypes.byref(handle)), "fa_decode_plan_ragged_q")
    total_q = int(np.asarray(qo_h)[B]) if B >= 0 else 0
    return DecodePlan(handle.value, indices, workspace, q_data_type, kv_data_type,
                      (B, num_qo_heads, num_kv_heads, head_dim, page_size),
                      total_q_rows=total_q)


def run(p: DecodePlan, q, paged_kv, **kw):
    return p.run(q, paged_kv, **kw)


def merge_states(o_a: torch.Tensor, lse_a: torch.Tensor, o_b: torch.Tensor, lse_b: torch.Tensor,
                 *, out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None,
                 stream=None):
    """Merge two sets of states o [n, H, D] (f32/bf16/f16) with lse [n, H] fp32."""
    if o_a.shape != o_b.shape or lse_a.shape != lse_b.shape or o_a.dtype != o_b.dtype:
        raise ValueError("state shapes / dtypes differ")
    if o_a.dim() != 3 or tuple(lse_a.shape) != tuple(o_a.shape[:2]):
        raise ValueError("o must be [n, H, D] and lse [n, H]")
    for t in (o_a, o_b, lse_a, lse_b):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    if lse_a.dtype != torch.float32 or lse_b.dtype != torch.float32:
        raise TypeError("lse must be float32")
    n, H, D = o_a.shape
    out = torch.empty_like(o_a) if out is None else out
    lse_out = torch.empty_like(lse_a) if lse_out is None else lse_out
    _check(_L().fa_merge_states(o_a.data_ptr(), lse_a.data_ptr(), o_b.data_ptr(),
                                lse_b.data_ptr(), out.data_ptr(), lse_out.data_ptr(), n, H, D,
                                _dtype_code(o_a.dtype), _stream_handle(stream)),
           "fa_merge_states")
    return out, lse_out


def plan_work_host(indptr, last_page_len, num_kv_heads: int, page_size: int, max_ctas: int,
                   min_pages_per_cta: int = 8, pool_fraction: float = 0.0, heads: bool = False):
    """Host-only work-list builder (no GPU).  Returns (cta_offsets, segments [n,8],
    merge [m,4], n_slots); segments cta_offsets[-1]: are the run-time pool.
    heads=True: the head-grouped plan fa_decode_plan makes by default
    (fa_plan_work_host_heads; no pool)."""
    indptr_h, indptr_p, n_indptr = _host_i32_ptr(indptr)
    last_h, last_p, n_last = _host_i32_ptr(last_page_len)
    B = n_indptr - 1
    if n_last < B:
        raise ValueError("last_page_len shorter than the batch")
    cuts = max_ctas * 7 + 1
    cta = np.zeros(max_ctas + 1, np.int32)
    seg = np.zeros(((B * num_kv_heads + cuts) * SEGMENT_INTS,), np.int32)
    mer = np.zeros((cuts * MERGE_INTS,), np.int32)
    n_c, n_s, n_m, n_sl = (ctypes.c_int() for _ in range(4))
    if heads:
        _check(_L().fa_plan_work_host_heads(
            indptr_p, last_p if B else None, B, num_kv_heads, page_size, max_ctas,
            min_pages_per_cta, cta.ctypes.data, seg.ctypes.data, mer.ctypes.data,
            ctypes.byref(n_c), ctypes.byref(n_s), ctypes.byref(n_m), ctypes.byref(n_sl)),
            "fa_plan_work_host_heads")
    else:
        _check(_L().fa_plan_work_host(indptr_p, last_p if B else None, B,
                                      num_kv_heads, page_size, max_ctas, min_pages_per_cta,
                                      float(pool_fraction), cta.ctypes.data, seg.ctypes.data,
                                      mer.ctypes.data, ctypes.byref(n_c), ctypes.byref(n_s),
                                      ctypes.byref(n_m), ctypes.byref(n_sl)), "fa_plan_work_host")
    return (cta[: n_c.value + 1].copy(), seg[: n_s.value * SEGMENT_INTS].reshape(-1, SEGMENT_INTS).copy(),
            mer[: n_m.value * MERGE_INTS].reshape(-1, MERGE_INTS).copy(), n_sl.value)


def plan_work_host_buckets(indptr, last_page_len, qo_indptr, group: int, num_kv_heads: int,
                           page_size: int, widest_tiles: int, max_ctas_by_tiles,
                           one_tile_own: bool = False, min_own_units: int = 0,
                           all_buckets: bool = False):
    """Host-only buckets of a ragged plan (fa_plan_work_host_buckets, no GPU).
    Returns None when the batch stays one launch of the widest kernel, else
    (cta_offsets, segments [n,8], merge [m,4], bucket_tiles, bucket_first_cta,
    slot_columns) for the buckets' concatenated work list."""
    indptr_h, indptr_p, n_indptr = _host_i32_ptr(indptr)
    last_h, last_p, n_last = _host_i32_ptr(last_page_len)
    qo_h, qo_p, n_qo = _host_i32_ptr(qo_indptr)
    B = n_indptr - 1
    if n_last < B or n_qo < B + 1:
        raise ValueError("last_page_len / qo_indptr shorter than the batch")
    mc = np.zeros(4, np.int32)
    mc[:len(max_ctas_by_tiles)] = max_ctas_by_tiles
    total = int(mc.sum())
    cuts = sum(int(m) * 7 + 1 for m in mc)
    cta = np.zeros(total + 1, np.int32)
    seg = np.zeros(((B * num_kv_heads + cuts) * SEGMENT_INTS,), np.int32)
    mer = np.zeros((cuts * MERGE_INTS,), np.int32)
    tiles = np.zeros(4, np.int32)
    first = np.zeros(4, np.int32)
    n_c, n_s, n_m, n_b = (ctypes.c_int() for _ in range(4))
    cols = ctypes.c_int64()
    flags = (1 if one_tile_own else 0) | (2 if all_buckets else 0)
    _check(_L().fa_plan_work_host_buckets(
        indptr_p, last_p if B else None, qo_p, B, group, num_kv_heads, page_size, widest_tiles,
        mc.ctypes.data, flags, int(min_own_units), cta.ctypes.data, seg.ctypes.data,
        mer.ctypes.data, ctypes.byref(n_c), ctypes.byref(n_s), ctypes.byref(n_m),
        ctypes.byref(n_b), tiles.ctypes.data, first.ctypes.data, ctypes.byref(cols)),
        "fa_plan_work_host_buckets")
    if n_b.value == 0:
        return None
    nb = n_b.value
    return (cta[: n_c.value + 1].copy(),
            seg[: n_s.value * SEGMENT_INTS].reshape(-1, SEGMENT_INTS).copy(),
            mer[: n_m.value * MERGE_INTS].reshape(-1, MERGE_INTS).copy(),
            tiles[:nb].copy(), first[:nb].copy(), cols.value)


class CascadePlan:
    """A planned cascade batch: one shared prefix of whole pages, then each
    request's own pages.  Keeps the index tensors and the workspace alive."""

    def __init__(self, handle, keep, q_dtype, shape, kv_dtype=None):
        self._h = handle
        self._keep = keep
        self.q_dtype = q_dtype
        self.kv_dtype = q_dtype if kv_dtype is None else kv_dtype
        self.batch, self.num_qo_heads, self.num_kv_heads, self.head_dim = shape

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _L().fa_cascade_plan_destroy(h)
            self._h = None

    def run(self, q: torch.Tensor, paged_kv: torch.Tensor, *, sm_scale: float | None = None,
            k_scale: float = 1.0, v_scale: float = 1.0, out: torch.Tensor | None = None,
            lse: torch.Tensor | None = None, return_lse: bool = True, stream=None):
        """Cascade decode; k_scale / v_scale are an E4M3 cache's per-tensor
        scales (1 for a 16-bit cache)."""
        B, Hq, D = self.batch, self.num_qo_heads, self.head_dim
        if q.dtype != self.q_dtype or paged_kv.dtype != self.kv_dtype:
            raise TypeError("q / paged_kv dtype differs from the plan")
        if tuple(q.shape) != (B, Hq, D) or not q.is_contiguous() or not paged_kv.is_contiguous():
            raise ValueError(f"q must be a contiguous CUDA tensor [{B}, {Hq}, {D}]")
        if out is None:
            out = torch.empty_like(q)
        if return_lse and lse is None:
            lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
        _check(_L().fa_cascade_run_scaled(
            self._h, q.data_ptr(), paged_kv.data_ptr(), paged_kv.shape[0],
            0.0 if sm_scale is None else float(sm_scale), float(k_scale), float(v_scale),
            out.data_ptr(), lse.data_ptr() if lse is not None else None,
            _stream_handle(stream)), "fa_cascade_run_scaled")
        return out, lse

    def set_timing_events(self, before, after) -> None:
        """Record torch.cuda.Events around the prefix kernel of later runs (None = off)."""
        _check(_L().fa_cascade_set_timing_events(self._h, *_event_handles(before, after)),
               "fa_cascade_set_timing_events")

    def check(self, stream=None) -> int:
        flags = ctypes.c_int(0)
        st = _L().fa_cascade_check(self._h, _stream_handle(stream), ctypes.byref(flags))
        if st not in (FA_OK, -5):
            _check(st, "fa_cascade_check")
        return int(flags.value)


def cascade_plan(prefix_indices: torch.Tensor, indptr, indices: torch.Tensor, last_page_len,
                 num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int, *,
                 q_data_type=torch.bfloat16, kv_data_type=None,
                 workspace: torch.Tensor | None = None, stream=None) -> CascadePlan:
    """Plan cascade decode: prefix_indices are the shared (full) pages every
    request starts with; indptr/indices/last_page_len describe each request's
    own pages after them."""
    indptr_h, indptr_p, n_indptr = _host_i32_ptr(indptr)
    last_h, last_p, n_last = _host_i32_ptr(last_page_len)
    B = n_indptr - 1
    if n_last < B:
        raise ValueError("last_page_len shorter than the batch")
    for t in (prefix_indices, indices):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("index arrays must be contiguous int32 CUDA tensors")
    if workspace is None:
        n = _L().fa_cascade_workspace_size(B, num_qo_heads, num_kv_heads, head_dim)
        if n == 0:
            raise ValueError("invalid shape or no CUDA device")
        workspace = torch.empty(int(n), dtype=torch.uint8, device=prefix_indices.device)
    handle = ctypes.c_void_p()
    kv_data_type = q_data_type if kv_data_type is None else kv_data_type
    _check(_L().fa_cascade_plan(
        prefix_indices.data_ptr(), prefix_indices.numel(), indptr_p,
        indices.data_ptr() if indices.numel() else None, last_p if B else None, B, num_qo_heads,
        num_kv_heads, head_dim, page_size, _dtype_code(q_data_type), _dtype_code(kv_data_type),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream_handle(stream), ctypes.byref(handle)), "fa_cascade_plan")
    return CascadePlan(handle.value, (prefix_indices, indices, workspace), q_data_type,
                       (B, num_qo_heads, num_kv_heads, head_dim), kv_dtype=kv_data_type)


class BatchDecodeWithPagedKVCacheWrapper:
    """plan/run wrapper in the shape the pages show: built once over a caller
    workspace with the "NHD" layout, planned per batch, run on the hot path."""

    def __init__(self, workspace_buffer: torch.Tensor, kv_layout: str = "NHD"):
        if kv_layout != "NHD":
            raise ValueError("only the NHD layout is supported")
        self._workspace = workspace_buffer
        self._plan: DecodePlan | None = None

    def plan(self, indptr, indices, last_page_len, num_qo_heads, num_kv_heads, head_dim,
             page_size, q_data_type=torch.bfloat16, kv_data_type=None, stream=None):
        self._plan = plan(indptr, indices, last_page_len, num_qo_heads, num_kv_heads, head_dim,
                          page_size, q_data_type=q_data_type, kv_data_type=kv_data_type,
                          workspace=self._workspace, stream=stream)
        return self._plan

    def run(self, q, paged_kv_cache, *, sm_scale=None, k_scale=1.0, v_scale=1.0,
            return_lse=False, out=None, lse=None, stream=None):
        if self._plan is None:
            raise RuntimeError("call plan() before run()")
        o, l = self._plan.run(q, paged_kv_cache, sm_scale=sm_scale, k_scale=k_scale,
                              v_scale=v_scale, out=out, lse=lse, return_lse=return_lse,
                              stream=stream)
        return (o, l) if return_lse else o
