"""Python binding of the pkv C ABI (``include/pkv.h``): argument marshalling only.

Every step of the attention call runs in the CUDA library ``_lib/libpkv.so``;
this module only turns PyTorch tensors into pointers, strides and sizes.  If
the library has not been built, importing works but every call raises
``RuntimeError`` -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpkv.so")

PKV_BF16 = 0
PKV_FP8_E4M3 = 1

STATUS_NAMES = {
    0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_WORKSPACE_TOO_SMALL",
    4: "PKV_ERR_CUDA", 5: "PKV_ERR_DEVICE_TIMEOUT", 6: "PKV_ERR_DEVICE_BOUNDS", 7: "PKV_ERR_PLAN_MISMATCH",
}

# every symbol the header declares
EXPORTED = ["pkv_plan", "pkv_plan_upload", "pkv_plan_get_stats", "pkv_plan_get_items", "pkv_attn_varlen_kvcache_fwd", "pkv_kv_append",
            "pkv_get_status", "pkv_plan_destroy", "pkv_last_error", "pkv_version", "pkv_set_profile_events",
            "pkv_attn_varlen_kvcache_fwd_noalloc", "pkv_plan_decode_dynamic", "pkv_get_status_noalloc"]


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_heads_q", ctypes.c_int32), ("num_heads_kv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("cache_capacity", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("cache_dtype", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float)]


class FwdArgs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("q_stride_tok", ctypes.c_int64), ("q_stride_head", ctypes.c_int64),
                ("out", ctypes.c_void_p), ("o_stride_tok", ctypes.c_int64), ("o_stride_head", ctypes.c_int64),
                ("lse", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p), ("max_seqlen_q", ctypes.c_int32),
                ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p), ("knew_stride_tok", ctypes.c_int64),
                ("knew_stride_head", ctypes.c_int64), ("cu_seqlens_knew", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("kc_stride_page", ctypes.c_int64),
                ("kc_stride_tok", ctypes.c_int64), ("kc_stride_head", ctypes.c_int64),
                ("cache_seqlens", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("block_table_stride", ctypes.c_int32), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("page_indptr", ctypes.c_void_p), ("q_scale", ctypes.c_void_p), ("q_rows", ctypes.c_int32)]


class WorkItemInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("seq", "kv_head", "q_row0", "q_index0", "n_q", "q_len", "kv_len",
                                               "kv_begin", "kv_end", "kind", "partial_slot", "cta",
                                               "head0", "num_heads")] + [
        ("cost", ctypes.c_double)]


class PlanStats(ctypes.Structure):
    _fields_ = [("num_items", ctypes.c_int32), ("num_decode_items", ctypes.c_int32),
                ("num_prefill_items", ctypes.c_int32), ("num_split_units", ctypes.c_int32),
                ("num_ctas", ctypes.c_int32), ("total_q", ctypes.c_int32), ("total_new", ctypes.c_int32),
                ("max_items_per_cta", ctypes.c_int32), ("max_cta_cost", ctypes.c_double),
                ("mean_cta_cost", ctypes.c_double), ("upload_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"pkv CUDA library not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.pkv_plan.argtypes = [ctypes.POINTER(Problem), vp, vp, vp, i32, ctypes.POINTER(vp), ctypes.POINTER(sz)]
        L.pkv_plan_decode_dynamic.argtypes = L.pkv_plan.argtypes
        L.pkv_plan_upload.argtypes = [vp, vp, sz, vp]
        L.pkv_plan_get_stats.argtypes = [vp, ctypes.POINTER(PlanStats)]
        L.pkv_plan_get_items.argtypes = [vp, ctypes.POINTER(WorkItemInfo), i32, ctypes.POINTER(i32)]
        L.pkv_attn_varlen_kvcache_fwd.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(FwdArgs), vp, vp, sz, vp]
        L.pkv_kv_append.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(FwdArgs), i32, vp, vp]
        L.pkv_get_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
        L.pkv_set_profile_events.argtypes = [vp, vp]
        L.pkv_attn_varlen_kvcache_fwd_noalloc.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(FwdArgs), vp, vp]
        L.pkv_get_status_noalloc.argtypes = [vp, ctypes.POINTER(i32)]
        L.pkv_plan_destroy.argtypes = [vp]
        L.pkv_plan_destroy.restype = None
        L.pkv_last_error.restype = ctypes.c_char_p
        L.pkv_version.restype = ctypes.c_char_p
        for name in ("pkv_plan", "pkv_plan_upload", "pkv_plan_get_stats", "pkv_plan_get_items", "pkv_attn_varlen_kvcache_fwd",
                     "pkv_kv_append", "pkv_get_status", "pkv_set_profile_events",
                     "pkv_attn_varlen_kvcache_fwd_noalloc", "pkv_get_status_noalloc"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise PkvError(status, lib().pkv_last_error().decode())


def last_error() -> str:
    return lib().pkv_last_error().decode()


def version() -> str:
    return lib().pkv_version().decode()


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_problem(*, batch, num_heads_q, num_heads_kv, head_dim, page_size, cache_capacity, num_pages,
                 cache_dtype, causal, softmax_scale) -> Problem:
    dt = {"bf16": PKV_BF16, "fp8": PKV_FP8_E4M3}.get(cache_dtype, cache_dtype)
    return Problem(batch, num_heads_q, num_heads_kv, head_dim, page_size, cache_capacity, num_pages, dt,
                   int(bool(causal)), softmax_scale)


def make_args(*, q, out, cu_seqlens_q, max_seqlen_q, k_cache, v_cache, cache_seqlens, lse=None, k_new=None,
              v_new=None, cu_seqlens_knew=None, block_table=None, k_scale=None, v_scale=None,
              page_indptr=None, q_scale=None, q_rows=0) -> FwdArgs:
    """Pointers and element strides of torch tensors laid out as in pkv.h."""
    a = FwdArgs()
    if q is not None:
        a.q, a.q_stride_tok, a.q_stride_head = q.data_ptr(), q.stride(0), q.stride(1)
    if out is not None:
        a.out, a.o_stride_tok, a.o_stride_head = out.data_ptr(), out.stride(0), out.stride(1)
    a.lse = _ptr(lse)
    a.cu_seqlens_q = _ptr(cu_seqlens_q)
    a.max_seqlen_q = int(max_seqlen_q)
    if k_new is not None:
        a.k_new, a.v_new = k_new.data_ptr(), _ptr(v_new)
        a.knew_stride_tok, a.knew_stride_head = k_new.stride(0), k_new.stride(1)
        a.cu_seqlens_knew = _ptr(cu_seqlens_knew)
    a.k_cache, a.v_cache = k_cache.data_ptr(), v_cache.data_ptr()
    a.kc_stride_page, a.kc_stride_tok, a.kc_stride_head = k_cache.stride(0), k_cache.stride(1), k_cache.stride(2)
    a.cache_seqlens = _ptr(cache_seqlens)
    if block_table is not None:
        a.block_table = block_table.data_ptr()
        a.block_table_stride = block_table.stride(0) if block_table.dim() > 1 else 0
    a.k_scale, a.v_scale = _ptr(k_scale), _ptr(v_scale)
    a.page_indptr = _ptr(page_indptr)
    a.q_scale = _ptr(q_scale)
    a.q_rows = int(q_rows)
    return a


class Plan:
    """Host work list made by ``pkv_plan`` (owned until ``close``)."""

    def __init__(self, problem: Problem, q_lens, cache_lens, new_lens, num_sms: int, dynamic: bool = False):
        import numpy as np
        self.problem = problem
        self._q = np.ascontiguousarray(q_lens, dtype=np.int32)
        self._c = np.ascontiguousarray(cache_lens, dtype=np.int32)
        self._n = None if new_lens is None else np.ascontiguousarray(new_lens, dtype=np.int32)
        h = ctypes.c_void_p()
        ws = ctypes.c_size_t()
        fn = lib().pkv_plan_decode_dynamic if dynamic else lib().pkv_plan
        _check(fn(ctypes.byref(problem), self._q.ctypes.data, self._c.ctypes.data,
                  None if self._n is None else self._n.ctypes.data, int(num_sms), ctypes.byref(h), ctypes.byref(ws)))
        self.handle = h
        self.workspace_bytes = int(ws.value)

    def stats(self) -> dict:
        s = PlanStats()
        _check(lib().pkv_plan_get_stats(self.handle, ctypes.byref(s)))
        return {k: getattr(s, k) for k, _ in PlanStats._fields_}

    def items(self) -> list[dict]:
        n = ctypes.c_int32()
        _check(lib().pkv_plan_get_items(self.handle, None, 0, ctypes.byref(n)))
        arr = (WorkItemInfo * max(1, n.value))()
        _check(lib().pkv_plan_get_items(self.handle, arr, n.value, ctypes.byref(n)))
        return [{k: getattr(arr[i], k) for k, _ in WorkItemInfo._fields_} for i in range(n.value)]

    def upload(self, workspace, stream=None) -> None:
        _check(lib().pkv_plan_upload(self.handle, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                     _stream_handle(stream)))

    def close(self) -> None:
        if self.handle:
            lib().pkv_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def plan(problem: Problem, q_lens, cache_lens, new_lens=None, num_sms: Optional[int] = None) -> Plan:
    if num_sms is None:
        import torch
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return Plan(problem, q_lens, cache_lens, new_lens, num_sms)


def plan_decode_dynamic(problem: Problem, q_lens, max_cache_lens, new_lens=None,
                        num_sms: Optional[int] = None) -> Plan:
    """A decode plan whose cache lengths are read on the device at every call
    (bounded by max_cache_lens), for a call captured once in a CUDA graph."""
    if num_sms is None:
        import torch
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return Plan(problem, q_lens, max_cache_lens, new_lens, num_sms, dynamic=True)


def attn_varlen_kvcache_fwd(problem: Problem, args: FwdArgs, plan_: Plan, workspace, stream=None) -> None:
    _check(lib().pkv_attn_varlen_kvcache_fwd(ctypes.byref(problem), ctypes.byref(args), plan_.handle,
                                             workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                             _stream_handle(stream)))


def attn_varlen_kvcache_fwd_noalloc(problem: Problem, args: FwdArgs, plan_: Plan, stream=None) -> None:
    """The attention call without a caller workspace (for callers that cannot
    allocate device memory); uses the library's fixed 32 MiB device scratch."""
    _check(lib().pkv_attn_varlen_kvcache_fwd_noalloc(ctypes.byref(problem), ctypes.byref(args), plan_.handle,
                                                     _stream_handle(stream)))


def get_status_noalloc(stream=None) -> int:
    """Device status word left by the last no-workspace call on this device (then reset)."""
    st = ctypes.c_int32()
    _check(lib().pkv_get_status_noalloc(_stream_handle(stream), ctypes.byref(st)))
    return int(st.value)


def kv_append(problem: Problem, args: FwdArgs, total_new: int, device_status=None, stream=None) -> None:
    _check(lib().pkv_kv_append(ctypes.byref(problem), ctypes.byref(args), int(total_new), _ptr(device_status),
                               _stream_handle(stream)))


def get_status(workspace, stream=None) -> int:
    st = ctypes.c_int32()
    _check(lib().pkv_get_status(workspace.data_ptr(), _stream_handle(stream), ctypes.byref(st)))
    return int(st.value)


def set_profile_events(start=None, stop=None) -> None:
    """Record torch.cuda.Event objects around the attention kernel of later calls.

    torch creates the CUDA event lazily, on its first record(); record both once
    here so that the handles passed to the library exist."""
    if start is not None:
        start.record()
        stop.record()
        assert start.cuda_event and stop.cuda_event
    _check(lib().pkv_set_profile_events(None if start is None else start.cuda_event,
                                        None if stop is None else stop.cuda_event))


def workspace_tensor(nbytes: int, device="cuda"):
    """A caller-owned, 256-byte aligned device workspace of at least nbytes."""
    import torch
    return torch.zeros(max(256, (nbytes + 255) // 256 * 256), dtype=torch.uint8, device=device)
