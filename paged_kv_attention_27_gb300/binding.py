"""ctypes binding of libfi.so: the C ABI of include/fi.h under the same names.

Argument marshalling only. Device buffers may be torch tensors (their
``data_ptr()`` is passed), raw integer addresses or None (NULL); host arrays
for ``fi_plan`` are numpy arrays (converted to contiguous int32). Every
computation happens in the library's CUDA kernels; if the library has not
been built, loading it raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libfi.so")

FI_OK = 0
FI_ERR_INVALID_ARG = 1
FI_ERR_UNSUPPORTED = 2
FI_ERR_WORKSPACE_TOO_SMALL = 3
FI_ERR_CUDA = 4
FI_ERR_DEVICE_TIMEOUT = 5
FI_ERR_DEVICE_BOUNDS = 6
FI_ERR_NO_DEVICE = 7

FI_DTYPE_BF16 = 0
FI_DTYPE_FP16 = 1
FI_DTYPE_E4M3 = 2

FI_LAYOUT_NHD = 0
FI_LAYOUT_HND = 1
FI_MODE_DECODE = 0
FI_MODE_PREFILL = 1

LAYOUTS = {"NHD": FI_LAYOUT_NHD, "HND": FI_LAYOUT_HND}

# every symbol include/fi.h declares
EXPORTED = ["fi_plan", "fi_plan_destroy", "fi_plan_get_info", "fi_plan_get_work",
            "fi_batch_decode_paged", "fi_batch_prefill_paged", "fi_merge_states",
            "fi_check_device_status", "fi_status_string", "fi_last_error_string",
            "fi_debug_set_fault", "fi_profile_next_launch", "fi_batch_decode_paged_noalloc",
            "fi_batch_attention_host", "fi_batch_attention_host_async", "fi_host_step_wait"]


class FiError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {status_string(status)} ({status})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


class PlanOptions(ctypes.Structure):
    """fi_plan_options: window_left (-1 = none), dtype and kv_dtype (FI_DTYPE_*;
    kv_dtype -1 = dtype), and the shared-prefix groups."""
    _fields_ = [("window_left", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("num_prefix_groups", ctypes.c_int32),
                ("prefix_group_indptr", ctypes.c_void_p), ("prefix_pages", ctypes.c_void_p)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("batch_size", ctypes.c_int32),
                ("num_items", ctypes.c_int32), ("num_decode_items", ctypes.c_int32),
                ("num_prefill_items", ctypes.c_int32), ("chunk_tokens", ctypes.c_int32),
                ("num_split_requests", ctypes.c_int32), ("num_partial_slots", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("total_kv_tokens", ctypes.c_int64),
                ("num_prefix_items", ctypes.c_int32), ("num_prefix_groups", ctypes.c_int32),
                ("host_io_bytes", ctypes.c_int64)]


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


def lib():
    """Load libfi.so once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "paged_kv_attention_27_gb300.build.build() first")
    L = ctypes.CDLL(LIB_PATH)
    L.fi_plan.argtypes = [_I32, _I32, _P, _P, _P, _I32, _I32, _I32, _I32, _I32,
                          ctypes.POINTER(PlanOptions), _I32, ctypes.POINTER(_P),
                          ctypes.POINTER(ctypes.c_size_t)]
    L.fi_plan_destroy.argtypes = [_P]
    L.fi_plan_get_info.argtypes = [_P, ctypes.POINTER(PlanInfo)]
    L.fi_plan_get_work.argtypes = [_P, _P, _I32, ctypes.POINTER(_I32)]
    _F = ctypes.c_float
    # ... sm_scale, k_scale, v_scale, k_head_scale, v_head_scale, out, lse, ...
    L.fi_batch_decode_paged.argtypes = [_P, _P, _P, _P, _I32, _I64, _I32, _P, _P, _P,
                                        _F, _F, _F, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.fi_batch_prefill_paged.argtypes = [_P, _P, _P, _P, _P, _I32, _I64, _I32, _P, _P, _P,
                                         _F, _F, _F, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.fi_merge_states.argtypes = [_P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P]
    L.fi_check_device_status.argtypes = [_P, _P]
    L.fi_status_string.argtypes = [_I32]
    L.fi_status_string.restype = ctypes.c_char_p
    L.fi_last_error_string.argtypes = []
    L.fi_last_error_string.restype = ctypes.c_char_p
    L.fi_debug_set_fault.argtypes = [_I32, _I64]
    L.fi_profile_next_launch.argtypes = [_P, _P]
    L.fi_batch_decode_paged_noalloc.argtypes = [_P, _P, _P, _P, _I32, _I64, _I32, _P, _P, _P,
                                                _F, _F, _F, _P, _P, _P, _P, _P]
    L.fi_batch_attention_host.argtypes = [_P, _P, _P, _P, _P, _I32, _I64, _I32, _P, _P, _P,
                                          _F, _F, _F, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.fi_batch_attention_host_async.argtypes = (L.fi_batch_attention_host.argtypes +
                                                [ctypes.POINTER(ctypes.c_uint64)])
    L.fi_host_step_wait.argtypes = [ctypes.c_uint64]
    for name in EXPORTED:
        if name not in ("fi_status_string", "fi_last_error_string"):
            getattr(L, name).restype = _I32
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().fi_status_string(int(status)).decode()


def last_error_string() -> str:
    return lib().fi_last_error_string().decode()


def _check(status: int, where: str):
    if status != FI_OK:
        raise FiError(status, where, last_error_string() if status == FI_ERR_CUDA else "")


def _ptr(x):
    """Device/host address of a tensor, numpy array, int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return stream


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


class Plan:
    """Owns an fi_plan_t handle (destroyed with the object)."""

    def __init__(self, handle: int, workspace_bytes: int):
        self.handle = handle
        self.workspace_bytes = workspace_bytes

    def __del__(self):
        if self.handle and _lib is not None:
            _lib.fi_plan_destroy(self.handle)
            self.handle = None


def fi_plan(mode, batch_size, qo_indptr_h, page_indptr_h, last_page_len_h, num_qo_heads,
            num_kv_heads, head_dim, page_size, causal, options, num_sms) -> Plan:
    """``options``: None (the defaults) or a dict with any of ``window_left``,
    ``dtype``, ``kv_dtype`` and the shared-prefix groups ``prefix_group_indptr``
    / ``prefix_pages`` (host arrays)."""
    qo, pi, lp = _i32(qo_indptr_h), _i32(page_indptr_h), _i32(last_page_len_h)
    opt = None
    keep = []
    if options is not None:
        gi = options.get("prefix_group_indptr")
        pg = options.get("prefix_pages")
        n_groups = 0
        if gi is not None:
            gi, pg = _i32(gi), _i32(pg)
            keep += [gi, pg]
            n_groups = len(gi) - 1
        opt = PlanOptions(int(options.get("window_left", -1)),
                          int(options.get("dtype", FI_DTYPE_BF16)),
                          int(options.get("kv_dtype", -1)), n_groups, _ptr(gi), _ptr(pg))
    h = _P()
    ws = ctypes.c_size_t()
    st = lib().fi_plan(int(mode), int(batch_size), _ptr(qo), _ptr(pi), _ptr(lp), int(num_qo_heads),
                       int(num_kv_heads), int(head_dim), int(page_size), int(bool(causal)),
                       None if opt is None else ctypes.byref(opt), int(num_sms),
                       ctypes.byref(h), ctypes.byref(ws))
    _check(st, "fi_plan")
    return Plan(h.value, ws.value)


def fi_plan_destroy(plan: Plan):
    if plan.handle:
        _check(lib().fi_plan_destroy(plan.handle), "fi_plan_destroy")
        plan.handle = None


def fi_plan_get_info(plan: Plan) -> dict:
    info = PlanInfo()
    _check(lib().fi_plan_get_info(plan.handle, ctypes.byref(info)), "fi_plan_get_info")
    return {k: getattr(info, k) for k, _ in PlanInfo._fields_}


def fi_plan_get_work(plan: Plan) -> np.ndarray:
    n = _I32()
    _check(lib().fi_plan_get_work(plan.handle, None, 0, ctypes.byref(n)), "fi_plan_get_work")
    out = np.zeros((max(n.value, 1), 8), dtype=np.int32)
    _check(lib().fi_plan_get_work(plan.handle, out.ctypes.data, n.value, ctypes.byref(n)),
           "fi_plan_get_work")
    return out[:n.value]


def fi_batch_decode_paged(plan: Plan, q, k_cache, v_cache, kv_layout, page_stride_elems,
                          num_pages, page_indptr_d, page_indices_d, last_page_len_d, sm_scale,
                          k_scale, v_scale, out, lse, workspace, workspace_bytes=None,
                          stream=None, k_head_scale=None, v_head_scale=None):
    """k_head_scale / v_head_scale: device fp32 [num_kv_heads] or None."""
    wsb = plan.workspace_bytes if workspace_bytes is None else workspace_bytes
    st = lib().fi_batch_decode_paged(plan.handle, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                     int(kv_layout), int(page_stride_elems), int(num_pages),
                                     _ptr(page_indptr_d), _ptr(page_indices_d),
                                     _ptr(last_page_len_d), float(sm_scale), float(k_scale),
                                     float(v_scale), _ptr(k_head_scale), _ptr(v_head_scale),
                                     _ptr(out), _ptr(lse), _ptr(workspace), int(wsb),
                                     _stream(stream))
    _check(st, "fi_batch_decode_paged")


def fi_batch_prefill_paged(plan: Plan, q, qo_indptr_d, k_cache, v_cache, kv_layout,
                           page_stride_elems, num_pages, page_indptr_d, page_indices_d,
                           last_page_len_d, sm_scale, k_scale, v_scale, out, lse, workspace,
                           workspace_bytes=None, stream=None, k_head_scale=None,
                           v_head_scale=None):
    wsb = plan.workspace_bytes if workspace_bytes is None else workspace_bytes
    st = lib().fi_batch_prefill_paged(plan.handle, _ptr(q), _ptr(qo_indptr_d), _ptr(k_cache),
                                      _ptr(v_cache), int(kv_layout), int(page_stride_elems),
                                      int(num_pages), _ptr(page_indptr_d), _ptr(page_indices_d),
                                      _ptr(last_page_len_d), float(sm_scale), float(k_scale),
                                      float(v_scale), _ptr(k_head_scale), _ptr(v_head_scale),
                                      _ptr(out), _ptr(lse), _ptr(workspace), int(wsb),
                                      _stream(stream))
    _check(st, "fi_batch_prefill_paged")


def fi_batch_attention_host(plan: Plan, q_h, qo_indptr_h, k_cache, v_cache, kv_layout,
                            page_stride_elems, num_pages, page_indptr_h, page_indices_h,
                            last_page_len_h, sm_scale, k_scale, v_scale, out_h, lse_h, workspace,
                            workspace_bytes, stream=None, k_head_scale=None, v_head_scale=None):
    """q_h / out_h / lse_h: host tensors or arrays (page-locked for
    asynchronous copies); the page-table arguments: host int32 arrays;
    the caches and the workspace (workspace_bytes + host_io_bytes of the
    plan): device memory."""
    st = lib().fi_batch_attention_host(plan.handle, _ptr(q_h), _ptr(qo_indptr_h), _ptr(k_cache),
                                       _ptr(v_cache), int(kv_layout), int(page_stride_elems),
                                       int(num_pages), _ptr(page_indptr_h), _ptr(page_indices_h),
                                       _ptr(last_page_len_h), float(sm_scale), float(k_scale),
                                       float(v_scale), _ptr(k_head_scale), _ptr(v_head_scale),
                                       _ptr(out_h), _ptr(lse_h), _ptr(workspace),
                                       int(workspace_bytes), _stream(stream))
    _check(st, "fi_batch_attention_host")


def fi_batch_attention_host_async(plan: Plan, q_h, qo_indptr_h, k_cache, v_cache, kv_layout,
                                  page_stride_elems, num_pages, page_indptr_h, page_indices_h,
                                  last_page_len_h, sm_scale, k_scale, v_scale, out_h, lse_h,
                                  workspace, workspace_bytes, stream=None, k_head_scale=None,
                                  v_head_scale=None) -> int:
    """fi_batch_attention_host without the wait; returns the step's ticket
    for fi_host_step_wait (q_h, out_h and lse_h belong to the step until
    then)."""
    ticket = ctypes.c_uint64(0)
    st = lib().fi_batch_attention_host_async(
        plan.handle, _ptr(q_h), _ptr(qo_indptr_h), _ptr(k_cache), _ptr(v_cache), int(kv_layout),
        int(page_stride_elems), int(num_pages), _ptr(page_indptr_h), _ptr(page_indices_h),
        _ptr(last_page_len_h), float(sm_scale), float(k_scale), float(v_scale),
        _ptr(k_head_scale), _ptr(v_head_scale), _ptr(out_h), _ptr(lse_h), _ptr(workspace),
        int(workspace_bytes), _stream(stream), ctypes.byref(ticket))
    _check(st, "fi_batch_attention_host_async")
    return ticket.value


def fi_host_step_wait(ticket: int):
    _check(lib().fi_host_step_wait(int(ticket)), "fi_host_step_wait")


def fi_merge_states(v, s, n, S, H, d, out_dtype, out, lse_out, stream=None):
    st = lib().fi_merge_states(_ptr(v), _ptr(s), int(n), int(S), int(H), int(d), int(out_dtype),
                               _ptr(out), _ptr(lse_out), _stream(stream))
    _check(st, "fi_merge_states")


def fi_check_device_status(workspace, stream=None) -> int:
    """Returns the status code (does not raise on device-side errors)."""
    return lib().fi_check_device_status(_ptr(workspace), _stream(stream))


def fi_debug_set_fault(kind: int, wait_limit_ns: int = 0):
    _check(lib().fi_debug_set_fault(int(kind), int(wait_limit_ns)), "fi_debug_set_fault")


def fi_profile_next_launch(start_event, stop_event):
    """torch.cuda.Event objects (or raw cudaEvent_t addresses, or None)."""
    sp = start_event.cuda_event if hasattr(start_event, "cuda_event") else start_event
    ep = stop_event.cuda_event if hasattr(stop_event, "cuda_event") else stop_event
    _check(lib().fi_profile_next_launch(sp, ep), "fi_profile_next_launch")


def fi_batch_decode_paged_noalloc(plan: Plan, q, k_cache, v_cache, kv_layout, page_stride_elems,
                                  num_pages, page_indptr_d, page_indices_d, last_page_len_d,
                                  sm_scale, k_scale, v_scale, out, lse, stream=None,
                                  k_head_scale=None, v_head_scale=None):
    """fi_batch_decode_paged with the library's own static scratch (no workspace)."""
    st = lib().fi_batch_decode_paged_noalloc(plan.handle, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                             int(kv_layout), int(page_stride_elems),
                                             int(num_pages), _ptr(page_indptr_d),
                                             _ptr(page_indices_d), _ptr(last_page_len_d),
                                             float(sm_scale), float(k_scale), float(v_scale),
                                             _ptr(k_head_scale), _ptr(v_head_scale),
                                             _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "fi_batch_decode_paged_noalloc")
