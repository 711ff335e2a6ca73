"""ctypes binding of libfa8.so (include/fa8.h): argument marshalling only.

Every step of the attention runs in the library's CUDA kernels.  This module turns torch
tensors into ``fa8_tensor`` views, allocates outputs and the split-KV workspace with torch
(device memory is the only thing torch provides here), and raises ``Fa8Error`` on any
non-zero status.  There is no fallback: if the library is missing or fails to load, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# FA8_LIBRARY may point at another build of the same library (e.g. one with FA8_TRACE)
LIB_PATH = os.environ.get("FA8_LIBRARY") or os.path.join(_HERE, "_build", "libfa8.so")

FA8_SUCCESS = 0
FA8_ERR_INVALID_ARG = 1
FA8_ERR_UNSUPPORTED = 2
FA8_ERR_WORKSPACE = 3
FA8_ERR_CUDA = 4
FA8_ERR_DEVICE_TIMEOUT = 5
FA8_ERR_DEVICE_BOUNDS = 6

_DTYPES = {
    torch.float8_e4m3fn: 1,
    torch.float8_e5m2: 2,
    torch.bfloat16: 3,
    torch.float16: 4,
    torch.float32: 5,
    torch.int32: 6,
}

# name -> (restype, argtypes); every function declared in include/fa8.h
_T = None  # filled after the struct is defined


class Fa8Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


_P = ctypes.POINTER(Fa8Tensor)
SIGNATURES = {
    "fa8_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, _P, ctypes.c_float, ctypes.c_int, ctypes.c_void_p,
                               ctypes.c_size_t, ctypes.c_void_p]),
    "fa8_fwd_workspace_size": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int,
                                              ctypes.POINTER(ctypes.c_int),
                                              ctypes.POINTER(ctypes.c_size_t)]),
    "fa8_fwd_plan": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_size_t),
                                    ctypes.POINTER(ctypes.c_int64)]),
    "fa8_fwd_static_scratch": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, _P, ctypes.c_float, ctypes.c_int,
                                              ctypes.c_void_p]),
    "fa8_check": (ctypes.c_int, [ctypes.c_void_p]),
    "fa8_set_wait_timeout_ns": (ctypes.c_int, [ctypes.c_uint64]),
    "fa8_set_decode_kernel": (ctypes.c_int, [ctypes.c_int]),
    "fa8_debug_wait_probe": (ctypes.c_int, [ctypes.c_void_p]),
    "fa8_debug_set_trace_buffer": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t]),
    "fa8_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fa8_last_error": (ctypes.c_char_p, []),
    "fa8_version": (ctypes.c_int, []),
}

_lib = None


class Fa8Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"fa8 status {status}: {msg}")
        self.status = status


def lib():
    """Loads libfa8.so (built by ``fp8_attention_forward_gb300.build``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libfa8.so not built ({LIB_PATH}); run fp8_attention_forward_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _view(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() > 4:
        raise ValueError("at most 4 dims")
    v = Fa8Tensor()
    v.data = t.data_ptr()
    v.dtype = _DTYPES[t.dtype]
    v.ndim = t.dim()
    for i in range(t.dim()):
        v.shape[i] = t.shape[i]
        v.stride[i] = t.stride(i)
    return v


def _ref(v):
    return None if v is None else ctypes.byref(v)


def _raise(st: int):
    if st != FA8_SUCCESS:
        raise Fa8Error(st, lib().fa8_last_error().decode())


def _on_device(device):
    """Makes ``device`` current for the library call: the library plans for, and looks up its
    per-device state on, the current CUDA device."""
    import contextlib

    if device.type != "cuda":
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def plan(q, k, v, *, cu_seqlens_q=None, cu_seqlens_k=None, block_table=None, page_size=0,
         num_splits=0, sm_count=None):
    """(splits, workspace_bytes, grid) chosen for these shapes; host-only when sm_count is given."""
    views = [_view(x) for x in (q, k, v, cu_seqlens_q, cu_seqlens_k, block_table)]
    splits = ctypes.c_int(0)
    nbytes = ctypes.c_size_t(0)
    if sm_count is None:
        with _on_device(q.device):
            st = lib().fa8_fwd_workspace_size(*[_ref(x) for x in views], int(page_size), int(num_splits),
                                              ctypes.byref(splits), ctypes.byref(nbytes))
        _raise(st)
        return splits.value, nbytes.value, None
    grid = (ctypes.c_int64 * 2)()
    st = lib().fa8_fwd_plan(*[_ref(x) for x in views], int(page_size), int(num_splits), int(sm_count),
                            ctypes.byref(splits), ctypes.byref(nbytes), grid)
    _raise(st)
    return splits.value, nbytes.value, (grid[0], grid[1])


def fwd(q, k, v, *, descale_q=None, descale_k=None, descale_v=None, out=None, lse=None,
        cu_seqlens_q=None, cu_seqlens_k=None, block_table=None, page_size=0, causal=False,
        window_left=-1, sink=None, softmax_scale=0.0, num_splits=0, workspace=None,
        out_dtype=torch.bfloat16, return_lse=True, stream=None):
    """Fused FP8 attention forward; returns (out, lse).  See include/fa8.h for layouts."""
    dev = q.device
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(tuple(q.shape[:-1]) + (dv,), dtype=out_dtype, device=dev)
    if lse is None and return_lse:
        if q.dim() == 4:
            lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=dev)
        else:
            lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=dev)
    if workspace is None:
        _, nbytes, _ = plan(q, k, v, cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k,
                            block_table=block_table, page_size=page_size, num_splits=num_splits)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev) if nbytes else None
    views = dict(q=_view(q), k=_view(k), v=_view(v), dq=_view(descale_q), dk=_view(descale_k),
                 dv=_view(descale_v), out=_view(out), lse=_view(lse), cq=_view(cu_seqlens_q),
                 ck=_view(cu_seqlens_k), bt=_view(block_table), sink=_view(sink))
    ws_ptr = ctypes.c_void_p(workspace.data_ptr() if workspace is not None else 0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with _on_device(dev):
        st = lib().fa8_fwd(_ref(views["q"]), _ref(views["k"]), _ref(views["v"]), _ref(views["dq"]),
                           _ref(views["dk"]), _ref(views["dv"]), _ref(views["out"]), _ref(views["lse"]),
                           _ref(views["cq"]), _ref(views["ck"]), _ref(views["bt"]), int(page_size),
                           int(bool(causal)), int(window_left), _ref(views["sink"]), float(softmax_scale),
                           int(num_splits), ws_ptr, ws_bytes,
                           _stream_handle(stream, dev) if dev.type == "cuda" else ctypes.c_void_p(0))
    _raise(st)
    return out, lse


STATIC_SCRATCH_BYTES = 32 * 1024 * 1024  # FA8_STATIC_SCRATCH_BYTES in include/fa8.h (a CPU test compares them)


def fwd_static_scratch(q, k, v, *, out, lse=None, descale_q=None, descale_k=None, descale_v=None,
                       cu_seqlens_q=None, cu_seqlens_k=None, block_table=None, page_size=0, causal=False,
                       window_left=-1, sink=None, softmax_scale=0.0, num_splits=0, stream=None):
    """``fa8_fwd_static_scratch``: the forward with split partials in the library's static
    device scratch.  ``out`` (and ``lse`` if wanted) are caller-provided; nothing is allocated."""
    views = dict(q=_view(q), k=_view(k), v=_view(v), dq=_view(descale_q), dk=_view(descale_k),
                 dv=_view(descale_v), out=_view(out), lse=_view(lse), cq=_view(cu_seqlens_q),
                 ck=_view(cu_seqlens_k), bt=_view(block_table), sink=_view(sink))
    with _on_device(q.device):
        st = lib().fa8_fwd_static_scratch(_ref(views["q"]), _ref(views["k"]), _ref(views["v"]),
                                          _ref(views["dq"]), _ref(views["dk"]), _ref(views["dv"]),
                                          _ref(views["out"]), _ref(views["lse"]), _ref(views["cq"]),
                                          _ref(views["ck"]), _ref(views["bt"]), int(page_size), int(bool(causal)),
                                          int(window_left), _ref(views["sink"]), float(softmax_scale),
                                          int(num_splits), _stream_handle(stream, q.device))
    _raise(st)
    return out, lse


def fwd_case(case, **kw):
    """Runs ``fwd`` on an ``inputs.Case`` (tensors already on the GPU)."""
    args = dict(descale_q=case.descale_q, descale_k=case.descale_k, descale_v=case.descale_v,
                cu_seqlens_q=case.cu_seqlens_q, cu_seqlens_k=case.cu_seqlens_k,
                block_table=case.block_table, page_size=case.page_size, causal=case.causal,
                window_left=case.window_left, sink=case.sink, softmax_scale=case.softmax_scale,
                out_dtype=case.out_dtype)
    args.update(kw)
    return fwd(case.q, case.k, case.v, **args)


def check(stream=None) -> int:
    """Synchronises and returns (and clears) the device status word; raises on a CUDA error."""
    dev = torch.device("cuda", torch.cuda.current_device())
    st = lib().fa8_check(_stream_handle(stream, dev))
    if st == FA8_ERR_CUDA:
        _raise(st)
    return st


def set_wait_timeout_ns(ns: int):
    _raise(lib().fa8_set_wait_timeout_ns(int(ns)))


def set_decode_kernel(enable: bool):
    """Routes decode shapes (<= 16 query rows per kv-head) to the decode kernel (default)."""
    _raise(lib().fa8_set_decode_kernel(1 if enable else 0))


def debug_wait_probe(stream=None) -> int:
    dev = torch.device("cuda", torch.cuda.current_device())
    return lib().fa8_debug_wait_probe(_stream_handle(stream, dev))


def version() -> int:
    return lib().fa8_version()
