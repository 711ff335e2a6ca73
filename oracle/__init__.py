"""fp64 CPU oracle for the fused FP8 attention forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this
package.  The product path (the CUDA library and its binding) never calls it, and it
imports nothing from the product package: it reads the case attributes it needs by
name (duck typing) and converts them to plain arrays for the C code in attn_ref.c.

``attention(case)`` returns (O, LSE) in fp64:
  * every row:   O (total_q, Hq, DV), LSE (total_q, Hq)
  * rows=[(token, head), ...]: O (n, DV), LSE (n,)
where ``token`` indexes the packed query tokens (batch-major for batched Q).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS = {}


def lib_path(mutant: int = 0) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_m{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compiles attn_ref.c with gcc (plain C, -O2, no fast-math) and returns the .so path."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
           f"-DORACLE_MUTANT={mutant}", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("D", ctypes.c_int32), ("DV", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("cu_q", ctypes.c_void_p), ("cu_k", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("max_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("sink", ctypes.c_void_p),
        ("softmax_scale", ctypes.c_double),
        ("causal", ctypes.c_int32), ("window_left", ctypes.c_int32),
        ("n_rows", ctypes.c_int64),
        ("rows_tok", ctypes.c_void_p), ("rows_head", ctypes.c_void_p),
    ]


def _load(mutant: int = 0):
    with _LOCK:
        if mutant not in _LIBS:
            lib = ctypes.CDLL(build(mutant))
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [ctypes.POINTER(_Problem), ctypes.c_void_p,
                                             ctypes.c_void_p]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            _LIBS[mutant] = lib
        return _LIBS[mutant]


def e4m3_decode(code: int, mutant: int = 0) -> float:
    return float(_load(mutant).oracle_e4m3_decode(int(code) & 0xFF))


def _np(t):
    """torch tensor (any device) or array -> numpy on host (no torch import needed)."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        t = t.detach()
        if str(t.dtype) == "torch.float8_e4m3fn":
            import torch  # local: only to reinterpret fp8 storage as bytes

            t = t.view(torch.uint8)
        return t.cpu().contiguous().numpy()
    return np.ascontiguousarray(t)


def _descale(d, B, Hkv):
    if d is None:
        return np.ones((B, Hkv), dtype=np.float64)
    a = _np(d).astype(np.float64)
    return np.ascontiguousarray(np.broadcast_to(a, (B, Hkv)))


def problem_arrays(case) -> dict:
    """Plain contiguous arrays describing ``case`` for the C oracle."""
    B, Hq, Hkv, D, DV = case.B, case.Hq, case.Hkv, case.D, case.DV
    q = _np(case.q).astype(np.uint8, copy=False)
    q = np.ascontiguousarray(q.reshape(-1, Hq, D))
    cu_q = np.zeros(B + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(np.asarray(case.seqlens_q, dtype=np.int64))
    cu_k = np.zeros(B + 1, dtype=np.int32)
    cu_k[1:] = np.cumsum(np.asarray(case.seqlens_k, dtype=np.int64))
    k = _np(case.k).astype(np.uint8, copy=False)
    v = _np(case.v).astype(np.uint8, copy=False)
    bt = None
    max_pages = page_size = 0
    if case.kv_layout == "paged":
        bt = np.ascontiguousarray(_np(case.block_table).astype(np.int32))
        max_pages = bt.shape[1]
        page_size = case.page_size
        k = np.ascontiguousarray(k)
        v = np.ascontiguousarray(v)
    else:
        k = np.ascontiguousarray(k.reshape(-1, Hkv, D))
        v = np.ascontiguousarray(v.reshape(-1, Hkv, DV))
    sink = None if case.sink is None else np.ascontiguousarray(_np(case.sink).astype(np.float64))
    return dict(B=B, Hq=Hq, Hkv=Hkv, D=D, DV=DV, q=q, k=k, v=v, cu_q=cu_q, cu_k=cu_k,
                block_table=bt, max_pages=max_pages, page_size=page_size,
                dq=_descale(case.descale_q, B, Hkv), dk=_descale(case.descale_k, B, Hkv),
                dv=_descale(case.descale_v, B, Hkv), sink=sink,
                softmax_scale=float(case.softmax_scale), causal=int(bool(case.causal)),
                window_left=int(case.window_left))


def attention_arrays(a: dict, rows=None, mutant: int = 0):
    """Runs the oracle on the dict produced by ``problem_arrays``."""
    lib = _load(mutant)
    keep = []

    def ptr(x):
        if x is None:
            return None
        keep.append(x)
        return x.ctypes.data

    p = _Problem()
    p.B, p.Hq, p.Hkv, p.D, p.DV = a["B"], a["Hq"], a["Hkv"], a["D"], a["DV"]
    p.q, p.k, p.v = ptr(a["q"]), ptr(a["k"]), ptr(a["v"])
    p.cu_q, p.cu_k = ptr(a["cu_q"]), ptr(a["cu_k"])
    p.block_table = ptr(a["block_table"])
    p.max_pages, p.page_size = a["max_pages"], a["page_size"]
    p.dq, p.dk, p.dv = ptr(a["dq"]), ptr(a["dk"]), ptr(a["dv"])
    p.sink = ptr(a["sink"])
    p.softmax_scale = a["softmax_scale"]
    p.causal, p.window_left = a["causal"], a["window_left"]
    total_q = int(a["cu_q"][-1])
    if rows is None:
        p.n_rows = -1
        o = np.zeros((total_q, a["Hq"], a["DV"]), dtype=np.float64)
        lse = np.zeros((total_q, a["Hq"]), dtype=np.float64)
    else:
        rows = list(rows)
        toks = np.ascontiguousarray(np.array([r[0] for r in rows], dtype=np.int64))
        heads = np.ascontiguousarray(np.array([r[1] for r in rows], dtype=np.int32))
        p.n_rows = len(rows)
        p.rows_tok, p.rows_head = ptr(toks), ptr(heads)
        o = np.zeros((len(rows), a["DV"]), dtype=np.float64)
        lse = np.zeros((len(rows),), dtype=np.float64)
    rc = lib.oracle_attention(ctypes.byref(p), o.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    return o, lse


def attention(case, rows=None, mutant: int = 0):
    """fp64 (O, LSE) for ``case`` (see module docstring for shapes)."""
    return attention_arrays(problem_arrays(case), rows=rows, mutant=mutant)
