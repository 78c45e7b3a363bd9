"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle for packed varlen attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the
``gqa_attention_cu_gb300`` package and its CUDA library) never imports, calls
or links it, and this package imports nothing from the product.

``pva_oracle.c`` is the definition of the operation written out as a plain
double-precision loop nest (see its header for the passages of the
"onnx-runtime-ep-cuda" pages it follows: packed_varlen_attention.rs, module
doc sections "Packed layout & cumulative offsets", "Schema (v1)", "Causal
alignment", and the five kernel stages).  This module only compiles it with
gcc, marshals numpy arrays, and widens bf16/f16/f32 inputs to float64 (exact).
``attention_padded`` is the padded form of the opset-24 ``nonpad_kv_seqlen``
input (attention.rs), written separately over the padded layout.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(library cross-checks, closed forms, invariants, hand-derived golden values).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pva_oracle.c")
_LIB = os.path.join(_HERE, "libpva_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libpva_oracle.so`` next to its source (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c99", _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB)
    return _lib


def _bind(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    lp = ctypes.POINTER(ctypes.c_int64)
    i, d = ctypes.c_int, ctypes.c_double
    lib.pva_oracle_forward.argtypes = [dp, dp, dp, ip, ip, dp, i, i, i, i, i, d, i, d, i]
    lib.pva_oracle_forward.restype = i
    lib.pva_oracle_rows.argtypes = [dp, dp, dp, ip, ip, lp, ctypes.c_int64, dp,
                                    i, i, i, i, i, d, i, d, i]
    lib.pva_oracle_rows.restype = i
    lib.pva_oracle_forward_window.argtypes = [dp, dp, dp, ip, ip, dp, i, i, i, i, i, d, i, d, i, i]
    lib.pva_oracle_forward_window.restype = i
    lib.pva_oracle_rows_window.argtypes = [dp, dp, dp, ip, ip, lp, ctypes.c_int64, dp,
                                           i, i, i, i, i, d, i, d, i, i]
    lib.pva_oracle_rows_window.restype = i
    lib.pva_oracle_forward_padded.argtypes = [dp, dp, dp, lp, dp, i, i, i, i, i, i, i, d, i, d,
                                              i]
    lib.pva_oracle_forward_padded.restype = i
    lib.pva_oracle_max_threads.argtypes = []
    lib.pva_oracle_max_threads.restype = i
    return lib


class use_library:
    """Context manager that points this module at another compiled copy of
    the oracle (the mutation tests compile deliberately broken copies of
    pva_oracle.c and check that the pins reject them)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        _lib = _bind(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _as_f64(x) -> np.ndarray:
    """Widen a torch tensor or array (f32/f16/bf16/f64) to contiguous float64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _as_i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _head_dims(qd: np.ndarray, vd: np.ndarray, H: int, Hkv: int):
    """head_size and v_head_size from rank-3 [T, heads, dim] or rank-2
    [T, heads*dim] packed tensors."""
    d = qd.shape[2] if qd.ndim == 3 else qd.shape[1] // H
    dv = vd.shape[2] if vd.ndim == 3 else vd.shape[1] // Hkv
    return int(d), int(dv)


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def resolve_scale(scale: float, head_size: int) -> float:
    """The scale the oracle applies: a nonzero scale is used as given; zero
    selects the default 1/sqrt(head_size), computed in float32 as the page
    does (packed_varlen_attention.rs, `execute`, scale fallback), then widened."""
    if scale != 0.0:
        return float(np.float32(scale))
    return float(np.float32(1.0) / np.sqrt(np.float32(head_size)))


def attention_padded(q, k, v, nonpad_kv_seqlen, num_heads: int, kv_num_heads: int,
                     scale: float = 0.0, is_causal: bool = False, softcap: float = 0.0,
                     threads: int = 0) -> np.ndarray:
    """fp64 attention in the padded layout of the opset-24 ``nonpad_kv_seqlen``
    input: q [B, q_seq, H, d], k [B, kv_seq, Hkv, d], v [B, kv_seq, Hkv, dv],
    nonpad int [B].  Returns float64 [B, q_seq, H, dv]."""
    lib = _load()
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    npd = nonpad_kv_seqlen
    if hasattr(npd, "detach"):
        npd = npd.detach().to("cpu").numpy()
    npd = np.ascontiguousarray(np.asarray(npd, dtype=np.int64))
    B, q_seq, H, d = qd.shape
    kv_seq, Hkv, dv = kd.shape[1], kd.shape[2], vd.shape[3]
    if H != int(num_heads) or Hkv != int(kv_num_heads) or npd.shape != (B,):
        raise ValueError("shapes do not match the head counts / batch")
    out = np.zeros((B, q_seq, H, dv), dtype=np.float64)
    rc = lib.pva_oracle_forward_padded(
        _ptr(qd, ctypes.c_double), _ptr(kd, ctypes.c_double), _ptr(vd, ctypes.c_double),
        _ptr(npd, ctypes.c_int64), _ptr(out, ctypes.c_double), B, q_seq, kv_seq, H, Hkv, d, dv,
        resolve_scale(scale, d), int(bool(is_causal)), float(np.float32(softcap)), int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def max_threads() -> int:
    return int(_load().pva_oracle_max_threads())


def attention(q, k, v, cu_seqlens_q, cu_seqlens_kv, num_heads: int, kv_num_heads: int,
              scale: float = 0.0, is_causal: bool = False, softcap: float = 0.0,
              threads: int = 0, local_window: int = 0) -> np.ndarray:
    """fp64 attention over packed sequences.

    q [total_q, H, d], k [total_kv, Hkv, d], v [total_kv, Hkv, dv] (any float
    dtype, torch or numpy); cu_* int32 [B+1].  ``local_window`` > 0 also masks
    keys before (causal limit + 1 - local_window).  Returns float64
    [total_q, H, dv].
    """
    lib = _load()
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    cq, ck = _as_i32(cu_seqlens_q), _as_i32(cu_seqlens_kv)
    B = cq.shape[0] - 1
    H, Hkv = int(num_heads), int(kv_num_heads)
    d, dv = _head_dims(qd, vd, H, Hkv)
    total_q = int(cq[-1])
    out = np.zeros((total_q, H, dv), dtype=np.float64)
    args = (_ptr(qd, ctypes.c_double), _ptr(kd, ctypes.c_double), _ptr(vd, ctypes.c_double),
            _ptr(cq, ctypes.c_int32), _ptr(ck, ctypes.c_int32), _ptr(out, ctypes.c_double),
            B, H, Hkv, d, dv, resolve_scale(scale, d), int(bool(is_causal)),
            float(np.float32(softcap)))
    if local_window:
        rc = lib.pva_oracle_forward_window(*args, int(local_window), int(threads))
    else:
        rc = lib.pva_oracle_forward(*args, int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def attention_rows(q, k, v, cu_seqlens_q, cu_seqlens_kv, rows, num_heads: int,
                   kv_num_heads: int, scale: float = 0.0, is_causal: bool = False,
                   softcap: float = 0.0, threads: int = 0,
                   local_window: int = 0) -> np.ndarray:
    """fp64 attention for selected output rows only (row = token * H + head).
    Returns float64 [len(rows), dv]."""
    lib = _load()
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    cq, ck = _as_i32(cu_seqlens_q), _as_i32(cu_seqlens_kv)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    B = cq.shape[0] - 1
    H, Hkv = int(num_heads), int(kv_num_heads)
    d, dv = _head_dims(qd, vd, H, Hkv)
    out = np.zeros((r.shape[0], dv), dtype=np.float64)
    args = (_ptr(qd, ctypes.c_double), _ptr(kd, ctypes.c_double), _ptr(vd, ctypes.c_double),
            _ptr(cq, ctypes.c_int32), _ptr(ck, ctypes.c_int32), _ptr(r, ctypes.c_int64),
            r.shape[0], _ptr(out, ctypes.c_double), B, H, Hkv, d, dv,
            resolve_scale(scale, d), int(bool(is_causal)), float(np.float32(softcap)))
    if local_window:
        rc = lib.pva_oracle_rows_window(*args, int(local_window), int(threads))
    else:
        rc = lib.pva_oracle_rows(*args, int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out
