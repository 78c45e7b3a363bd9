"""Packed variable-length GQA attention for GB300 (sm_103a).

A thin ctypes binding over ``libpva.so`` (declared in ``include/pva.h``):
the functions below only marshal arguments -- every step of the computation
runs in the library's CUDA kernels.  There is no CPU fallback: if the
compiled library is missing, every call raises.

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import workloads  # noqa: F401  (seeded synthetic inputs)

__all__ = ["pva_forward", "pva_forward_local", "pva_forward_padded", "pva_gqa_kvcache", "pva_get_status", "pva_schedule", "pva_status_string",
           "pva_last_error", "pva_release", "pva_version", "pva_profile", "pva_kernel_times",
           "pva_selftest_wait", "load_library", "build", "PvaError", "DTYPE_CODES", "DEV_FLAGS"]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpva.so")

PVA_OK, PVA_ERR_INVALID_ARG, PVA_ERR_UNSUPPORTED, PVA_ERR_CUDA, PVA_ERR_OOM = 0, -1, -2, -3, -4
DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}
DEV_FLAGS = {"cu_q_start": 0x1, "cu_kv_start": 0x2, "cu_q_order": 0x4, "cu_kv_order": 0x8,
             "too_many": 0x10, "null_tensor": 0x20, "kv_len": 0x40, "kv_cache": 0x80,
             "wait_timeout": 0x100}

_lock = threading.Lock()
_lib = None


class PvaError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"pva error {code}: {message}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile libpva.so in-tree (nvcc, sm_103a)."""
    from ._build import build as _b
    return _b(force=force)


def load_library(path: str | None = None):
    """Load libpva.so and declare its C signatures.  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise PvaError(PVA_ERR_CUDA, f"{p} not found: build it with "
                           "`python -m gqa_attention_cu_gb300._build`")
        lib = ctypes.CDLL(p)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.pva_forward.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, f, i, vp]
        lib.pva_forward.restype = i
        lib.pva_forward_local.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, f, i, i,
                                          vp]
        lib.pva_forward_from_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i,
                                              i, i, f, i, f, i, i, vp]
        lib.pva_forward_from_host.restype = i
        lib.pva_forward_local.restype = i
        lib.pva_forward_padded.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, f, i,
                                           vp]
        lib.pva_forward_padded.restype = i
        lib.pva_gqa_kvcache.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                        i, i, i, i, i, f, f, i, i, vp]
        lib.pva_gqa_kvcache.restype = i
        lib.pva_get_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.pva_get_status.restype = i
        lib.pva_schedule.argtypes = [vp, vp, i, i, i, i, i, i, i,
                                     ctypes.POINTER(ctypes.c_int32), ctypes.c_size_t, vp]
        lib.pva_schedule.restype = i
        lib.pva_status_string.argtypes = [i]
        lib.pva_status_string.restype = ctypes.c_char_p
        lib.pva_last_error.argtypes = []
        lib.pva_last_error.restype = ctypes.c_char_p
        lib.pva_release.argtypes = []
        lib.pva_release.restype = None
        lib.pva_version.argtypes = []
        lib.pva_version.restype = i
        lib.pva_profile.argtypes = [i]
        lib.pva_profile.restype = i
        lib.pva_kernel_times.argtypes = [ctypes.POINTER(ctypes.c_float), i]
        lib.pva_kernel_times.restype = i
        lib.pva_selftest_wait.argtypes = [ctypes.c_uint32, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.pva_selftest_wait.restype = i
        lib.pva_forward_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, f, i,
                                            vp, vp]
        lib.pva_forward_noalloc.restype = i
        if path is None:
            _lib = lib
        return lib


def _check(rc: int):
    if rc != PVA_OK:
        lib = load_library()
        raise PvaError(rc, f"{lib.pva_status_string(rc).decode()}: {lib.pva_last_error().decode()}")


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t) -> int:
    import torch
    codes = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
    if t.dtype not in codes:
        raise PvaError(PVA_ERR_INVALID_ARG, f"dtype {t.dtype} not supported (f32, f16, bf16)")
    return codes[t.dtype]


def pva_forward(q, k, v, cu_seqlens_q, cu_seqlens_kv, out, B: int, num_heads: int,
                kv_num_heads: int, head_size: int, v_head_size: int, scale: float = 0.0,
                is_causal: int = 0, softcap: float = 0.0, dtype: int | None = None,
                stream=None) -> None:
    """Enqueue out = attention(q, k, v) on ``stream`` (torch stream, raw
    cudaStream_t int, or None for the current stream).  Tensors are CUDA
    tensors; their data pointers are passed as they are (contiguous layouts
    as in include/pva.h)."""
    lib = load_library()
    code = _dtype_code(q) if dtype is None else int(dtype)
    rc = lib.pva_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), cu_seqlens_q.data_ptr(),
                         cu_seqlens_kv.data_ptr(), out.data_ptr(), int(B), int(num_heads),
                         int(kv_num_heads), int(head_size), int(v_head_size), float(scale),
                         int(is_causal), float(softcap), code, _stream_ptr(stream))
    _check(rc)


def pva_forward_from_host(q_host, k_host, v_host, cu_seqlens_q_host, cu_seqlens_kv_host,
                          out_host, q_dev, k_dev, v_dev, out_dev, cu_dev, B: int,
                          num_heads: int, kv_num_heads: int, head_size: int, v_head_size: int,
                          scale: float = 0.0, is_causal: int = 0, softcap: float = 0.0,
                          chunks: int = 0, dtype: int | None = None, stream=None) -> None:
    """pva_forward on a batch in host memory (the *_host tensors, pinned for
    overlap; the offsets are host int32 tensors): the call copies it into the
    caller's device buffers (*_dev, cu_dev of >= 4 B + 34 int32) chunk by
    chunk, overlapping the copies with the attention, and copies the output
    back into out_host; ``stream`` completes after the last copy."""
    lib = load_library()
    code = _dtype_code(q_host) if dtype is None else int(dtype)
    rc = lib.pva_forward_from_host(q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(),
                                   cu_seqlens_q_host.data_ptr(), cu_seqlens_kv_host.data_ptr(),
                                   out_host.data_ptr(), q_dev.data_ptr(), k_dev.data_ptr(),
                                   v_dev.data_ptr(), out_dev.data_ptr(), cu_dev.data_ptr(),
                                   int(B), int(num_heads), int(kv_num_heads), int(head_size),
                                   int(v_head_size), float(scale), int(is_causal),
                                   float(softcap), code, int(chunks), _stream_ptr(stream))
    _check(rc)


def pva_forward_local(q, k, v, cu_seqlens_q, cu_seqlens_kv, out, B: int, num_heads: int,
                      kv_num_heads: int, head_size: int, v_head_size: int, scale: float = 0.0,
                      is_causal: int = 0, softcap: float = 0.0, local_window: int = 0,
                      dtype: int | None = None, stream=None) -> None:
    """pva_forward with a local window: with local_window = W > 0 each query
    row also ignores keys before (its causal limit + 1 - W)."""
    lib = load_library()
    code = _dtype_code(q) if dtype is None else int(dtype)
    rc = lib.pva_forward_local(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                               cu_seqlens_q.data_ptr(), cu_seqlens_kv.data_ptr(), out.data_ptr(),
                               int(B), int(num_heads), int(kv_num_heads), int(head_size),
                               int(v_head_size), float(scale), int(is_causal), float(softcap),
                               int(local_window), code, _stream_ptr(stream))
    _check(rc)


def pva_forward_padded(q, k, v, nonpad_kv_seqlen, out, B: int, q_seq: int, kv_seq: int,
                       num_heads: int, kv_num_heads: int, head_size: int, v_head_size: int,
                       scale: float = 0.0, is_causal: int = 0, softcap: float = 0.0,
                       dtype: int | None = None, stream=None) -> None:
    """The padded form: q [B, q_seq, H, d], k/v [B, kv_seq, Hkv, d/dv], out
    [B, q_seq, H, dv]; batch entry b's keys are the first
    ``nonpad_kv_seqlen[b]`` (CUDA int64 [B]) rows of its slot, and the causal
    limit of query row i is i + nonpad_kv_seqlen[b] - q_seq."""
    lib = load_library()
    code = _dtype_code(q) if dtype is None else int(dtype)
    rc = lib.pva_forward_padded(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                nonpad_kv_seqlen.data_ptr(), out.data_ptr(), int(B), int(q_seq),
                                int(kv_seq), int(num_heads), int(kv_num_heads), int(head_size),
                                int(v_head_size), float(scale), int(is_causal), float(softcap),
                                code, _stream_ptr(stream))
    _check(rc)


def _ptr_or_none(t):
    return None if t is None else t.data_ptr()


def pva_gqa_kvcache(q, k_new, v_new, k_cache, v_cache, seqlens_k, out, num_heads: int,
                    kv_num_heads: int, cos_cache=None, sin_cache=None, position_ids=None,
                    rotary_interleaved: bool = False, scale: float = 0.0, softcap: float = 0.0,
                    local_window: int = 0, dtype: int | None = None, stream=None) -> None:
    """One GroupQueryAttention step on a fixed-capacity BNSH cache: q
    [B, q_seq, H, d], k_new/v_new [B, k_seq, Hkv, d] (or None), caches
    [B, Hkv, capacity, d] (appended in place), seqlens_k int32 [B] (= keys
    after the step - 1), optional cos/sin tables [rows, rotary_dim/2] and
    position_ids int64 [B, q_seq]; out [B, q_seq, H, d]."""
    lib = load_library()
    code = _dtype_code(q) if dtype is None else int(dtype)
    B, q_seq, _, d = q.shape
    k_seq = 0 if k_new is None else int(k_new.shape[1])
    capacity = int(k_cache.shape[2])
    rot = rows = 0
    rot_code = 0
    if cos_cache is not None:
        rows, rot = int(cos_cache.shape[0]), 2 * int(cos_cache.shape[1])
        rot_code = _dtype_code(cos_cache)
    rc = lib.pva_gqa_kvcache(q.data_ptr(), _ptr_or_none(k_new), _ptr_or_none(v_new),
                             k_cache.data_ptr(), v_cache.data_ptr(), seqlens_k.data_ptr(),
                             _ptr_or_none(cos_cache), _ptr_or_none(sin_cache),
                             _ptr_or_none(position_ids), out.data_ptr(), int(B), int(q_seq),
                             k_seq, capacity, int(num_heads), int(kv_num_heads), int(d), rot,
                             rows, int(bool(rotary_interleaved)), rot_code, float(scale),
                             float(softcap), int(local_window), code, _stream_ptr(stream))
    _check(rc)


def pva_forward_noalloc(q, k, v, cu_seqlens_q, cu_seqlens_kv, out, B: int, num_heads: int,
                        kv_num_heads: int, head_size: int, v_head_size: int, scale: float = 0.0,
                        is_causal: int = 0, softcap: float = 0.0, dtype: int | None = None,
                        device_status=None, stream=None) -> None:
    """pva_forward for callers that cannot allocate device memory at call
    time: the library uses its fixed 4 MiB per-device scratch array instead of
    a per-stream workspace (see include/pva.h for the limits and the rule that
    overlapping calls race).  ``device_status`` is an optional CUDA uint32
    tensor the call ORs its status bits into."""
    lib = load_library()
    code = _dtype_code(q) if dtype is None else int(dtype)
    st = device_status.data_ptr() if device_status is not None else None
    rc = lib.pva_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                 cu_seqlens_q.data_ptr(), cu_seqlens_kv.data_ptr(),
                                 out.data_ptr(), int(B), int(num_heads), int(kv_num_heads),
                                 int(head_size), int(v_head_size), float(scale), int(is_causal),
                                 float(softcap), code, st, _stream_ptr(stream))
    _check(rc)


def pva_get_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) its latched device bits."""
    lib = load_library()
    flags = ctypes.c_uint32(0)
    _check(lib.pva_get_status(_stream_ptr(stream), ctypes.byref(flags)))
    return int(flags.value)


def pva_schedule(cu_seqlens_q, cu_seqlens_kv, B: int, num_heads: int, kv_num_heads: int,
                 head_size: int, v_head_size: int, is_causal: int, dtype: int, stream=None):
    """Run only the on-device scheduler; returns its int32 words as a list."""
    lib = load_library()
    n = 8 + 4 * int(B) + 2
    buf = (ctypes.c_int32 * n)()
    _check(lib.pva_schedule(cu_seqlens_q.data_ptr(), cu_seqlens_kv.data_ptr(), int(B),
                            int(num_heads), int(kv_num_heads), int(head_size), int(v_head_size),
                            int(is_causal), int(dtype), buf, n, _stream_ptr(stream)))
    return list(buf)


def pva_status_string(code: int) -> str:
    return load_library().pva_status_string(int(code)).decode()


def pva_last_error() -> str:
    return load_library().pva_last_error().decode()


def pva_release() -> None:
    load_library().pva_release()


def pva_version() -> int:
    return int(load_library().pva_version())


def pva_selftest_wait(limit_us: int = 20000, stream=None) -> int:
    """Run the bounded-wait self-test; returns the device bits it latched."""
    lib = load_library()
    flags = ctypes.c_uint32(0)
    _check(lib.pva_selftest_wait(int(limit_us), _stream_ptr(stream), ctypes.byref(flags)))
    return int(flags.value)


def pva_profile(enable: bool) -> None:
    """Bracket each later launch (this thread) with CUDA events (benchmarks)."""
    _check(load_library().pva_profile(int(bool(enable))))


def pva_kernel_times():
    """Device durations (ms) of the last profiled call's launches:
    (scheduler, prefill, decode or -1)."""
    buf = (ctypes.c_float * 3)()
    _check(load_library().pva_kernel_times(buf, 3))
    return tuple(float(x) for x in buf)
