"""Seeded synthetic workloads for packed variable-length attention.

This module only draws sequence lengths and random Q/K/V values.  It holds
none of the attention arithmetic, so both the CUDA path and the CPU oracle
can be fed from it.

Recipe (one ``torch.Generator('cpu')`` per workload, seeded; draws happen in
this order): the sequence lengths, then Q, then K, then V, each as float32
``randn`` multiplied by ``sigma`` and rounded to the workload dtype
(round-to-nearest-even).  ``N(0, 2)`` means variance 2 (sigma = sqrt(2)).

Named workloads (sizes of the packed batches the benchmark and the parity
tests use):

* ``fp32_small``   : L_q = L_kv = {17, 64, 1, 130}, H = Hkv = 4, d = dv = 64,
                     scale 1/8, non-causal, fp32, N(0, 1).
* ``bf16_prefill`` : B = 16, L_q = L_kv ~ U{128..2048}, H = 32, Hkv = 8,
                     d = dv = 128, default scale, causal, N(0, 1).
* ``bf16_chunked`` : B = 32, L_q ~ U{1..512}, past ~ U{0..4096},
                     L_kv = L_q + past, H = 32, Hkv = 8, d = 128, causal.
* ``bf16_decode``  : B = 256, L_q = 1, L_kv ~ U{512..8192}, H = 32, Hkv = 8,
                     d = 128, causal (a no-op for one query row).
* ``bf16_longctx`` : B = 4, L_q = L_kv = round(exp(U(ln 8192, ln 32768))),
                     H = 8, Hkv = 1, d = dv = 256, causal, softcap 50,
                     N(0, 2).
* ``bf16_mla``     : B = 8, L_q = L_kv ~ U{512..4096}, H = Hkv = 32,
                     d = 192, dv = 128 (q.k wider than v), causal, N(0, 1).
* ``bf16_decode_g16``: the decode batch with H = 32, Hkv = 2 (16 query heads
                     per kv head).
* ``bf16_decode_mla``: the decode batch with d = 192, dv = 128, H = 32, Hkv = 8.
* ``bf16_window``  : B = 4, L_q = L_kv = round(exp(U(ln 8192, ln 32768))),
                     H = 32, Hkv = 8, d = dv = 128, causal, local window 4096,
                     N(0, 1).

``shrink`` divides the length ranges (``B=`` overrides the batch size) to make a same-shaped
small case that the CPU oracle finishes quickly.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}


@dataclass
class Workload:
    name: str
    B: int
    num_heads: int
    kv_num_heads: int
    head_size: int
    v_head_size: int
    dtype: str
    is_causal: bool
    scale: float          # 0.0 selects the default 1/sqrt(head_size)
    softcap: float
    sigma: float
    lengths: str          # length recipe key
    fixed_lq: tuple = ()
    fixed_lkv: tuple = ()
    params: dict = field(default_factory=dict)
    window: int = 0       # local window (pva_forward_local); 0 = none


WORKLOADS = {
    "fp32_small": Workload("fp32_small", 4, 4, 4, 64, 64, "f32", False, 0.125, 0.0, 1.0,
                           "fixed", (17, 64, 1, 130), (17, 64, 1, 130)),
    "bf16_prefill": Workload("bf16_prefill", 16, 32, 8, 128, 128, "bf16", True, 0.0, 0.0, 1.0,
                             "uniform_self", params={"lo": 128, "hi": 2048}),
    "bf16_chunked": Workload("bf16_chunked", 32, 32, 8, 128, 128, "bf16", True, 0.0, 0.0, 1.0,
                             "chunked", params={"q_lo": 1, "q_hi": 512, "past_lo": 0,
                                                "past_hi": 4096}),
    "bf16_decode": Workload("bf16_decode", 256, 32, 8, 128, 128, "bf16", True, 0.0, 0.0, 1.0,
                            "decode", params={"lo": 512, "hi": 8192}),
    "bf16_longctx": Workload("bf16_longctx", 4, 8, 1, 256, 256, "bf16", True, 0.0, 50.0,
                             math.sqrt(2.0), "loguniform_self", params={"lo": 8192, "hi": 32768}),
    "bf16_mla": Workload("bf16_mla", 8, 32, 32, 192, 128, "bf16", True, 0.0, 0.0, 1.0,
                         "uniform_self", params={"lo": 512, "hi": 4096}),
    # the decode batch with 16 query heads per kv head, and with MLA-style
    # head sizes (q.k over 192 dims, v 128)
    "bf16_decode_g16": Workload("bf16_decode_g16", 256, 32, 2, 128, 128, "bf16", True, 0.0, 0.0,
                                1.0, "decode", params={"lo": 512, "hi": 8192}),
    "bf16_decode_mla": Workload("bf16_decode_mla", 256, 32, 8, 192, 128, "bf16", True, 0.0, 0.0,
                                1.0, "decode", params={"lo": 512, "hi": 8192}),
    "bf16_window": Workload("bf16_window", 4, 32, 8, 128, 128, "bf16", True, 0.0, 0.0, 1.0,
                            "loguniform_self", params={"lo": 8192, "hi": 32768}, window=4096),
    # one decode step against a fixed-capacity BNSH KV cache (pva_gqa_kvcache):
    # totals after the append ~ U[lo, hi], rotary embedding on all 128 dims
    "bf16_kvcache_decode": Workload("bf16_kvcache_decode", 256, 32, 8, 128, 128, "bf16", True,
                                    0.0, 0.0, 1.0, "decode",
                                    params={"lo": 512, "hi": 8192, "capacity": 8192,
                                            "rotary_dim": 128, "cache_rows": 8192}),
}


def draw_lengths(w: Workload, gen: torch.Generator, shrink: int = 1):
    """Per-sequence (L_q, L_kv) lists for workload ``w``."""
    B = w.B
    p = w.params
    if w.lengths == "fixed":
        return list(w.fixed_lq), list(w.fixed_lkv)
    if w.lengths == "uniform_self":
        lo, hi = max(1, p["lo"] // shrink), max(1, p["hi"] // shrink)
        L = torch.randint(lo, hi + 1, (B,), generator=gen).tolist()
        return L, list(L)
    if w.lengths == "chunked":
        lq = torch.randint(max(1, p["q_lo"]), max(1, p["q_hi"] // shrink) + 1, (B,), generator=gen)
        past = torch.randint(p["past_lo"], p["past_hi"] // shrink + 1, (B,), generator=gen)
        return lq.tolist(), (lq + past).tolist()
    if w.lengths == "decode":
        lkv = torch.randint(max(1, p["lo"] // shrink), max(1, p["hi"] // shrink) + 1, (B,),
                            generator=gen)
        return [1] * B, lkv.tolist()
    if w.lengths == "loguniform_self":
        lo, hi = p["lo"] / shrink, p["hi"] / shrink
        u = torch.rand((B,), generator=gen, dtype=torch.float64)
        L = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
        L = torch.clamp(torch.round(L), lo, hi).to(torch.int64).tolist()
        return L, list(L)
    raise ValueError(w.lengths)


def cu_from_lengths(lengths) -> torch.Tensor:
    """int32 [B+1] exclusive prefix sum of the lengths (the packed ABI)."""
    out = [0]
    for L in lengths:
        out.append(out[-1] + int(L))
    return torch.tensor(out, dtype=torch.int32)


def make_packed(lq, lkv, H, Hkv, d, dv, dtype: str, sigma: float = 1.0, seed: int = 0,
                gen: torch.Generator | None = None, device: str = "cpu"):
    """Random packed Q/K/V (tensors of ``dtype`` on ``device``) for given
    lengths.  Values come from ``gen`` (or a generator on ``device`` seeded
    with ``seed``); generation on a CUDA device uses that device's generator,
    so its values differ from the CPU recipe but are just as reproducible."""
    if gen is None:
        gen = torch.Generator(device)
        gen.manual_seed(seed)
    dev = gen.device
    tq, tkv = int(sum(lq)), int(sum(lkv))
    td = DTYPES[dtype]
    q = (torch.randn((tq, H, d), generator=gen, device=dev) * sigma).to(td)
    k = (torch.randn((tkv, Hkv, d), generator=gen, device=dev) * sigma).to(td)
    v = (torch.randn((tkv, Hkv, dv), generator=gen, device=dev) * sigma).to(td)
    return q, k, v, cu_from_lengths(lq).to(dev), cu_from_lengths(lkv).to(dev)


def make(name: str, seed: int = 0, shrink: int = 1, B: int | None = None,
         device: str = "cpu"):
    """Inputs for a named workload: dict with q, k, v, cu_q, cu_kv and the
    attention parameters.  Lengths always come from a CPU generator seeded
    with ``seed``; on ``device='cpu'`` the values continue that generator's
    stream, on a CUDA device they come from a generator on that device seeded
    with ``seed + 1`` (used for the full-size workloads)."""
    w = WORKLOADS[name]
    if B is not None:
        w = Workload(**{**w.__dict__, "B": B})
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    lq, lkv = draw_lengths(w, gen, shrink)
    if device != "cpu":
        gen = torch.Generator(device)
        gen.manual_seed(seed + 1)
    q, k, v, cu_q, cu_kv = make_packed(lq, lkv, w.num_heads, w.kv_num_heads, w.head_size,
                                       w.v_head_size, w.dtype, w.sigma, gen=gen)
    return {
        "name": name, "q": q, "k": k, "v": v, "cu_q": cu_q, "cu_kv": cu_kv,
        "lq": lq, "lkv": lkv, "B": len(lq),
        "num_heads": w.num_heads, "kv_num_heads": w.kv_num_heads,
        "head_size": w.head_size, "v_head_size": w.v_head_size,
        "dtype": w.dtype, "is_causal": w.is_causal, "scale": w.scale,
        "softcap": w.softcap, "sigma": w.sigma, "window": w.window,
    }


def rotary_tables(rows: int, rotary_dim: int, base: float = 10000.0, dtype=torch.float32):
    """cos/sin tables [rows, rotary_dim/2]: angle p * base^(-k / (rotary_dim/2))."""
    half = rotary_dim // 2
    theta = base ** (-torch.arange(half, dtype=torch.float64) / half)
    ang = torch.arange(rows, dtype=torch.float64)[:, None] * theta[None, :]
    return torch.cos(ang).to(dtype), torch.sin(ang).to(dtype)


def make_cache_step(name: str, seed: int = 0, B: int | None = None, device: str = "cpu"):
    """Inputs of one decode step against a KV cache for workload ``name``:
    q [B, 1, H, d], k_new/v_new [B, 1, Hkv, d], caches [B, Hkv, capacity, d]
    (every row drawn, so rows past each total are finite), seqlens_k int32
    [B] = totals - 1, rotary tables.  Totals come from a CPU generator seeded
    with ``seed``; values from a generator on ``device`` seeded with seed + 1."""
    w = WORKLOADS[name]
    p = w.params
    B = w.B if B is None else B
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    totals = torch.randint(p["lo"], p["hi"] + 1, (B,), generator=gen).tolist()
    vg = torch.Generator(device)
    vg.manual_seed(seed + 1)
    td = DTYPES[w.dtype]
    H, Hkv, d, cap = w.num_heads, w.kv_num_heads, w.head_size, p["capacity"]

    def draw(*shape):
        return (torch.randn(shape, generator=vg, device=device) * w.sigma).to(td)

    cos, sin = rotary_tables(p["cache_rows"], p["rotary_dim"])
    return {
        "name": name, "B": B, "num_heads": H, "kv_num_heads": Hkv, "head_size": d,
        "capacity": cap, "totals": totals,
        "q": draw(B, 1, H, d), "k_new": draw(B, 1, Hkv, d), "v_new": draw(B, 1, Hkv, d),
        "k_cache": draw(B, Hkv, cap, d), "v_cache": draw(B, Hkv, cap, d),
        "seqlens_k": torch.tensor([t - 1 for t in totals], dtype=torch.int32, device=device),
        "cos": cos.to(device), "sin": sin.to(device), "dtype": w.dtype,
    }
