"""One GroupQueryAttention step against a fixed-capacity KV cache
(pva_gqa_kvcache) against the cache-step oracle.

group_query_attention.rs: metadata (totals = seqlens_k + 1, past, first query
row, bounds with a sticky latch), in-place append, rotary embedding of the
queries and appended keys, causal attention over the valid cache rows read
from the BNSH planes.  The attention output is held to the bf16/f16/f32
tolerances; the cache after the step must match the oracle's bit for bit
(append and rotation are exact given the page's f32 arithmetic).
"""
import math

import numpy as np
import pytest
import torch

import gqa_attention_cu_gb300 as pva
from oracle import gqa_cache
from test_gpu_parity import check

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def tables(rows, rot, dtype=torch.float32):
    theta = 10000.0 ** (-torch.arange(rot // 2, dtype=torch.float64) / (rot // 2))
    ang = torch.arange(rows, dtype=torch.float64)[:, None] * theta[None, :]
    return torch.cos(ang).to(dtype), torch.sin(ang).to(dtype)


def make_step(B, q_seq, k_seq, H, Hkv, d, cap, dtype, seed, totals=None, stale=0.0):
    """Random step inputs; cache rows at or past each total are set to
    `stale` (the step must never read them)."""
    g = torch.Generator().manual_seed(seed)
    td = DT[dtype]
    q = torch.randn(B, q_seq, H, d, generator=g).to(td)
    kn = torch.randn(B, k_seq, Hkv, d, generator=g).to(td) if k_seq else None
    vn = torch.randn(B, k_seq, Hkv, d, generator=g).to(td) if k_seq else None
    kc = torch.randn(B, Hkv, cap, d, generator=g).to(td)
    vc = torch.randn(B, Hkv, cap, d, generator=g).to(td)
    if totals is None:
        lo = max(q_seq, k_seq, 1)
        totals = torch.randint(lo, cap + 1, (B,), generator=g).tolist()
    for b, t in enumerate(totals):
        kc[b, :, t:] = stale
        vc[b, :, t:] = stale
    sk = torch.tensor([t - 1 for t in totals], dtype=torch.int32)
    return q, kn, vn, kc, vc, sk


def run_step(q, kn, vn, kc, vc, sk, H, Hkv, cos=None, sin=None, pid=None, inter=False,
             scale=0.0, softcap=0.0, window=0, expect=0):
    dev = torch.device("cuda:0")
    to = (lambda t: None if t is None else t.to(dev))
    qd, knd, vnd, kcd, vcd, skd = (to(t) for t in (q, kn, vn, kc, vc, sk))
    cosd, sind = to(cos), to(sin)
    pidd = None if pid is None else torch.as_tensor(pid, dtype=torch.int64).to(dev)
    out = torch.full(q.shape, float("nan"), dtype=q.dtype, device=dev)
    pva.pva_gqa_kvcache(qd, knd, vnd, kcd, vcd, skd, out, H, Hkv, cosd, sind, pidd, inter,
                        scale, softcap, window)
    flags = pva.pva_get_status()
    assert flags == expect, f"device status bits {flags:#x}"
    return out, kcd.cpu(), vcd.cpu()


def same_bits(a, b):
    """Bitwise equality (NaN payloads included)."""
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def step_parity(B, q_seq, k_seq, H, Hkv, d, cap, dtype, seed, rot=0, rows=0, inter=False,
                table_dtype=torch.float32, use_pid=False, scale=0.0, softcap=0.0, window=0,
                totals=None, stale=0.0):
    q, kn, vn, kc, vc, sk = make_step(B, q_seq, k_seq, H, Hkv, d, cap, dtype, seed, totals,
                                      stale)
    cos = sin = pid = None
    if rot:
        cos, sin = tables(rows, rot, table_dtype)
    if use_pid:
        g = torch.Generator().manual_seed(seed + 7)
        pid = torch.randint(0, rows, (B, q_seq), generator=g).numpy()
    out, ka, va = run_step(q, kn, vn, kc, vc, sk, H, Hkv, cos, sin, pid, inter, scale,
                           softcap, window)
    ref, ka_ref, va_ref, bits = gqa_cache.gqa_cache_step(
        q, kn, vn, kc, vc, sk.tolist(), H, Hkv, cos, sin, pid, inter, scale, softcap, window)
    assert bits == 0
    assert same_bits(ka, ka_ref), "key cache differs from the oracle's"
    assert same_bits(va, va_ref), "value cache differs from the oracle's"
    return check(out.reshape(-1, H, d), ref.reshape(-1, H, d), dtype)


# ---- decode (q_seq = 1): the split-KV kernel reads the cache planes ---------
def test_decode_bf16_rotary_half_split():
    step_parity(32, 1, 1, 32, 8, 128, 2048, "bf16", 1, rot=128, rows=2048)


def test_decode_f16_partial_interleaved_rotary_f16_tables_position_ids():
    step_parity(16, 1, 1, 16, 2, 128, 700, "f16", 2, rot=64, rows=900, inter=True,
                table_dtype=torch.float16, use_pid=True)


@pytest.mark.parametrize("H,Hkv,d", [(8, 8, 64), (16, 2, 256), (8, 4, 128)])
def test_decode_shapes_no_rotary(H, Hkv, d):
    step_parity(12, 1, 1, H, Hkv, d, 1500, "bf16", d + H)


def test_decode_attend_without_append_window_softcap():
    step_parity(20, 1, 0, 32, 8, 128, 3000, "bf16", 4, window=700, softcap=30.0)


def test_decode_ignores_whatever_the_unused_cache_rows_hold():
    # rows at or past each total hold NaN and are never read
    totals = [1, 63, 64, 65, 500, 1000, 129, 2047]
    step_parity(8, 1, 1, 32, 8, 128, 2047, "bf16", 5, rot=128, rows=2048, totals=totals,
                stale=float("nan"))


# ---- chunks of queries (q_seq > 1): the tensor-core prefill kernels ----------
@pytest.mark.parametrize("d", [128, 256])
def test_chunk_ignores_whatever_the_unused_cache_rows_hold(d):
    # totals below, at and just past one key tile (128 keys for d = 128, 64
    # for d = 256): the last tile is shifted to end at the last key, reading
    # zeros before row 0 when the sequence is shorter than a tile
    totals = [40, 63, 64, 65, 100, 128, 129, 1000]
    step_parity(8, 40, 40, 16, 4, d, 1024, "bf16", 30 + d, rot=d, rows=1024, totals=totals,
                stale=float("nan"))


@pytest.mark.parametrize("d", [128, 64, 256])
def test_chunk_rotary(d):
    step_parity(4, 100, 100, 16, 4, d, 1024, "bf16", 10 + d, rot=d, rows=1024)


def test_chunk_window_softcap_f16_interleaved():
    step_parity(3, 130, 130, 8, 2, 128, 900, "f16", 11, rot=96, rows=1200, inter=True,
                window=200, softcap=25.0)


def test_chunk_without_append_and_uneven_k_seq():
    # k_seq = 0 (queries against the cache as it is) and k_seq != q_seq (no rotary)
    step_parity(3, 64, 0, 8, 2, 128, 512, "bf16", 12)
    step_parity(3, 40, 17, 8, 2, 128, 512, "bf16", 13)


def test_fp32_step():
    step_parity(3, 5, 5, 4, 2, 64, 90, "f32", 14, rot=32, rows=100)
    step_parity(5, 1, 1, 4, 1, 64, 90, "f32", 15, rot=64, rows=100, inter=True)


def test_full_capacity_and_single_row_totals():
    step_parity(4, 1, 1, 32, 8, 128, 4096, "bf16", 16, rot=128, rows=4096,
                totals=[4096, 1, 2, 4095])
    step_parity(3, 50, 50, 16, 4, 128, 300, "bf16", 17, rot=128, rows=300,
                totals=[300, 50, 51])


# ---- rejected steps -----------------------------------------------------------
def test_rejected_step_writes_nothing_and_poisons_until_read():
    dev = torch.device("cuda:0")
    q, kn, vn, kc, vc, sk = make_step(3, 1, 1, 8, 2, 128, 64, "bf16", 20, totals=[10, 64, 3])
    kcd, vcd = kc.to(dev), vc.to(dev)
    out = torch.full(q.shape, float("nan"), dtype=q.dtype, device=dev)
    bad = sk.clone()
    bad[1] = 64  # total 65 > capacity 64
    args = (q.to(dev), kn.to(dev), vn.to(dev), kcd, vcd)
    pva.pva_gqa_kvcache(*args, bad.to(dev), out, 8, 2)
    # a valid step right after the rejected one is refused too (latch-first)
    pva.pva_gqa_kvcache(*args, sk.to(dev), out, 8, 2)
    assert pva.pva_get_status() == pva.DEV_FLAGS["kv_cache"]
    assert same_bits(kcd.cpu(), kc) and same_bits(vcd.cpu(), vc)
    assert torch.isnan(out.float()).all()
    # once the bit is read (and cleared) the valid step goes through
    pva.pva_gqa_kvcache(*args, sk.to(dev), out, 8, 2)
    assert pva.pva_get_status() == 0
    ref, ka_ref, _, bits = gqa_cache.gqa_cache_step(q, kn, vn, kc, vc, sk.tolist(), 8, 2)
    assert bits == 0 and same_bits(kcd.cpu(), ka_ref)
    check(out.reshape(-1, 8, 128), ref.reshape(-1, 8, 128), "bf16")


@pytest.mark.parametrize("case", ["first_negative", "position_outside_table"])
def test_other_bounds_reject_the_step(case):
    dev = torch.device("cuda:0")
    if case == "first_negative":
        q, kn, vn, kc, vc, sk = make_step(2, 8, 0, 8, 2, 128, 64, "bf16", 21, totals=[10, 5])
        cos = sin = None
    else:
        q, kn, vn, kc, vc, sk = make_step(2, 1, 1, 8, 2, 128, 64, "bf16", 22, totals=[10, 40])
        cos, sin = tables(32, 128)  # position 39 is outside the 32-row tables
    kcd, vcd = kc.to(dev), vc.to(dev)
    out = torch.full(q.shape, float("nan"), dtype=q.dtype, device=dev)
    to = (lambda t: None if t is None else t.to(dev))
    pva.pva_gqa_kvcache(q.to(dev), to(kn), to(vn), kcd, vcd, sk.to(dev), out, 8, 2, to(cos),
                        to(sin))
    assert pva.pva_get_status() == pva.DEV_FLAGS["kv_cache"]
    assert same_bits(kcd.cpu(), kc) and torch.isnan(out.float()).all()


def test_full_size_step_sampled_sequences():
    """The step the benchmark times (B = 256, capacity 8192, totals up to
    8192, rotary on 128 dims), checked on sampled sequences: their appended
    cache rows bit for bit and their outputs within the bf16 tolerance."""
    from gqa_attention_cu_gb300 import workloads
    c = workloads.make_cache_step("bf16_kvcache_decode", seed=0, device="cuda:0")
    B, H, Hkv, d = c["B"], c["num_heads"], c["kv_num_heads"], c["head_size"]
    pick = [0, 1, B // 2, B - 1]
    k0, v0 = c["k_cache"][pick].cpu(), c["v_cache"][pick].cpu()
    out = torch.empty_like(c["q"])
    pva.pva_gqa_kvcache(c["q"], c["k_new"], c["v_new"], c["k_cache"], c["v_cache"],
                        c["seqlens_k"], out, H, Hkv, c["cos"], c["sin"])
    assert pva.pva_get_status() == 0
    ref, ka, va, bits = gqa_cache.gqa_cache_step(
        c["q"][pick].cpu(), c["k_new"][pick].cpu(), c["v_new"][pick].cpu(), k0, v0,
        c["seqlens_k"][pick].cpu().tolist(), H, Hkv, c["cos"].cpu(), c["sin"].cpu())
    assert bits == 0
    assert same_bits(c["k_cache"][pick].cpu(), ka) and same_bits(c["v_cache"][pick].cpu(), va)
    check(out[pick].reshape(-1, H, d), ref.reshape(-1, H, d), "bf16")
