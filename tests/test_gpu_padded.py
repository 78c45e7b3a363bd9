"""The padded front end (pva_forward_padded) against the oracle.

The opset-24 Attention input ``nonpad_kv_seqlen`` (attention.rs: per-batch
causal offset nonpad[b] - q_seq and padding frontier j >= nonpad[b]; the
packed_varlen_attention.rs module doc relates it to the packed op through the
exclusive prefix sum).  Each case runs the CUDA path on the padded tensors --
whose padding rows hold values that would wreck any output attending them --
and compares it with ``oracle.attention_padded`` element by element; one case
also checks the packed entry point on the same rows, and one that NaN or Inf
padding changes no output bit.
"""
import numpy as np
import pytest
import torch

import gqa_attention_cu_gb300 as pva
import oracle
from gqa_attention_cu_gb300 import workloads
from test_gpu_parity import TOL, check, run_gpu

pytestmark = pytest.mark.gpu

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def padded_inputs(B, q_seq, kv_seq, nonpad, H, Hkv, d, dv, dtype, sigma=1.0, seed=0,
                  pad=(60.0, -300.0)):
    g = torch.Generator().manual_seed(seed)
    td = DTYPES[dtype]
    q = (torch.randn(B, q_seq, H, d, generator=g) * sigma).to(td)
    k = (torch.randn(B, kv_seq, Hkv, d, generator=g) * sigma).to(td)
    v = (torch.randn(B, kv_seq, Hkv, dv, generator=g) * sigma).to(td)
    for b, n in enumerate(nonpad):  # padding: large, finite, never attended
        k[b, n:] = pad[0]
        v[b, n:] = pad[1]
    return q, k, v, torch.tensor(nonpad, dtype=torch.int64)


def run_padded(q, k, v, nonpad, H, Hkv, scale=0.0, causal=False, softcap=0.0, expect=0):
    dev = torch.device("cuda:0")
    B, q_seq, _, d = q.shape
    kv_seq, dv = k.shape[1], v.shape[-1]
    q, k, v, nonpad = (t.to(dev) for t in (q, k, v, nonpad))
    out = torch.full((B, q_seq, H, dv), float("nan"), dtype=q.dtype, device=dev)
    pva.pva_forward_padded(q, k, v, nonpad, out, B, q_seq, kv_seq, H, Hkv, d, dv, scale,
                           int(causal), softcap)
    flags = pva.pva_get_status()
    assert flags == expect, f"device status bits {flags:#x}"
    return out


def padded_parity(B, q_seq, kv_seq, nonpad, H, Hkv, d, dv, dtype, causal, softcap=0.0,
                  sigma=1.0, seed=0):
    q, k, v, npd = padded_inputs(B, q_seq, kv_seq, nonpad, H, Hkv, d, dv, dtype, sigma, seed)
    out = run_padded(q, k, v, npd, H, Hkv, 0.0, causal, softcap)
    ref = oracle.attention_padded(q, k, v, npd, H, Hkv, 0.0, causal, softcap)
    return check(out, ref, dtype)


# q_seq = 1 rows of d = dv in {64, 128, 256} go to the split-KV decode kernel
@pytest.mark.parametrize("H,Hkv,d", [(32, 8, 128), (8, 8, 64), (16, 2, 256)])
def test_padded_decode(H, Hkv, d):
    g = torch.Generator().manual_seed(d)
    kv_seq = 3000
    nonpad = torch.randint(0, kv_seq + 1, (24,), generator=g).tolist()
    nonpad[:4] = [0, kv_seq, 1, 129]
    padded_parity(24, 1, kv_seq, nonpad, H, Hkv, d, d, "bf16", True, seed=d)


# prefill rows through the paired kernel (d = 128, 64) and the single-tile
# kernel (256, 192/128); nonpad below q_seq leaves leading rows fully masked
@pytest.mark.parametrize("d,dv", [(128, 128), (64, 64), (256, 256), (192, 128)])
def test_padded_prefill_causal(d, dv):
    padded_parity(5, 300, 900, [900, 300, 517, 100, 0], 16, 4, d, dv, "bf16", True, seed=d)


# bf16 keeps unit-variance inputs (outputs near 8 would put one bf16 ulp,
# 0.03, above the 2e-2 bound); f16 takes the wider draw
@pytest.mark.parametrize("dtype,sigma", [("bf16", 1.0), ("f16", 2.0)])
def test_padded_prefill_noncausal_softcap(dtype, sigma):
    padded_parity(4, 129, 640, [640, 1, 333, 64], 8, 2, 128, 128, dtype, False, softcap=20.0,
                  sigma=sigma, seed=4)


@pytest.mark.parametrize("q_seq,causal", [(1, True), (129, False), (300, True)])
def test_padding_contents_do_not_change_a_bit(q_seq, causal):
    """Keys past nonpad get weight exactly 0 and the row maximum is taken over
    visible keys only, so any finite padding gives bit-identical outputs."""
    args = (5, q_seq, 900, [900, 1, 0, 517, 100], 16, 4, 128, 128, "bf16")
    outs = []
    for pad in ((0.0, 0.0), (60.0, -300.0), (-1e4, 3e4)):
        q, k, v, npd = padded_inputs(*args, seed=8, pad=pad)
        outs.append(run_padded(q, k, v, npd, 16, 4, 0.0, causal, softcap=30.0))
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("q_seq,kv_seq,H,Hkv,d,dv,dtype", [
    (1, 3000, 32, 8, 128, 128, "bf16"),   # split-KV decode
    (1, 700, 8, 1, 256, 256, "bf16"),
    (1, 40, 16, 2, 192, 128, "bf16"),     # decode, slots shorter than a tile
    (300, 900, 16, 4, 128, 128, "bf16"),  # paired prefill
    (129, 5, 8, 2, 64, 64, "f16"),        # paired prefill, 5-row slots
    (200, 640, 8, 1, 256, 256, "bf16"),   # single-tile prefill
    (130, 300, 16, 4, 192, 128, "bf16"),
    (17, 90, 4, 2, 64, 48, "f32"),        # fp32 kernel
])
def test_nan_and_inf_padding_give_the_outputs_of_zero_padding(q_seq, kv_seq, H, Hkv, d, dv,
                                                             dtype):
    """No kernel ever loads a row past nonpad[b]: the last key tile of each
    slot ends at its last key, so padding may hold anything -- NaN and Inf
    included -- and the outputs are bit for bit those of zero padding."""
    nonpad = [kv_seq, 1, 0, max(1, kv_seq // 3), max(1, kv_seq - 7)]
    B = len(nonpad)
    causal = q_seq != 129
    outs = []
    for pad in ((0.0, 0.0), (float("nan"), float("nan")), (float("inf"), float("-inf"))):
        q, k, v, npd = padded_inputs(B, q_seq, kv_seq, nonpad, H, Hkv, d, dv, dtype, seed=9,
                                     pad=pad)
        outs.append(run_padded(q, k, v, npd, H, Hkv, 0.0, causal, softcap=20.0))
    ref = oracle.attention_padded(*padded_inputs(B, q_seq, kv_seq, nonpad, H, Hkv, d, dv, dtype,
                                                 seed=9, pad=(0.0, 0.0))[:4], H, Hkv, 0.0,
                                  causal, 20.0)
    check(outs[0], ref, dtype)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_padded_fp32():
    padded_parity(3, 17, 90, [90, 5, 0], 4, 2, 64, 48, "f32", True, seed=5)
    padded_parity(3, 17, 90, [33, 90, 17], 4, 2, 64, 48, "f32", False, seed=6)


def test_padded_equals_packed_entry_point():
    """The same logical batch through pva_forward (rows packed on the host)
    and pva_forward_padded: both within tolerance of the oracle and of each
    other."""
    B, q_seq, kv_seq, H, Hkv, d = 6, 200, 700, 16, 4, 128
    nonpad = [700, 650, 200, 513, 1, 380]
    q, k, v, npd = padded_inputs(B, q_seq, kv_seq, nonpad, H, Hkv, d, d, "bf16", seed=9)
    a = run_padded(q, k, v, npd, H, Hkv, 0.0, True)
    kp = torch.cat([k[b, :n] for b, n in enumerate(nonpad)])
    vp = torch.cat([v[b, :n] for b, n in enumerate(nonpad)])
    b_ = run_gpu(q.reshape(B * q_seq, H, d), kp, vp, workloads.cu_from_lengths([q_seq] * B),
                 workloads.cu_from_lengths(nonpad), H, Hkv, 0.0, True)
    ref = oracle.attention_padded(q, k, v, npd, H, Hkv, 0.0, True)
    check(a, ref, "bf16")
    check(b_, ref.reshape(B * q_seq, H, d), "bf16")
    diff = (a.reshape(B * q_seq, H, d).double() - b_.double()).abs().max().item()
    assert diff <= TOL["bf16"][0]


@pytest.mark.parametrize("bad", [-1, 701, 1 << 40])
def test_padded_length_outside_slot_is_reported_and_writes_nothing(bad):
    q, k, v, npd = padded_inputs(3, 50, 700, [700, 20, 300], 8, 2, 128, 128, "bf16", seed=1)
    npd[1] = bad
    out = run_padded(q, k, v, npd, 8, 2, 0.0, True, expect=pva.DEV_FLAGS["kv_len"])
    assert torch.isnan(out.float()).all()


def test_padded_empty_slots_and_queries():
    # kv_seq = 0: every row fully masked -> zeros; q_seq = 0: nothing to do
    q, k, v, npd = padded_inputs(3, 7, 0, [0, 0, 0], 4, 4, 128, 128, "bf16", seed=2)
    out = run_padded(q, k, v, npd, 4, 4, 0.0, False)
    assert torch.equal(out.float().cpu(), torch.zeros(out.shape))
    q, k, v, npd = padded_inputs(2, 0, 64, [64, 10], 4, 4, 128, 128, "bf16", seed=3)
    out = run_padded(q, k, v, npd, 4, 4, 0.0, True)
    assert out.numel() == 0
