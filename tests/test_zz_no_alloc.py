"""pva_forward_noalloc: the entry point for callers that cannot allocate
device memory at call time (planned arenas, memory governors, fixed device
footprints).  It runs on the library's fixed per-device scratch array, so its
output must match pva_forward's and the fp64 oracle's -- twice in a row,
since the array keeps the previous call's contents and each call must clear
what has to start at zero.  Besides the GQA batch of the main parity tests it
covers a decode batch whose split partials do not all fit in the array (the
scheduler must fall back to fewer, longer splits), the single-tile kernel
(d = 256) and the fp32 kernel, and checks that no call changes the device's
free memory.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import gqa_attention_cu_gb300 as pva
import oracle
from gqa_attention_cu_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 2e-3), "f32": (2e-5, None)}  # the parity tests' tolerances
DCODE = {"f32": 0, "f16": 1, "bf16": 2}

# Size of the static scratch regions (the library's pva_noalloc.cu): 256-byte
# status word, 1 MiB of work lists, the rest of 4 MiB for decode partials.
PARTIAL_BYTES = (4 << 20) - 256 - (1 << 20)


@pytest.fixture(scope="module")
def lib(cuda_device):
    pva.build()
    return pva.load_library()


def _batch(lq, lkv, H, Hkv, d, dv, dtype, seed, scale=0.0, causal=True, softcap=0.0):
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, H, Hkv, d, dv, dtype, seed=seed)
    dev = torch.device("cuda:0")
    return {"host": (q, k, v, cq, ck), "q": q.to(dev), "k": k.to(dev), "v": v.to(dev),
            "cu_q": cq.to(dev), "cu_kv": ck.to(dev), "B": len(lq), "H": H, "Hkv": Hkv,
            "d": d, "dv": dv, "dtype": dtype, "scale": scale, "causal": causal,
            "softcap": softcap}


def _gqa_batch(seed):
    # prefill sequences, decode sequences long enough to be split, an empty one
    return _batch([300, 1, 1, 77, 0, 1, 129], [300, 6000, 2500, 900, 5, 1, 129], 32, 8, 128,
                  128, "bf16", seed)


def _call_noalloc(lib, w, out, status, stream):
    rc = lib.pva_forward_noalloc(
        w["q"].data_ptr(), w["k"].data_ptr(), w["v"].data_ptr(), w["cu_q"].data_ptr(),
        w["cu_kv"].data_ptr(), out.data_ptr(), w["B"], w["H"], w["Hkv"], w["d"], w["dv"],
        ctypes.c_float(w["scale"]), int(w["causal"]), ctypes.c_float(w["softcap"]),
        DCODE[w["dtype"]], status.data_ptr() if status is not None else None, stream)
    assert rc == 0, pva.pva_last_error()


def _empty_out(w):
    return torch.full((w["q"].shape[0], w["H"], w["dv"]), float("nan"), dtype=w["q"].dtype,
                      device="cuda:0")


def _oracle(w):
    q, k, v, cq, ck = w["host"]
    return oracle.attention(q, k, v, cq, ck, w["H"], w["Hkv"], w["scale"], w["causal"],
                            w["softcap"])


def _check(out, ref, dtype):
    tol_max, tol_mean = TOL[dtype]
    got = out.double().cpu().numpy().reshape(ref.shape)
    assert np.isfinite(got).all(), "non-finite outputs"
    err = np.abs(got - ref)
    assert err.max() <= tol_max, f"max-abs {err.max():.3e} > {tol_max}"
    if tol_mean is not None:
        assert err.mean() <= tol_mean, f"mean-abs {err.mean():.3e} > {tol_mean}"


def _run_twice_against_oracle(lib, batches):
    """Each batch through pva_forward_noalloc with a caller status word; the
    calls follow each other on one stream, so every call starts from what the
    previous one left in the array."""
    stream = torch.cuda.current_stream().cuda_stream
    for w in batches:
        out = _empty_out(w)
        status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        _call_noalloc(lib, w, out, status, stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"device status {int(status.item()):#x}"
        _check(out, _oracle(w), w["dtype"])


def test_noalloc_matches_pva_forward_on_two_calls_in_a_row(lib):
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((5, 6)):
        w = _gqa_batch(seed)
        ref = torch.empty(w["q"].shape[0], 32, 128, dtype=torch.bfloat16, device="cuda:0")
        pva.pva_forward(w["q"], w["k"], w["v"], w["cu_q"], w["cu_kv"], ref, w["B"], 32, 8, 128,
                        128, 0.0, 1, 0.0)
        assert pva.pva_get_status() == 0
        out = _empty_out(w)
        status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        _call_noalloc(lib, w, out, status, stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item()):#x}"
        err = (out.double() - ref.double()).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= TOL["bf16"][0] and err.mean().item() <= TOL["bf16"][1]


def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(lib):
    _run_twice_against_oracle(lib, [_gqa_batch(8), _gqa_batch(9)])


def test_noalloc_decode_with_fewer_partial_slots_than_splits(lib):
    """d = dv = 256, G = 16, 64 long single-row sequences: the split size the
    scheduler aims at (about 2 units per SM) gives more split units than the
    static array has partial slots for, so it has to choose longer splits to
    fit."""
    G, Hkv, d = 16, 1, 256
    per_unit = (G * d + 2 * G) * 4
    fit = PARTIAL_BYTES // per_unit
    B = 64
    gen = np.random.default_rng(3)
    lkv = [int(x) for x in gen.integers(5000, 8193, size=B)]
    # the scheduler's first split size (its rule restated): keys over 2 units per SM
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    chunk = max(256, -(-(-(-sum(lkv) * Hkv // (2 * sms))) // 64) * 64)
    units = sum(min(16, -(-n // chunk)) for n in lkv) * Hkv
    assert units > fit, "the case must exceed the static partial slots"
    batches = [_batch([1] * B, lkv, G * Hkv, Hkv, d, d, "bf16", seed=s) for s in (11, 12)]
    _run_twice_against_oracle(lib, batches)
    # the same batch through pva_forward (room for every split) agrees too
    w = batches[-1]
    ref = torch.empty_like(_empty_out(w))
    pva.pva_forward(w["q"], w["k"], w["v"], w["cu_q"], w["cu_kv"], ref, B, G * Hkv, Hkv, d, d,
                    0.0, 1, 0.0)
    assert pva.pva_get_status() == 0
    out = _empty_out(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    _call_noalloc(lib, w, out, status, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert (out.double() - ref.double()).abs().max().item() <= TOL["bf16"][0]


def test_noalloc_single_tile_kernel_and_fp32(lib):
    big = _batch([300, 1, 70, 2], [420, 900, 70, 2], 16, 2, 256, 256, "bf16", seed=21,
                 softcap=30.0)
    f32 = _batch([17, 64, 1, 130], [17, 64, 1, 130], 4, 4, 64, 64, "f32", seed=0, scale=0.125,
                 causal=False)
    _run_twice_against_oracle(lib, [big, f32, big, f32])


def test_noalloc_internal_status_and_repeat(lib):
    """Without a caller status word the call uses (and first clears) its own;
    a repeat of the same call reproduces the output."""
    stream = torch.cuda.current_stream().cuda_stream
    w = _gqa_batch(7)
    a = torch.empty(w["q"].shape[0], 32, 128, dtype=torch.bfloat16, device="cuda:0")
    b = torch.empty_like(a)
    _call_noalloc(lib, w, a, None, stream)
    _call_noalloc(lib, w, b, None, stream)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_noalloc_calls_leave_free_device_memory_unchanged(lib):
    """After one warm-up call per kernel family (module loading happens
    there), further calls of several sizes change the device's free memory by
    nothing: the entry point allocates no device memory."""
    stream = torch.cuda.current_stream().cuda_stream
    batches = [_gqa_batch(31),
               _batch([1] * 40, [3000] * 40, 8, 1, 256, 256, "bf16", seed=32),
               _batch([17, 64, 1, 130], [17, 64, 1, 130], 4, 4, 64, 64, "f32", seed=33,
                      scale=0.125, causal=False),
               _batch([700, 5], [900, 5], 16, 2, 192, 128, "bf16", seed=34)]
    outs = [_empty_out(w) for w in batches]
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    for w, o in zip(batches, outs):
        _call_noalloc(lib, w, o, status, stream)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        for w, o in zip(batches, outs):
            _call_noalloc(lib, w, o, status, stream)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert int(status.item()) == 0


def test_noalloc_rejects_batches_beyond_its_scratch(lib):
    big_b = 60000  # B * (4 + Hkv) int32 words > 1 MiB
    dev = torch.device("cuda:0")
    cq = torch.zeros(big_b + 1, dtype=torch.int32, device=dev)
    x = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    rc = lib.pva_forward_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), cq.data_ptr(),
                                 cq.data_ptr(), x.data_ptr(), big_b, 32, 8, 128, 128,
                                 ctypes.c_float(0.0), 1, ctypes.c_float(0.0), 2, None,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == pva.PVA_ERR_UNSUPPORTED
    assert "static scratch" in pva.pva_last_error()
