"""pva_forward_noalloc: the entry point for callers that cannot allocate
device memory at call time (planned arenas, memory governors, fixed device
footprints).  It runs on the library's fixed per-device scratch array, so
its output must match pva_forward's -- twice in a row, since the array keeps
the previous call's contents and each call must clear what has to start at
zero.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import gqa_attention_cu_gb300 as pva
from gqa_attention_cu_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN = 2e-2, 2e-3  # the bf16 tolerances of the parity tests


@pytest.fixture(scope="module")
def lib(cuda_device):
    pva.build()
    return pva.load_library()


def _call_noalloc(lib, w, out, status, stream):
    rc = lib.pva_forward_noalloc(
        w["q"].data_ptr(), w["k"].data_ptr(), w["v"].data_ptr(), w["cu_q"].data_ptr(),
        w["cu_kv"].data_ptr(), out.data_ptr(), w["B"], w["H"], w["Hkv"], w["d"], w["d"],
        ctypes.c_float(0.0), 1, ctypes.c_float(0.0), 2,
        status.data_ptr() if status is not None else None, stream)
    assert rc == 0, pva.pva_last_error()


def _batch(seed):
    # prefill sequences, decode sequences long enough to be split, an empty one
    lq = [300, 1, 1, 77, 0, 1, 129]
    lkv = [300, 6000, 2500, 900, 5, 1, 129]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 32, 8, 128, 128, "bf16", seed=seed,
                                            device="cuda:0")
    return {"q": q, "k": k, "v": v, "cu_q": cq, "cu_kv": ck, "B": len(lq), "H": 32, "Hkv": 8,
            "d": 128}


def _compare(a, b):
    err = (a.double() - b.double()).abs()
    assert torch.isfinite(a.float()).all()
    assert err.max().item() <= TOL_MAX and err.mean().item() <= TOL_MEAN


def test_noalloc_matches_pva_forward_on_two_calls_in_a_row(lib):
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((5, 6)):
        w = _batch(seed)
        ref = torch.empty(w["q"].shape[0], 32, 128, dtype=torch.bfloat16, device="cuda:0")
        pva.pva_forward(w["q"], w["k"], w["v"], w["cu_q"], w["cu_kv"], ref, w["B"], 32, 8, 128,
                        128, 0.0, 1, 0.0)
        assert pva.pva_get_status() == 0
        out = torch.full_like(ref, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        _call_noalloc(lib, w, out, status, stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item()):#x}"
        _compare(out, ref)


def test_noalloc_internal_status_and_repeat(lib):
    """Without a caller status word the call uses (and first clears) its own;
    a repeat of the same call reproduces the output."""
    stream = torch.cuda.current_stream().cuda_stream
    w = _batch(7)
    a = torch.empty(w["q"].shape[0], 32, 128, dtype=torch.bfloat16, device="cuda:0")
    b = torch.empty_like(a)
    _call_noalloc(lib, w, a, None, stream)
    _call_noalloc(lib, w, b, None, stream)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


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
