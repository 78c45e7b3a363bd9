"""Local (sliding) window through every kernel path, against the oracle.

pva_forward_local with local_window = W > 0 masks, for query row i of a
sequence (causal limit c = i + L_kv - L_q), the keys j < c + 1 - W -- the
`local_window` of the softmax / grouped-query reference kernels on the
attention.rs and group_query_attention.rs pages.
"""
import numpy as np
import pytest
import torch

import gqa_attention_cu_gb300 as pva
import oracle
from gqa_attention_cu_gb300 import workloads
from test_gpu_parity import check

pytestmark = pytest.mark.gpu


def run_local(q, k, v, cq, ck, H, Hkv, scale, causal, softcap, window):
    dev = torch.device("cuda:0")
    q, k, v, cq, ck = (t.to(dev) for t in (q, k, v, cq, ck))
    out = torch.full((q.shape[0], H, v.shape[-1]), float("nan"), dtype=q.dtype, device=dev)
    pva.pva_forward_local(q, k, v, cq, ck, out, cq.numel() - 1, H, Hkv, q.shape[-1],
                          v.shape[-1], scale, int(causal), softcap, window)
    assert pva.pva_get_status() == 0
    return out


def window_parity(lq, lkv, H, Hkv, d, dv, dtype, causal, window, softcap=0.0, sigma=1.0, seed=0):
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, H, Hkv, d, dv, dtype, sigma=sigma, seed=seed)
    out = run_local(q, k, v, cq, ck, H, Hkv, 0.0, causal, softcap, window)
    ref = oracle.attention(q, k, v, cq, ck, H, Hkv, 0.0, causal, softcap, local_window=window)
    return check(out, ref, dtype)


# d = 128 and 64 run the paired kernel (128-key tiles), 256 and 192/128 the
# single-tile kernel (64-key tiles); windows below, at and across tile edges.
@pytest.mark.parametrize("window", [1, 17, 64, 128, 129, 700])
@pytest.mark.parametrize("d,dv", [(128, 128), (64, 64), (256, 256), (192, 128)])
def test_window_prefill_causal(window, d, dv):
    window_parity([300, 1, 77, 520, 129], [300, 900, 77, 520, 140], 16, 4, d, dv, "bf16",
                  True, window, seed=window + d)


@pytest.mark.parametrize("window", [1, 40, 300])
@pytest.mark.parametrize("d", [128, 256])
def test_window_prefill_noncausal(window, d):
    window_parity([200, 64, 3], [260, 500, 3], 8, 2, d, d, "bf16", False, window, seed=window)


@pytest.mark.parametrize("window", [5, 100])
def test_window_chunked_f16_softcap(window):
    window_parity([37, 256, 1], [1000, 300, 1], 16, 8, 128, 128, "f16", True, window,
                  softcap=20.0, sigma=2.0, seed=3)


@pytest.mark.parametrize("window", [1, 33, 2000])
def test_window_decode_rows(window):
    # single-row sequences go to the split-KV decode kernel (G = 4, d = 128)
    window_parity([1] * 12, [1, 7, 64, 65, 500, 1024, 3000, 4097, 8192, 100, 129, 2048],
                  32, 8, 128, 128, "bf16", True, window, seed=window)


@pytest.mark.parametrize("window", [1, 9, 50])
def test_window_fp32(window):
    window_parity([17, 64, 1, 130], [40, 64, 90, 130], 4, 2, 64, 48, "f32", True, window,
                  seed=window)


def test_window_zero_is_pva_forward_bitwise():
    q, k, v, cq, ck = workloads.make_packed([300, 5, 129], [400, 5, 129], 16, 4, 128, 128,
                                            "bf16", seed=2)
    dev = torch.device("cuda:0")
    a = run_local(q, k, v, cq, ck, 16, 4, 0.0, True, 0.0, 0)
    b = torch.empty_like(a)
    pva.pva_forward(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), b, 3, 16, 4, 128,
                    128, 0.0, 1, 0.0)
    assert torch.equal(a, b)
    c = run_local(q, k, v, cq, ck, 16, 4, 0.0, True, 0.0, -5)
    assert torch.equal(a, c)


def test_window_full_size_workload_sampled_rows():
    """The windowed long-context workload the benchmark runs (4 sequences of
    8k-32k tokens, window 4096), checked on sampled rows of every sequence."""
    w = workloads.make("bf16_window", device="cuda:0")
    H, Hkv, d = w["num_heads"], w["kv_num_heads"], w["head_size"]
    out = torch.empty(w["q"].shape[0], H, d, dtype=w["q"].dtype, device="cuda:0")
    pva.pva_forward_local(w["q"], w["k"], w["v"], w["cu_q"], w["cu_kv"], out, w["B"], H, Hkv,
                          d, d, w["scale"], 1, 0.0, w["window"])
    assert pva.pva_get_status() == 0
    g = np.random.default_rng(3)
    cq = w["cu_q"].cpu()
    for b in range(w["B"]):
        L = w["lq"][b]
        s0 = int(cq[b])
        q = w["q"][s0:s0 + L].cpu()
        k = w["k"][s0:s0 + L].cpu()
        v = w["v"][s0:s0 + L].cpu()
        c1 = torch.tensor([0, L], dtype=torch.int32)
        cand = np.unique(np.concatenate([np.arange(16), np.arange(L - 16, L),
                                         g.integers(0, L, size=24)]))
        rows = np.array([int(i) * H + hh for i in cand for hh in range(0, H, 5)], dtype=np.int64)
        ref = oracle.attention_rows(q, k, v, c1, c1, rows, H, Hkv, 0.0, True, 0.0,
                                    local_window=w["window"])
        got = out[s0:s0 + L].reshape(-1, d)[torch.tensor(rows, device="cuda:0")]
        check(got, ref, "bf16")
