"""pva_forward_from_host: the batch in (pinned) host memory, copied in and out
by the call chunk by chunk and overlapped with the attention.  The output
must match the fp64 oracle, and pva_forward on device copies of the same
batch up to rounding: a chunk ends its packed K/V earlier than the whole
batch does, so the last key tile of a chunk's last sequence is shifted
differently and its products are summed in another order."""
import pytest
import torch

import gqa_attention_cu_gb300 as pva
from gqa_attention_cu_gb300 import workloads
import oracle

from test_gpu_parity import check

pytestmark = pytest.mark.gpu


def _host_call(q, k, v, cq, ck, H, Hkv, d, dv, causal, softcap, chunks):
    dev = torch.device("cuda:0")
    B = cq.numel() - 1
    host = {n: t.cpu().contiguous().pin_memory() for n, t in
            (("q", q), ("k", k), ("v", v), ("cq", cq.to(torch.int32)), ("ck", ck.to(torch.int32)))}
    out_host = torch.full((q.shape[0], H, dv), float("nan"), dtype=q.dtype).pin_memory()
    qd, kd, vd = (torch.empty_like(host[n], device=dev) for n in ("q", "k", "v"))
    od = torch.empty(out_host.shape, dtype=q.dtype, device=dev)
    cu = torch.zeros(4 * B + 34, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream()
    pva.pva_forward_from_host(host["q"], host["k"], host["v"], host["cq"], host["ck"], out_host,
                              qd, kd, vd, od, cu, B, H, Hkv, d, dv, 0.0, int(causal), softcap,
                              chunks=chunks, stream=s)
    s.synchronize()
    assert pva.pva_get_status(s) == 0
    return out_host


def _device_call(q, k, v, cq, ck, H, Hkv, d, dv, causal, softcap):
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty(q.shape[0], H, dv, dtype=q.dtype, device=dev)
    pva.pva_forward(qd, kd, vd, cq.to(dev), ck.to(dev), out, cq.numel() - 1, H, Hkv, d, dv, 0.0,
                    int(causal), softcap)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("chunks", [0, 1, 3, 16])
def test_prefill_batch_matches_device_call(chunks):
    lq = [300, 0, 77, 520, 129, 1000, 3]
    lkv = [300, 40, 200, 520, 129, 1000, 3]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 16, 4, 128, 128, "bf16", seed=51)
    got = _host_call(q, k, v, cq, ck, 16, 4, 128, 128, True, 0.0, chunks)
    ref = _device_call(q, k, v, cq, ck, 16, 4, 128, 128, True, 0.0)
    assert torch.isfinite(got.float()).all()
    assert (got.float() - ref.float()).abs().max().item() <= 1.6e-2
    check(got, oracle.attention(q, k, v, cq, ck, 16, 4, 0.0, True, 0.0), "bf16")


@pytest.mark.parametrize("d,dv,chunks", [(256, 256, 2), (192, 128, 5), (64, 64, 0)])
def test_mixed_prefill_and_decode_rows_against_the_oracle(d, dv, chunks):
    # single-row sequences (split-KV decode) among prefill ones; a chunk's
    # decode splits depend on its batch, so only the oracle bound applies
    lq = [1, 200, 1, 1, 64, 0, 1]
    lkv = [900, 260, 3000, 1, 64, 10, 129]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 8, 2, d, dv, "bf16", seed=52 + d)
    got = _host_call(q, k, v, cq, ck, 8, 2, d, dv, True, 30.0, chunks)
    check(got, oracle.attention(q, k, v, cq, ck, 8, 2, 0.0, True, 30.0), "bf16")


def test_fp32_batch_and_empty_chunks():
    # zero-length sequences on both sides make chunks with nothing to move
    lq = [0, 0, 17, 64, 0, 1, 130]
    lkv = [0, 5, 17, 64, 0, 30, 130]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 4, 4, 64, 64, "f32", seed=53)
    got = _host_call(q, k, v, cq, ck, 4, 4, 64, 64, False, 0.0, 7)
    check(got, oracle.attention(q, k, v, cq, ck, 4, 4, 0.0, False, 0.0), "f32")


def test_release_between_calls():
    """pva_release destroys the entry point's copy streams and events; the
    next call creates them again."""
    lq, lkv = [40, 1, 300], [40, 700, 300]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 8, 2, 128, 128, "bf16", seed=54)
    ref = oracle.attention(q, k, v, cq, ck, 8, 2, 0.0, True, 0.0)
    check(_host_call(q, k, v, cq, ck, 8, 2, 128, 128, True, 0.0, 2), ref, "bf16")
    pva.pva_release()
    check(_host_call(q, k, v, cq, ck, 8, 2, 128, 128, True, 0.0, 2), ref, "bf16")
