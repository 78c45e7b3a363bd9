"""pva_forward inside a CUDA graph: once a call on a stream has grown that
stream's workspace, calls on it allocate nothing and synchronise nothing, so
they can be captured; replays recompute from whatever the input buffers hold
at replay time."""
import pytest
import torch

import gqa_attention_cu_gb300 as pva
from gqa_attention_cu_gb300 import workloads
import oracle

from test_gpu_parity import check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,dv,lq,lkv", [
    (128, 128, [300, 1, 77, 520], [300, 900, 77, 600]),   # paired prefill + decode rows
    (256, 256, [200, 64], [260, 64]),                     # single-tile kernel
])
def test_captured_forward_replays_on_new_inputs(d, dv, lq, lkv):
    dev = torch.device("cuda:0")
    H, Hkv = 8, 2
    q1, k1, v1, cq, ck = workloads.make_packed(lq, lkv, H, Hkv, d, dv, "bf16", seed=61 + d)
    q2, k2, v2, _, _ = workloads.make_packed(lq, lkv, H, Hkv, d, dv, "bf16", seed=62 + d)
    q, k, v = q1.to(dev), k1.to(dev), v1.to(dev)
    cqd, ckd = cq.to(dev), ck.to(dev)
    out = torch.empty(q.shape[0], H, dv, dtype=q.dtype, device=dev)
    s = torch.cuda.Stream()
    B = cq.numel() - 1
    # the first call on `s` grows its workspace (outside the capture)
    pva.pva_forward(q, k, v, cqd, ckd, out, B, H, Hkv, d, dv, 0.0, 1, 0.0, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pva.pva_forward(q, k, v, cqd, ckd, out, B, H, Hkv, d, dv, 0.0, 1, 0.0, stream=s)
    for (qs, ks, vs) in ((q2, k2, v2), (q1, k1, v1)):
        q.copy_(qs.to(dev)); k.copy_(ks.to(dev)); v.copy_(vs.to(dev))
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert pva.pva_get_status(s) == 0
        check(out, oracle.attention(qs, ks, vs, cq, ck, H, Hkv, 0.0, True, 0.0), "bf16")


def test_two_streams_run_independent_batches_concurrently():
    """Calls on different streams use different workspaces, so two batches
    enqueued on two streams without any ordering between them both come out
    right."""
    dev = torch.device("cuda:0")
    cases = []
    for seed, (lq, lkv) in ((71, ([300, 1, 50], [300, 700, 90])), (72, ([1] * 40, [900] * 40))):
        q, k, v, cq, ck = workloads.make_packed(lq, lkv, 8, 2, 128, 128, "bf16", seed=seed)
        out = torch.full((q.shape[0], 8, 128), float("nan"), dtype=q.dtype, device=dev)
        cases.append((q, k, v, cq, ck, out, torch.cuda.Stream()))
    torch.cuda.synchronize()
    for rep in range(3):
        for q, k, v, cq, ck, out, s in cases:
            with torch.cuda.stream(s):
                pva.pva_forward(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), out,
                                cq.numel() - 1, 8, 2, 128, 128, 0.0, 1, 0.0, stream=s)
    torch.cuda.synchronize()
    for q, k, v, cq, ck, out, s in cases:
        assert pva.pva_get_status(s) == 0
        check(out, oracle.attention(q, k, v, cq, ck, 8, 2, 0.0, True, 0.0), "bf16")
