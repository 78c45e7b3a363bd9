"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances: fp32 max-abs <= 2e-5; bf16/f16 max-abs <= 2e-2 and mean-abs
<= 2e-3, element by element on the same seeded inputs (bf16/f16 inputs are
widened exactly for the oracle).  Integer work (the scheduler's lists) is
compared bit for bit with a host mirror.
"""
import math

import numpy as np
import pytest
import torch

import gqa_attention_cu_gb300 as pva
import oracle
from gqa_attention_cu_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {"f32": (2e-5, None), "bf16": (2e-2, 2e-3), "f16": (2e-2, 2e-3)}


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    pva.build()
    pva.load_library()
    yield
    torch.cuda.synchronize()


def run_gpu(q, k, v, cq, ck, H, Hkv, scale=0.0, causal=False, softcap=0.0, out=None):
    dev = torch.device("cuda:0")
    q, k, v, cq, ck = (t.to(dev) for t in (q, k, v, cq, ck))
    d, dv = q.shape[-1], v.shape[-1]
    if out is None:
        out = torch.full((q.shape[0], H, dv), float("nan"), dtype=q.dtype, device=dev)
    pva.pva_forward(q, k, v, cq, ck, out, cq.numel() - 1, H, Hkv, d, dv, scale, int(causal),
                    softcap)
    flags = pva.pva_get_status()
    assert flags == 0, f"device status bits {flags:#x}"
    return out


def check(out, ref, dtype):
    tol_max, tol_mean = TOL[dtype]
    got = out.double().cpu().numpy().reshape(ref.shape)
    assert np.isfinite(got).all(), "non-finite outputs"
    err = np.abs(got - ref)
    assert err.max() <= tol_max, f"max-abs {err.max():.3e} > {tol_max}"
    if tol_mean is not None and err.size:
        assert err.mean() <= tol_mean, f"mean-abs {err.mean():.3e} > {tol_mean}"
    return float(err.max()) if err.size else 0.0


def parity(lq, lkv, H, Hkv, d, dtype, causal, softcap=0.0, scale=0.0, sigma=1.0, seed=0):
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, H, Hkv, d, d, dtype, sigma=sigma, seed=seed)
    out = run_gpu(q, k, v, cq, ck, H, Hkv, scale, causal, softcap)
    ref = oracle.attention(q, k, v, cq, ck, H, Hkv, scale, causal, softcap)
    return check(out, ref, dtype)


# ---------------------------------------------------------------------------
# The five workloads (small cases: full outputs against the oracle)
# ---------------------------------------------------------------------------
def test_fp32_small_workload_full():
    w = workloads.make("fp32_small")
    out = run_gpu(w["q"], w["k"], w["v"], w["cu_q"], w["cu_kv"], 4, 4, 0.125, False, 0.0)
    ref = oracle.attention(w["q"], w["k"], w["v"], w["cu_q"], w["cu_kv"], 4, 4, 0.125)
    check(out, ref, "f32")


@pytest.mark.parametrize("name,shrink", [("bf16_prefill", 4), ("bf16_chunked", 4),
                                         ("bf16_decode", 8), ("bf16_longctx", 16),
                                         ("bf16_mla", 8)])
def test_bf16_workloads_shrunk_full(name, shrink):
    w = workloads.make(name, shrink=shrink)
    out = run_gpu(w["q"], w["k"], w["v"], w["cu_q"], w["cu_kv"], w["num_heads"],
                  w["kv_num_heads"], w["scale"], w["is_causal"], w["softcap"])
    ref = oracle.attention(w["q"], w["k"], w["v"], w["cu_q"], w["cu_kv"], w["num_heads"],
                           w["kv_num_heads"], w["scale"], w["is_causal"], w["softcap"])
    check(out, ref, "bf16")


# ---------------------------------------------------------------------------
# Shapes, head groupings, dtypes, edge cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_prefill_head_sizes_and_groups(d, G):
    Hkv = 2 if G <= 8 else 1
    lq = [1, 200, 77, 3, 129]
    lkv = [1, 200, 300, 3, 129]
    parity(lq, lkv, G * Hkv, Hkv, d, "bf16", causal=True, seed=G * 7 + d)


@pytest.mark.parametrize("G", [3, 5, 6, 12])
def test_group_sizes_not_dividing_the_tile(G):
    parity([45, 130, 9], [60, 130, 9], G * 2, 2, 128, "bf16", causal=True, seed=G)


@pytest.mark.parametrize("causal", [False, True])
def test_f16(causal):
    parity([100, 37, 260], [140, 37, 260], 16, 4, 128, "f16", causal=causal, seed=5)


# Head sizes of the single-tile kernel beyond 256: 96 (loaded in 64-column
# boxes with a zero-filled tail), 192, and q.k wider than v (192/128).
@pytest.mark.parametrize("d,dv", [(96, 96), (192, 192), (192, 128)])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_prefill_extra_head_sizes(d, dv, G):
    Hkv = 2
    lq, lkv = [1, 200, 77, 3, 130], [1, 260, 300, 3, 130]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, G * Hkv, Hkv, d, dv, "bf16", seed=d + dv + G)
    out = run_gpu(q, k, v, cq, ck, G * Hkv, Hkv, 0.0, True, 0.0)
    check(out, oracle.attention(q, k, v, cq, ck, G * Hkv, Hkv, 0.0, True, 0.0), "bf16")


# Single-tile kernel edges: sequences shorter than a query tile, L_kv < L_q
# (early rows see no key and come out zero), G not dividing 128, and the
# packed tail shifting the last item's tile back.
@pytest.mark.parametrize("d,dv", [(192, 128), (96, 96)])
@pytest.mark.parametrize("G,causal", [(1, True), (3, True), (2, False), (6, True)])
def test_single_tile_kernel_edges(d, dv, G, causal):
    Hkv = 2
    lq = [5, 128, 300, 700, 129, 40, 257]
    lkv = [5, 100, 300, 900, 1, 700, 257]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, G * Hkv, Hkv, d, dv, "bf16",
                                            seed=7 * d + dv + G)
    out = run_gpu(q, k, v, cq, ck, G * Hkv, Hkv, 0.0, causal, 0.0)
    check(out, oracle.attention(q, k, v, cq, ck, G * Hkv, Hkv, 0.0, causal, 0.0), "bf16")


# Split-KV decode for every head-size pair of the tensor-core path and every
# grouping it serves (G = 16 runs as head groups over the same tiles: two of
# 8 heads at d = 64, four of 4 heads at larger head sizes; 12 or 8 compute
# warps by shape), with keys enough for several splits and the log-sum-exp
# combine.
@pytest.mark.parametrize("d,dv", [(64, 64), (96, 96), (128, 128), (192, 192), (256, 256),
                                  (192, 128)])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_split_kv_decode_every_shape_and_group(d, dv, G):
    Hkv = 2 if G < 16 else 1
    lq = [1, 1, 1, 1, 1, 1]
    lkv = [1, 37, 700, 2500, 64, 6000]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, G * Hkv, Hkv, d, dv, "bf16",
                                            seed=3 * d + dv + G)
    out = run_gpu(q, k, v, cq, ck, G * Hkv, Hkv, 0.0, True, 0.0)
    check(out, oracle.attention(q, k, v, cq, ck, G * Hkv, Hkv, 0.0, True, 0.0), "bf16")


# Shapes the split-KV kernel serves only for small batches (G = 8 and 16,
# d = 256 with G = 4, head sizes 96/192): with single-row sequences x kv
# heads >= 2 x SMs they go through the tensor-core prefill kernel instead (no
# key splits), so both routes are checked.
@pytest.mark.parametrize("d,dv,G,Hkv", [(128, 128, 16, 2), (192, 128, 4, 8), (96, 96, 8, 4),
                                        (128, 128, 8, 2), (64, 64, 8, 2), (256, 256, 8, 2),
                                        (256, 256, 4, 2)])
def test_many_single_row_sequences_take_the_prefill_route(d, dv, G, Hkv):
    B = 200
    g = torch.Generator().manual_seed(d + G)
    lkv = torch.randint(1, 700, (B,), generator=g).tolist()
    q, k, v, cq, ck = workloads.make_packed([1] * B, lkv, G * Hkv, Hkv, d, dv, "bf16", seed=G)
    words = pva.pva_schedule(cq.to("cuda:0"), ck.to("cuda:0"), B, G * Hkv, Hkv, d, dv, 1, 2)
    assert words[3] == 0 and words[1] == B  # all routed to the prefill list
    out = run_gpu(q, k, v, cq, ck, G * Hkv, Hkv, 0.0, True, 0.0)
    check(out, oracle.attention(q, k, v, cq, ck, G * Hkv, Hkv, 0.0, True, 0.0), "bf16")


@pytest.mark.parametrize("d,dv,G,dtype,softcap", [(96, 96, 16, "f16", 0.0),
                                                 (192, 128, 4, "f16", 30.0),
                                                 (128, 128, 16, "bf16", 5.0),
                                                 (192, 192, 8, "bf16", 2.0)])
def test_split_kv_decode_f16_and_softcap(d, dv, G, dtype, softcap):
    # unit-variance inputs (the bf16 tolerance is set for them); a small
    # softcap keeps the tanh far from linear
    Hkv = 2
    lq, lkv = [1, 1, 1, 40], [3000, 17, 900, 300]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, G * Hkv, Hkv, d, dv, dtype, seed=d + G)
    out = run_gpu(q, k, v, cq, ck, G * Hkv, Hkv, 0.0, True, softcap)
    check(out, oracle.attention(q, k, v, cq, ck, G * Hkv, Hkv, 0.0, True, softcap), dtype)


@pytest.mark.parametrize("d,dv,dtype,causal,softcap", [(96, 96, "f16", False, 0.0),
                                                      (192, 128, "bf16", True, 30.0),
                                                      (192, 128, "f16", False, 0.0)])
def test_prefill_extra_head_sizes_variants(d, dv, dtype, causal, softcap):
    lq, lkv = [64, 1, 129, 300], [64, 700, 200, 300]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 8, 2, d, dv, dtype, sigma=1.5, seed=7)
    out = run_gpu(q, k, v, cq, ck, 8, 2, 0.0, causal, softcap)
    check(out, oracle.attention(q, k, v, cq, ck, 8, 2, 0.0, causal, softcap), dtype)


@pytest.mark.parametrize("d,dv", [(64, 64), (32, 48), (128, 96), (8, 256), (256, 16)])
def test_fp32_head_sizes(d, dv):
    q, k, v, cq, ck = workloads.make_packed([5, 40, 33], [9, 40, 70], 6, 3, d, dv, "f32", seed=d)
    out = run_gpu(q, k, v, cq, ck, 6, 3, 0.0, True, 0.0)
    check(out, oracle.attention(q, k, v, cq, ck, 6, 3, 0.0, True), "f32")


def test_fp32_softcap_and_causal_chunks():
    q, k, v, cq, ck = workloads.make_packed([7, 64, 2], [20, 64, 90], 4, 2, 64, 64, "f32", seed=4,
                                            sigma=2.0)
    out = run_gpu(q, k, v, cq, ck, 4, 2, 0.3, True, 5.0)
    check(out, oracle.attention(q, k, v, cq, ck, 4, 2, 0.3, True, 5.0), "f32")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_empty_and_degenerate_sequences(dtype):
    """L_q = 0, L_kv = 0 (zero rows), L_q > L_kv causal (leading rows fully
    masked), single-token sequences, one-key sequences."""
    lq = [0, 4, 3, 1, 0, 130, 1, 2]
    lkv = [5, 0, 1, 1, 0, 2, 0, 200]
    d = 128 if dtype == "bf16" else 64
    parity(lq, lkv, 8, 2, d, dtype, causal=True, seed=11)
    parity(lq, lkv, 8, 2, d, dtype, causal=False, seed=12)


def test_all_sequences_empty_writes_nothing():
    """total_q = 0: an empty Q tensor (null data pointer) is accepted, nothing
    is written."""
    dev = torch.device("cuda:0")
    q = torch.zeros(0, 4, 128, dtype=torch.bfloat16, device=dev)
    assert q.data_ptr() == 0
    k = torch.randn(10, 2, 128, device=dev).to(torch.bfloat16)
    v = torch.randn(10, 2, 128, device=dev).to(torch.bfloat16)
    cq = torch.tensor([0, 0, 0], dtype=torch.int32, device=dev)
    ck = torch.tensor([0, 4, 10], dtype=torch.int32, device=dev)
    canary = torch.full((16,), 7.0, dtype=torch.bfloat16, device=dev)
    pva.pva_forward(q, k, v, cq, ck, canary, 2, 4, 2, 128, 128, 0.0, 1, 0.0)
    assert pva.pva_get_status() == 0
    assert torch.all(canary == 7.0)
    empty_out = torch.empty(0, 4, 128, dtype=torch.bfloat16, device=dev)
    pva.pva_forward(q, k, v, cq, ck, empty_out, 2, 4, 2, 128, 128, 0.0, 1, 0.0)
    assert pva.pva_get_status() == 0


def test_null_tensor_with_nonzero_extent_latches_status():
    """A null Q with cu_seqlens_q[B] > 0 is caught on the device: status bit,
    nothing computed."""
    dev = torch.device("cuda:0")
    k = torch.randn(10, 2, 128, device=dev).to(torch.bfloat16)
    cq = torch.tensor([0, 3], dtype=torch.int32, device=dev)
    ck = torch.tensor([0, 10], dtype=torch.int32, device=dev)
    out = torch.full((3, 4, 128), 5.0, dtype=torch.bfloat16, device=dev)
    lib = pva.load_library()
    rc = lib.pva_forward(None, k.data_ptr(), k.data_ptr(), cq.data_ptr(), ck.data_ptr(),
                         out.data_ptr(), 1, 4, 2, 128, 128, 0.0, 1, 0.0, 2,
                         torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert pva.pva_get_status() & pva.DEV_FLAGS["null_tensor"]
    assert torch.all(out == 5.0)


def test_single_short_batch_smaller_than_a_tile():
    """Total tokens below one tile: tiles start before row 0 (zero fill)."""
    parity([3], [5], 4, 1, 128, "bf16", causal=True, seed=21)
    parity([1], [1], 8, 8, 64, "bf16", causal=False, seed=22)


def test_long_ragged_tails_spanning_many_tiles():
    parity([1000, 513, 257], [1100, 700, 257], 8, 2, 128, "bf16", causal=True, seed=23)
    parity([1000, 513, 257], [1100, 700, 257], 8, 2, 128, "bf16", causal=False, seed=24)


def test_softcap_bf16_with_large_scores():
    parity([300, 77], [300, 150], 8, 1, 256, "bf16", causal=True, softcap=50.0,
           sigma=math.sqrt(2.0), seed=25)
    parity([90], [400], 4, 2, 128, "bf16", causal=False, softcap=5.0, scale=0.5, sigma=2.0,
           seed=26)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_running_maximum_growing_across_and_within_key_tiles(d, causal):
    """Keys grow along each sequence, most in the second half of every 128-key
    tile, so the row maximum rises by more than the rescale threshold after
    a sequence's first key tile, also between the two halves of a tile: the
    paths that rescale O in the middle of an item."""
    lq, lkv = [700, 300, 129], [700, 460, 129]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 8, 2, d, d, "bf16", seed=d + int(causal))
    kf = k.float()
    for b in range(len(lkv)):
        j = torch.arange(lkv[b], dtype=torch.float32)
        grow = 1.0 + j / 48.0 + 3.0 * ((j % 128) >= 64).float() * (j >= 128).float()
        kf[int(ck[b]):int(ck[b + 1])] *= grow[:, None, None]
    k = kf.to(torch.bfloat16)
    # the softmax is sharply peaked here (outputs near single V rows): V at
    # half scale keeps the outputs within the magnitudes the bf16 bound is for
    v = (v.float() * 0.5).to(torch.bfloat16)
    out = run_gpu(q, k, v, cq, ck, 8, 2, 0.0, causal, 0.0)
    check(out, oracle.attention(q, k, v, cq, ck, 8, 2, 0.0, causal, 0.0), "bf16")


# A negative scale flips the direction of the score transform: every kernel
# takes the row's extreme from the other side (the paired kernel by template,
# the single-tile kernel's one-pass and two-pass paths by the sign, the
# decode kernel through its running maximum).  Prefill and single-row
# sequences, with and without a softcap.
@pytest.mark.parametrize("d,dv", [(128, 128), (64, 64), (256, 256), (192, 128)])
@pytest.mark.parametrize("softcap", [0.0, 20.0])
def test_negative_scale_every_kernel(d, dv, softcap):
    lq, lkv = [200, 1, 77, 1, 300], [260, 900, 77, 40, 300]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 8, 2, d, dv, "bf16", seed=9 * d + dv)
    out = run_gpu(q, k, v, cq, ck, 8, 2, -0.07, True, softcap)
    check(out, oracle.attention(q, k, v, cq, ck, 8, 2, -0.07, True, softcap), "bf16")


def test_explicit_scale():
    parity([64, 10], [64, 90], 4, 4, 64, "bf16", causal=False, scale=0.05, seed=27)


# ---------------------------------------------------------------------------
# Invariants on the GPU path
# ---------------------------------------------------------------------------
def _case(seed=31, dtype="bf16"):
    lq, lkv = [50, 1, 200, 7, 1], [120, 700, 200, 7, 33]
    return workloads.make_packed(lq, lkv, 8, 2, 128, 128, dtype, seed=seed), lq, lkv


def test_rerun_is_bitwise_deterministic():
    (q, k, v, cq, ck), _, _ = _case()
    a = run_gpu(q, k, v, cq, ck, 8, 2, causal=True)
    for _ in range(3):
        b = run_gpu(q, k, v, cq, ck, 8, 2, causal=True)
        assert torch.equal(a, b)


def test_softcap_sign_gives_identical_bits():
    (q, k, v, cq, ck), _, _ = _case()
    a = run_gpu(q, k, v, cq, ck, 8, 2, causal=True, softcap=20.0)
    b = run_gpu(q, k, v, cq, ck, 8, 2, causal=True, softcap=-20.0)
    assert torch.equal(a, b)


def test_decode_causal_equals_noncausal_bitwise():
    q, k, v, cq, ck = workloads.make_packed([1] * 6, [5, 900, 4000, 1, 64, 300], 32, 8, 128, 128,
                                            "bf16", seed=32)
    a = run_gpu(q, k, v, cq, ck, 32, 8, causal=True)
    b = run_gpu(q, k, v, cq, ck, 32, 8, causal=False)
    assert torch.equal(a, b)
    check(a, oracle.attention(q, k, v, cq, ck, 32, 8, 0.0, True), "bf16")


def test_batch_permutation_permutes_outputs_bitwise():
    (q, k, v, cq, ck), lq, lkv = _case()
    out = run_gpu(q, k, v, cq, ck, 8, 2, causal=True).cpu()
    order = [3, 0, 4, 2, 1]
    q2 = torch.cat([q[int(cq[b]):int(cq[b + 1])] for b in order])
    k2 = torch.cat([k[int(ck[b]):int(ck[b + 1])] for b in order])
    v2 = torch.cat([v[int(ck[b]):int(ck[b + 1])] for b in order])
    out2 = run_gpu(q2, k2, v2, workloads.cu_from_lengths([lq[b] for b in order]),
                   workloads.cu_from_lengths([lkv[b] for b in order]), 8, 2, causal=True).cpu()
    expect = torch.cat([out[int(cq[b]):int(cq[b + 1])] for b in order])
    assert torch.equal(out2, expect)


def test_perturbing_one_sequence_leaves_others_bitwise_unchanged():
    (q, k, v, cq, ck), lq, lkv = _case()
    out = run_gpu(q, k, v, cq, ck, 8, 2, causal=True).cpu()
    b0 = 2
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[int(cq[b0]):int(cq[b0 + 1])] *= -1
    k2[int(ck[b0]):int(ck[b0 + 1])] += 1
    v2[int(ck[b0]):int(ck[b0 + 1])] *= 3
    out2 = run_gpu(q2, k2, v2, cq, ck, 8, 2, causal=True).cpu()
    for b in range(len(lq)):
        if b == b0:
            continue
        sl = slice(int(cq[b]), int(cq[b + 1]))
        assert torch.equal(out[sl], out2[sl])


def test_constant_value_rows_and_first_causal_row():
    lq = lkv = [300, 5, 64]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 4, 2, 128, 128, "bf16", seed=33)
    r = torch.linspace(-2, 2, 128).to(torch.bfloat16)
    vc = r.view(1, 1, -1).expand_as(v).contiguous()
    out = run_gpu(q, k, vc, cq, ck, 4, 2, causal=True).float().cpu()
    assert torch.allclose(out, r.float().view(1, 1, -1).expand_as(out), atol=2e-2)
    out = run_gpu(q, k, v, cq, ck, 4, 2, causal=True).cpu()
    for b in range(3):
        first = out[int(cq[b])]
        vrow = v[int(ck[b])].repeat_interleave(2, dim=0)
        assert torch.allclose(first.float(), vrow.float(), atol=1e-2)


def test_canaries_outside_the_packed_ranges_are_never_read_or_written():
    """NaN after cu[B] in Q/K/V must not leak in; guard bands around out stay
    untouched."""
    lq, lkv = [70, 3, 200], [90, 3, 260]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 8, 2, 128, 128, "bf16", seed=34)
    pad = 300
    nan = float("nan")
    qp = torch.cat([q, torch.full((pad,) + q.shape[1:], nan, dtype=q.dtype)])
    kp = torch.cat([k, torch.full((pad,) + k.shape[1:], nan, dtype=k.dtype)])
    vp = torch.cat([v, torch.full((pad,) + v.shape[1:], nan, dtype=v.dtype)])
    dev = torch.device("cuda:0")
    n_out = q.shape[0] * 8 * 128
    guard = 4096
    buf = torch.full((n_out + 2 * guard,), 3.0, dtype=torch.bfloat16, device=dev)
    out = buf[guard:guard + n_out].view(q.shape[0], 8, 128)
    for causal in (True, False):
        run_gpu(qp, kp, vp, cq, ck, 8, 2, causal=causal, out=out)
        assert torch.all(buf[:guard] == 3.0) and torch.all(buf[guard + n_out:] == 3.0)
        check(out, oracle.attention(q, k, v, cq, ck, 8, 2, 0.0, causal), "bf16")


@pytest.mark.parametrize("bad", ["q_start", "kv_start", "q_order", "kv_order"])
def test_malformed_offsets_latch_status_and_write_nothing(bad):
    dev = torch.device("cuda:0")
    q, k, v, cq, ck = workloads.make_packed([10, 20], [10, 20], 4, 2, 128, 128, "bf16", seed=35)
    cq, ck = cq.clone(), ck.clone()
    if bad == "q_start":
        cq[0] = 1
    elif bad == "kv_start":
        ck[0] = 2
    elif bad == "q_order":
        cq[1] = 35   # [0, 35, 30]: decreases
    else:
        ck[1] = 35
    out = torch.full((30, 4, 128), 5.0, dtype=torch.bfloat16, device=dev)
    pva.pva_forward(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), out, 2, 4, 2, 128,
                    128, 0.0, 1, 0.0)
    flags = pva.pva_get_status()
    expect = {"q_start": 0x1, "kv_start": 0x2, "q_order": 0x4, "kv_order": 0x8}[bad]
    assert flags & expect
    assert torch.all(out == 5.0)
    assert pva.pva_get_status() == 0  # cleared on read


# ---------------------------------------------------------------------------
# Scheduler: bit-exact against a host mirror
# ---------------------------------------------------------------------------
def sched_mirror(lq, lkv, H, Hkv, d, dtype, num_sms, dv=None):
    B = len(lq)
    dv = d if dv is None else dv
    if dtype == 0:
        tile, units, dec = 16, H, False
    else:
        G = H // Hkv
        paired = d == dv and d in (64, 128)
        tile, units = (128 // G) * (2 if paired else 1), Hkv
        dec = G in (1, 2, 4, 8, 16)
        tuned = d == dv and ((d in (64, 128) and G <= 4) or (d == 256 and G <= 2))
        if dec and not tuned:  # adaptive: only when too few to fill the SMs
            dec = sum(1 for a in lq if a == 1) * Hkv < 2 * num_sms
    cap = min(B * Hkv * 16, 16384)
    INT_MAX = 2 ** 31 - 1
    chunk = INT_MAX
    if dec:
        keyrows = sum(b for a, b in zip(lq, lkv) if a == 1) * Hkv
        target = num_sms * 2
        chunk = -(-keyrows // target)
        chunk = -(-chunk // 64) * 64
        chunk = max(chunk, 256)

        def splits(L, c):
            return 1 if L <= c else min(-(-L // c), 16)
        for _ in range(40):
            sp = [splits(b, chunk) for a, b in zip(lq, lkv) if a == 1]
            units_tot = sum(sp) * Hkv
            if not any(s > 1 for s in sp) or units_tot <= cap:
                break
            chunk *= 2
        chunk = min(chunk, INT_MAX)
    else:
        def splits(L, c):
            return 1

    def is_dec(b):
        return dec and lq[b] == 1
    pref = [b for b in range(B) if lq[b] > 0 and not is_dec(b)]
    decs = [b for b in range(B) if lq[b] > 0 and is_dec(b)]
    if B <= 16384:
        pref.sort(key=lambda b: (-lkv[b], b))
        decs.sort(key=lambda b: (-lkv[b], b))

    def prefix(lst, work):
        out, run = [], 0
        for b in lst:
            out.append(run)
            run += work(b)
        out += [run] * (B + 1 - len(lst))
        return out, run
    pp, n_items = prefix(pref, lambda b: -(-lq[b] // tile) * units)
    dp, n_units = prefix(decs, lambda b: splits(lkv[b], chunk) * Hkv)
    hdr = [0, len(pref), n_items, len(decs), n_units, tile, units, chunk if dec else INT_MAX]
    return (hdr + pref + [-1] * (B - len(pref)) + pp + decs + [-1] * (B - len(decs)) + dp)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("cfg", [(32, 8, 128, 128, 2), (8, 1, 256, 256, 2), (6, 2, 64, 64, 1),
                                 (4, 4, 64, 64, 0), (64, 2, 128, 128, 2), (16, 4, 192, 128, 2),
                                 (8, 2, 96, 96, 1), (32, 2, 128, 128, 2), (16, 1, 64, 64, 1)])
def test_scheduler_matches_host_mirror(seed, cfg):
    H, Hkv, d, dv, dtype = cfg
    g = torch.Generator().manual_seed(seed)
    B = int(torch.randint(1, 300, (1,), generator=g))
    lq = torch.randint(0, 600, (B,), generator=g)
    lq = torch.where(torch.rand(B, generator=g) < 0.4, torch.ones_like(lq), lq).tolist()
    lkv = (torch.tensor(lq) + torch.randint(0, 9000, (B,), generator=g)).tolist()
    dev = torch.device("cuda:0")
    words = pva.pva_schedule(workloads.cu_from_lengths(lq).to(dev),
                             workloads.cu_from_lengths(lkv).to(dev), B, H, Hkv, d, dv, 1, dtype)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert words == sched_mirror(lq, lkv, H, Hkv, d, dtype, sms, dv)


@pytest.mark.parametrize("B", [1, 2, 7, 31, 32, 33])
@pytest.mark.parametrize("cfg", [(32, 8, 128, 128, 2), (8, 1, 256, 256, 2), (4, 4, 64, 64, 0),
                                 (16, 4, 192, 128, 2), (32, 2, 128, 128, 2)])
def test_scheduler_small_batches_match_host_mirror(B, cfg):
    """B <= 32 runs the one-warp scheduler (33 the CTA one): same words."""
    H, Hkv, d, dv, dtype = cfg
    g = torch.Generator().manual_seed(B)
    lq = torch.randint(0, 400, (B,), generator=g)
    r = torch.rand(B, generator=g)
    lq = torch.where(r < 0.35, torch.ones_like(lq), torch.where(r > 0.9, torch.zeros_like(lq), lq))
    lq = lq.tolist()
    lkv = (torch.tensor(lq) + torch.randint(0, 20000, (B,), generator=g)).tolist()
    dev = torch.device("cuda:0")
    words = pva.pva_schedule(workloads.cu_from_lengths(lq).to(dev),
                             workloads.cu_from_lengths(lkv).to(dev), B, H, Hkv, d, dv, 1, dtype)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert words == sched_mirror(lq, lkv, H, Hkv, d, dtype, sms, dv)


@pytest.mark.parametrize("B", [33, 128, 129, 300, 512, 513, 1000])
def test_scheduler_ties_in_key_length_match_host_mirror(B):
    """Many sequences share an L_kv, so the order among them rests on the
    index tie-break alone: the rank sort (B <= 512) and the bitonic network
    above it must both put equal lengths in index order."""
    g = torch.Generator().manual_seed(1000 + B)
    lq = torch.randint(0, 300, (B,), generator=g)
    lq = torch.where(torch.rand(B, generator=g) < 0.5, torch.ones_like(lq), lq)
    # key lengths from only five values (decode rows) or lq + one of five pasts
    lkv = torch.where(lq == 1, 1 + 1000 * torch.randint(1, 6, (B,), generator=g),
                      lq + 512 * torch.randint(0, 5, (B,), generator=g))
    lq, lkv = lq.tolist(), lkv.tolist()
    dev = torch.device("cuda:0")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for H, Hkv, d, dv in ((32, 8, 128, 128), (64, 4, 64, 64)):
        words = pva.pva_schedule(workloads.cu_from_lengths(lq).to(dev),
                                 workloads.cu_from_lengths(lkv).to(dev), B, H, Hkv, d, dv, 1, 2)
        assert words == sched_mirror(lq, lkv, H, Hkv, d, 2, sms, dv)


@pytest.mark.parametrize("B", [2048, 2049, 4096, 9000, 16384, 16385])
def test_scheduler_large_batches_match_host_mirror(B):
    """Up to 16384 sequences are sorted longest first on the device (shared
    memory sized by B); beyond that they keep their input order."""
    g = torch.Generator().manual_seed(B)
    lq = torch.randint(0, 64, (B,), generator=g)
    lq = torch.where(torch.rand(B, generator=g) < 0.5, torch.ones_like(lq), lq).tolist()
    lkv = (torch.tensor(lq) + torch.randint(0, 3000, (B,), generator=g)).tolist()
    dev = torch.device("cuda:0")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for H, Hkv, d, dv in ((32, 8, 128, 128), (16, 2, 192, 128)):
        words = pva.pva_schedule(workloads.cu_from_lengths(lq).to(dev),
                                 workloads.cu_from_lengths(lkv).to(dev), B, H, Hkv, d, dv, 1, 2)
        assert words == sched_mirror(lq, lkv, H, Hkv, d, 2, sms, dv)


def test_scheduler_configs_match_host_mirror():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    dev = torch.device("cuda:0")
    for name, w in workloads.WORKLOADS.items():
        lq, lkv = workloads.draw_lengths(w, torch.Generator().manual_seed(0))
        dt = workloads.DTYPE_CODE[w.dtype]
        words = pva.pva_schedule(workloads.cu_from_lengths(lq).to(dev),
                                 workloads.cu_from_lengths(lkv).to(dev), len(lq), w.num_heads,
                                 w.kv_num_heads, w.head_size, w.v_head_size, int(w.is_causal), dt)
        assert words == sched_mirror(lq, lkv, w.num_heads, w.kv_num_heads, w.head_size, dt,
                                     sms, w.v_head_size), name


# ---------------------------------------------------------------------------
# Full-size workloads, as the benchmark runs them: sampled sequences/rows
# ---------------------------------------------------------------------------
def _sub_batch(w, seqs):
    """Packed sub-batch holding only sequences `seqs` (CPU)."""
    cq, ck = w["cu_q"].cpu(), w["cu_kv"].cpu()
    qs = [w["q"][int(cq[b]):int(cq[b + 1])].cpu() for b in seqs]
    ks = [w["k"][int(ck[b]):int(ck[b + 1])].cpu() for b in seqs]
    vs = [w["v"][int(ck[b]):int(ck[b + 1])].cpu() for b in seqs]
    return (torch.cat(qs), torch.cat(ks), torch.cat(vs),
            workloads.cu_from_lengths([w["lq"][b] for b in seqs]),
            workloads.cu_from_lengths([w["lkv"][b] for b in seqs]))


@pytest.mark.parametrize("name", ["bf16_prefill", "bf16_chunked", "bf16_decode", "bf16_longctx",
                                  "bf16_mla"])
def test_full_size_workload_sampled_rows(name):
    w = workloads.make(name, device="cuda:0")
    H, Hkv, dv = w["num_heads"], w["kv_num_heads"], w["v_head_size"]
    out = torch.empty(w["q"].shape[0], H, dv, dtype=w["q"].dtype, device="cuda:0")
    pva.pva_forward(w["q"], w["k"], w["v"], w["cu_q"], w["cu_kv"], out, w["B"], H, Hkv,
                    w["head_size"], dv, w["scale"], int(w["is_causal"]), w["softcap"])
    assert pva.pva_get_status() == 0
    # sequences: the longest, the shortest, and two more at fixed positions
    order = sorted(range(w["B"]), key=lambda b: w["lkv"][b])
    seqs = sorted({order[0], order[-1], order[len(order) // 3], order[2 * len(order) // 3]})
    q, k, v, cq, ck = _sub_batch(w, seqs)
    g = np.random.default_rng(1)
    rows = []
    for j, b in enumerate(seqs):
        L = w["lq"][b]
        cand = np.unique(np.concatenate([np.arange(min(L, 64)), np.arange(max(0, L - 64), L),
                                         g.integers(0, L, size=min(L, 256))]))
        if name == "bf16_longctx":
            cand = np.unique(np.concatenate([np.arange(min(L, 16)), np.arange(max(0, L - 16), L),
                                             g.integers(0, L, size=48)]))
        for i in cand:
            for hh in range(H):
                rows.append((int(cq[j]) + int(i)) * H + hh)
    rows = np.array(rows, dtype=np.int64)
    ref = oracle.attention_rows(q, k, v, cq, ck, rows, H, Hkv, w["scale"], w["is_causal"],
                                w["softcap"])
    # the same rows from the GPU output
    cqf = w["cu_q"].cpu()
    full_index = []
    for r in rows:
        tok_sub, hh = divmod(int(r), H)
        j = int(np.searchsorted(cq.numpy(), tok_sub, side="right") - 1)
        b = seqs[j]
        tok = int(cqf[b]) + tok_sub - int(cq[j])
        full_index.append(tok * H + hh)
    got = out.view(-1, dv)[torch.tensor(full_index, device="cuda:0")]
    check(got, ref, "bf16")


# ---------------------------------------------------------------------------
# Failure detection: a bounded wait that nothing satisfies
# ---------------------------------------------------------------------------
def test_bounded_wait_gives_up_with_status_and_context_survives():
    """The wait helper every pipeline barrier uses gives up after its limit,
    latches the timeout bit and returns; the context stays usable."""
    t0 = torch.cuda.Event(enable_timing=True)
    flags = pva.pva_selftest_wait(20000)  # 20 ms
    assert flags & pva.DEV_FLAGS["wait_timeout"]
    # the device still computes correctly afterwards
    parity([33, 5], [40, 5], 8, 2, 128, "bf16", causal=True, seed=41)
    assert pva.pva_get_status() == 0
    del t0


def test_negative_scale_fp32():
    parity([33, 1, 70], [40, 90, 70], 4, 2, 64, "f32", causal=True, scale=-0.2, seed=57)
