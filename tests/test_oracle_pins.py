"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test checks the oracle against something the pages or the mathematics
fix independently of its loop nest:

* library routines: torch float64 ``scaled_dot_product_attention`` on padded
  batches (its own causal mask, scale and GQA head mapping);
* the padded/packed equivalences the pages state (packed_varlen_attention.rs,
  module doc "Relationship to ONNX Attention-24 nonpad_kv_seqlen"; the padded
  op's per-batch offsets in standard_attention.rs, `execute`, "Per-batch causal
  offset and padding frontier");
* tail alignment as the suffix of ordinary causal self-attention
  (packed_varlen_attention.rs, "Causal alignment");
* closed forms, invariants and hand-derived worked examples
  (``tests/golden/worked_examples.json``).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from gqa_attention_cu_gb300 import workloads

pytestmark = pytest.mark.filterwarnings("ignore")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _rand_case(seed, B, lmax, H, Hkv, d, dv, chunked=False):
    g = torch.Generator().manual_seed(seed)
    lq = torch.randint(0, lmax + 1, (B,), generator=g).tolist()
    if chunked:
        lkv = [a + int(torch.randint(0, lmax + 1, (1,), generator=g)) for a in lq]
    else:
        lkv = torch.randint(0, lmax + 1, (B,), generator=g).tolist()
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, H, Hkv, d, dv, "f32", gen=g)
    return q.double(), k.double(), v.double(), cq, ck, lq, lkv


def _sdpa_seq(q, k, v, scale, mask):
    """torch float64 SDPA for one sequence: q [Lq,H,d], k/v [Lkv,Hkv,*],
    boolean mask [Lq,Lkv] (True = visible) or None.  Rows with no visible key
    come back as NaN from torch; the caller handles them."""
    qq = q.permute(1, 0, 2).unsqueeze(0)
    kk = k.permute(1, 0, 2).unsqueeze(0)
    vv = v.permute(1, 0, 2).unsqueeze(0)
    out = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale,
                                         enable_gqa=True)
    return out.squeeze(0).permute(1, 0, 2)


# ---------------------------------------------------------------------------
# Worked examples (exact fractions derived by hand)
# ---------------------------------------------------------------------------
def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_worked_examples(case):
    q = np.array(case["q"], dtype=np.float64)
    k = np.array(case["k"], dtype=np.float64)
    v = np.array(case["v"], dtype=np.float64)
    out = oracle.attention(q, k, v, case["cu_q"], case["cu_kv"], case["H"], case["Hkv"],
                           scale=case["scale"], is_causal=bool(case["is_causal"]),
                           softcap=case["softcap"])
    exp = np.array(case["expected"], dtype=np.float64)
    exp = exp[..., 0] / exp[..., 1]
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-12)


def test_softcap_sign_symmetry_exact():
    """c*tanh(s/c) is even in c: softcap -c and +c agree bit for bit."""
    q, k, v, cq, ck, _, _ = _rand_case(3, 3, 9, 4, 2, 8, 8)
    a = oracle.attention(q, k, v, cq, ck, 4, 2, scale=0.7, softcap=1.5, is_causal=True)
    b = oracle.attention(q, k, v, cq, ck, 4, 2, scale=0.7, softcap=-1.5, is_causal=True)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# Library routine: torch float64 SDPA
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("H,Hkv", [(1, 1), (4, 4), (4, 2), (6, 1)])
def test_padded_equal_lengths_match_sdpa(seed, H, Hkv):
    """All L_q == L_kv == L: packed output equals padded SDPA (its own causal
    mask, GQA head map and scale)."""
    g = torch.Generator().manual_seed(100 + seed)
    B, L, d, dv = 3, int(torch.randint(1, 9, (1,), generator=g)), 8, 5
    causal = bool(seed % 2)
    scale = 0.0 if seed % 3 == 0 else 0.3 + 0.1 * seed
    q, k, v, cq, ck = workloads.make_packed([L] * B, [L] * B, H, Hkv, d, dv, "f32", gen=g)
    q, k, v = q.double(), k.double(), v.double()
    out = oracle.attention(q, k, v, cq, ck, H, Hkv, scale=scale, is_causal=causal)
    qq = q.view(B, L, H, d).permute(0, 2, 1, 3)
    kk = k.view(B, L, Hkv, d).permute(0, 2, 1, 3)
    vv = v.view(B, L, Hkv, dv).permute(0, 2, 1, 3)
    # the default scale is 1/sqrt(d) rounded to float32 (the page computes it
    # in f32); SDPA receives that same value
    ref = F.scaled_dot_product_attention(qq, kk, vv, is_causal=causal,
                                         scale=oracle.resolve_scale(scale, d), enable_gqa=True)
    ref = ref.permute(0, 2, 1, 3).reshape(B * L, H, dv).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(8))
def test_tail_aligned_is_suffix_of_self_attention(seed):
    """A chunk of L_q queries against L_kv = past + L_q keys, causal, gives the
    last L_q rows of ordinary causal self-attention over all L_kv tokens."""
    g = torch.Generator().manual_seed(200 + seed)
    B, H, Hkv, d, dv = 2, 4, 2, 8, 8
    lkv = torch.randint(1, 12, (B,), generator=g).tolist()
    lq = [int(torch.randint(1, L + 1, (1,), generator=g)) for L in lkv]
    full_q, k, v, _, ck = workloads.make_packed(lkv, lkv, H, Hkv, d, dv, "f32", gen=g)
    full_q, k, v = full_q.double(), k.double(), v.double()
    qs, pos = [], 0
    for a, L in zip(lq, lkv):
        qs.append(full_q[pos + L - a: pos + L])
        pos += L
    q = torch.cat(qs)
    cq = workloads.cu_from_lengths(lq)
    out = oracle.attention(q, k, v, cq, ck, H, Hkv, scale=0.0, is_causal=True)
    pos_q = pos_kv = 0
    for a, L in zip(lq, lkv):
        ref = _sdpa_seq(full_q[pos_kv:pos_kv + L], k[pos_kv:pos_kv + L], v[pos_kv:pos_kv + L],
                        oracle.resolve_scale(0.0, d), torch.ones(L, L, dtype=torch.bool).tril())
        np.testing.assert_allclose(out[pos_q:pos_q + a], ref[L - a:].numpy(), rtol=0, atol=1e-12)
        pos_q += a
        pos_kv += L


@pytest.mark.parametrize("seed", range(6))
def test_nonpad_kv_seqlen_prefix_sum_reproduces_padded_masking(seed):
    """The padded op with nonpad_kv_seqlen (pad frontier j >= nonpad[b],
    causal offset nonpad[b] - q_seq) equals the packed op fed
    cu_seqlens_kv = exclusive prefix sum of nonpad and cu_seqlens_q of equal
    q_seq lengths."""
    g = torch.Generator().manual_seed(300 + seed)
    B, H, Hkv, d, dv = 3, 4, 2, 8, 6
    q_seq = int(torch.randint(1, 6, (1,), generator=g))
    nonpad = torch.randint(0, 10, (B,), generator=g).tolist()
    cap = max(max(nonpad), 1)
    causal = bool(seed % 2)
    qp = torch.randn(B, q_seq, H, d, generator=g, dtype=torch.float64)
    kp = torch.randn(B, cap, Hkv, d, generator=g, dtype=torch.float64)
    vp = torch.randn(B, cap, Hkv, dv, generator=g, dtype=torch.float64)
    # padded reference: explicit mask with the padded op's two frontiers
    ref = torch.zeros(B, q_seq, H, dv, dtype=torch.float64)
    visible_any = torch.zeros(B, q_seq, dtype=torch.bool)
    for b in range(B):
        i = torch.arange(q_seq).view(-1, 1)
        j = torch.arange(cap).view(1, -1)
        mask = j < nonpad[b]
        if causal:
            mask = mask & (j <= i + (nonpad[b] - q_seq))
        visible_any[b] = mask.any(dim=1)
        r = _sdpa_seq(qp[b], kp[b], vp[b], oracle.resolve_scale(0.0, d), mask)
        ref[b] = torch.nan_to_num(r, nan=0.0)
    # packed run
    q = qp.reshape(B * q_seq, H, d)
    k = torch.cat([kp[b, :nonpad[b]] for b in range(B)])
    v = torch.cat([vp[b, :nonpad[b]] for b in range(B)])
    cq = workloads.cu_from_lengths([q_seq] * B)
    ck = workloads.cu_from_lengths(nonpad)
    out = oracle.attention(q, k, v, cq, ck, H, Hkv, is_causal=causal).reshape(B, q_seq, H, dv)
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)
    # rows the padded op fully masks are zero in the packed op
    assert np.all(out[~visible_any.numpy()] == 0.0)


@pytest.mark.parametrize("seed", range(10))
def test_bruteforce_tiny_random_against_sdpa(seed):
    """Tiny random batches (B<=3, L<=8, d<=8, mixed L_q != L_kv, GQA, softcap
    off) against per-sequence torch SDPA with the suffix-of-self-attention mask
    built as a lower-triangular band over the last L_q rows."""
    g = torch.Generator().manual_seed(400 + seed)
    H, Hkv = [(2, 1), (4, 2), (3, 3), (4, 4)][seed % 4]
    d = int(torch.randint(1, 9, (1,), generator=g))
    dv = int(torch.randint(1, 9, (1,), generator=g))
    q, k, v, cq, ck, lq, lkv = _rand_case(500 + seed, 3, 8, H, Hkv, d, dv, chunked=True)
    causal = seed % 2 == 0
    out = oracle.attention(q, k, v, cq, ck, H, Hkv, scale=0.0, is_causal=causal)
    for b in range(len(lq)):
        a, L = lq[b], lkv[b]
        qs = q[int(cq[b]):int(cq[b + 1])]
        ks = k[int(ck[b]):int(ck[b + 1])]
        vs = v[int(ck[b]):int(ck[b + 1])]
        if a == 0:
            continue
        if L == 0:
            assert np.all(out[int(cq[b]):int(cq[b + 1])] == 0)
            continue
        mask = torch.ones(L, L, dtype=torch.bool).tril()[L - a:] if causal else None
        ref = _sdpa_seq(qs, ks, vs, oracle.resolve_scale(0.0, d), mask)
        np.testing.assert_allclose(out[int(cq[b]):int(cq[b + 1])], ref.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------
def test_constant_value_rows_return_that_row():
    q, k, v, cq, ck, lq, lkv = _rand_case(7, 4, 10, 4, 2, 8, 6)
    r = torch.tensor([1.5, -2.0, 0.25, 3.0, -0.5, 7.0], dtype=torch.float64)
    v = r.view(1, 1, -1).expand(v.shape[0], 2, -1).contiguous()
    out = oracle.attention(q, k, v, cq, ck, 4, 2, is_causal=False)
    for b in range(len(lq)):
        rows = out[int(cq[b]):int(cq[b + 1])]
        if lkv[b] == 0:
            assert np.all(rows == 0)
        else:
            np.testing.assert_allclose(rows, np.broadcast_to(r.numpy(), rows.shape), atol=1e-12)


def test_first_causal_row_is_v0_and_single_key_is_that_row():
    g = torch.Generator().manual_seed(11)
    lq = lkv = [5, 1, 9]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 2, 1, 8, 4, "f32", gen=g)
    q, k, v = q.double(), k.double(), v.double()
    out = oracle.attention(q, k, v, cq, ck, 2, 1, is_causal=True)
    for b in range(3):
        np.testing.assert_array_equal(out[int(cq[b])], v[int(ck[b])].expand(2, -1).numpy())
    # L_kv == 1, non-causal: every query returns that V row
    lq2, lkv2 = [3, 2], [1, 1]
    q2, k2, v2, cq2, ck2 = workloads.make_packed(lq2, lkv2, 2, 2, 4, 3, "f32", gen=g)
    out2 = oracle.attention(q2.double(), k2.double(), v2.double(), cq2, ck2, 2, 2)
    for b in range(2):
        for t in range(int(cq2[b]), int(cq2[b + 1])):
            np.testing.assert_array_equal(out2[t], v2[int(ck2[b])].double().numpy())


def test_zero_query_gives_mean_of_visible_values():
    g = torch.Generator().manual_seed(12)
    lq, lkv = [3, 4], [6, 4]
    _, k, v, cq, ck = workloads.make_packed(lq, lkv, 2, 2, 8, 5, "f32", gen=g)
    k, v = k.double(), v.double()
    q = torch.zeros(7, 2, 8, dtype=torch.float64)
    out = oracle.attention(q, k, v, cq, ck, 2, 2, is_causal=True)
    for b in range(2):
        off = lkv[b] - lq[b]
        for i in range(lq[b]):
            hi = min(lkv[b], i + off + 1)
            vis = v[int(ck[b]):int(ck[b]) + hi]
            np.testing.assert_allclose(out[int(cq[b]) + i], vis.mean(dim=0).numpy(), atol=1e-12)


def test_empty_sequences_and_fully_masked_rows_are_zero():
    g = torch.Generator().manual_seed(13)
    lq, lkv = [0, 4, 3, 2], [5, 0, 1, 2]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, 2, 1, 4, 4, "f32", gen=g)
    out = oracle.attention(q, k, v, cq, ck, 2, 1, is_causal=True)
    # seq1: L_kv = 0 -> zeros; seq2: offset -2 -> rows 0,1 masked, row 2 = v
    assert np.all(out[0:4] == 0)
    assert np.all(out[4:6] == 0)
    np.testing.assert_array_equal(out[6], v[5].double().expand(2, -1).numpy())


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------
def test_gqa_equals_mha_with_repeated_kv_heads():
    q, k, v, cq, ck, _, _ = _rand_case(21, 3, 9, 8, 2, 8, 8, chunked=True)
    a = oracle.attention(q, k, v, cq, ck, 8, 2, is_causal=True, softcap=3.0)
    b = oracle.attention(q, k.repeat_interleave(4, dim=1), v.repeat_interleave(4, dim=1), cq, ck,
                         8, 8, is_causal=True, softcap=3.0)
    assert np.array_equal(a, b)


def test_key_permutation_invariance_noncausal():
    q, k, v, cq, ck, lq, lkv = _rand_case(22, 3, 9, 4, 2, 8, 8)
    a = oracle.attention(q, k, v, cq, ck, 4, 2)
    g = torch.Generator().manual_seed(5)
    perm = []
    for b in range(len(lkv)):
        perm.append(int(ck[b]) + torch.randperm(lkv[b], generator=g))
    perm = torch.cat(perm) if perm else torch.zeros(0, dtype=torch.long)
    b_ = oracle.attention(q, k[perm], v[perm], cq, ck, 4, 2)
    np.testing.assert_allclose(a, b_, rtol=0, atol=1e-12)


def test_batch_permutation_permutes_outputs_exactly():
    q, k, v, cq, ck, lq, lkv = _rand_case(23, 4, 9, 4, 1, 8, 8, chunked=True)
    out = oracle.attention(q, k, v, cq, ck, 4, 1, is_causal=True)
    order = [2, 0, 3, 1]
    q2 = torch.cat([q[int(cq[b]):int(cq[b + 1])] for b in order])
    k2 = torch.cat([k[int(ck[b]):int(ck[b + 1])] for b in order])
    v2 = torch.cat([v[int(ck[b]):int(ck[b + 1])] for b in order])
    cq2 = workloads.cu_from_lengths([lq[b] for b in order])
    ck2 = workloads.cu_from_lengths([lkv[b] for b in order])
    out2 = oracle.attention(q2, k2, v2, cq2, ck2, 4, 1, is_causal=True)
    expect = np.concatenate([out[int(cq[b]):int(cq[b + 1])] for b in order])
    assert np.array_equal(out2, expect)


def test_perturbing_one_sequence_leaves_the_others_unchanged():
    q, k, v, cq, ck, lq, lkv = _rand_case(24, 4, 9, 4, 2, 8, 8, chunked=True)
    out = oracle.attention(q, k, v, cq, ck, 4, 2, is_causal=True)
    b0 = 1
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[int(cq[b0]):int(cq[b0 + 1])] += 1.0
    k2[int(ck[b0]):int(ck[b0 + 1])] *= -2.0
    v2[int(ck[b0]):int(ck[b0 + 1])] += 3.0
    out2 = oracle.attention(q2, k2, v2, cq, ck, 4, 2, is_causal=True)
    for b in range(4):
        sl = slice(int(cq[b]), int(cq[b + 1]))
        if b == b0:
            continue
        assert np.array_equal(out[sl], out2[sl])


def test_decode_causal_equals_noncausal():
    """L_q = 1: the tail-aligned frontier is L_kv - 1, so every key is visible."""
    q, k, v, cq, ck = workloads.make_packed([1, 1, 1], [4, 9, 1], 4, 2, 8, 8, "f32", seed=3)
    a = oracle.attention(q, k, v, cq, ck, 4, 2, is_causal=True)
    b = oracle.attention(q, k, v, cq, ck, 4, 2, is_causal=False)
    assert np.array_equal(a, b)


def test_softcap_limits():
    q, k, v, cq, ck, lq, lkv = _rand_case(25, 3, 9, 2, 2, 8, 8)
    q = q * 30.0
    plain = oracle.attention(q, k, v, cq, ck, 2, 2)
    # a cap far above every score is (numerically) no cap
    huge = oracle.attention(q, k, v, cq, ck, 2, 2, softcap=1e7)
    np.testing.assert_allclose(huge, plain, rtol=0, atol=1e-6)
    # a tiny cap squeezes all scores into [-c, c]: output -> mean of V rows
    tiny = oracle.attention(q, k, v, cq, ck, 2, 2, softcap=1e-9)
    for b in range(len(lq)):
        if lq[b] == 0 or lkv[b] == 0:
            continue
        mean = v[int(ck[b]):int(ck[b + 1])].mean(dim=0).numpy()
        np.testing.assert_allclose(tiny[int(cq[b]):int(cq[b + 1])],
                                   np.broadcast_to(mean, (lq[b],) + mean.shape), atol=1e-7)


def test_rows_api_matches_full_forward():
    q, k, v, cq, ck, _, _ = _rand_case(26, 4, 9, 4, 2, 8, 6, chunked=True)
    full = oracle.attention(q, k, v, cq, ck, 4, 2, is_causal=True, softcap=2.0)
    n = full.shape[0] * 4
    rows = np.arange(n)[::3][::-1].copy()
    part = oracle.attention_rows(q, k, v, cq, ck, rows, 4, 2, is_causal=True, softcap=2.0)
    np.testing.assert_array_equal(part, full.reshape(n, -1)[rows])


def test_default_scale_is_float32_inverse_sqrt():
    for d in (1, 3, 8, 64, 96, 128, 256):
        assert abs(oracle.resolve_scale(0.0, d) - 1 / math.sqrt(d)) <= 2 ** -24 / math.sqrt(d)
    assert oracle.resolve_scale(0.0, 128) == float(np.float32(1) / np.sqrt(np.float32(128)))
    assert oracle.resolve_scale(0.0, 64) == 0.125
    assert math.isclose(oracle.resolve_scale(0.0, 256), 1 / 16)


# ---------------------------------------------------------------------------
# Local (sliding) window: keys before causal limit + 1 - W are masked
# (attention.rs / group_query_attention.rs `local_window`).
# ---------------------------------------------------------------------------
def _window_case(seed, causal):
    g = torch.Generator().manual_seed(700 + seed)
    B, H, Hkv, d, dv = 3, 4, 2, 8, 6
    lkv = torch.randint(1, 14, (B,), generator=g).tolist()
    lq = [int(torch.randint(1, L + 1, (1,), generator=g)) for L in lkv]
    q, k, v, cq, ck = workloads.make_packed(lq, lkv, H, Hkv, d, dv, "f32", gen=g)
    return q.double(), k.double(), v.double(), cq, ck, lq, lkv, H, Hkv, d


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("causal", [False, True])
def test_window_row_is_plain_attention_over_the_window_keys(seed, causal):
    """Every output row under a window W equals the un-windowed oracle run on
    that single query row against only the keys the window leaves visible
    (a one-row problem in which nothing else is masked)."""
    q, k, v, cq, ck, lq, lkv, H, Hkv, d = _window_case(seed, causal)
    for W in (1, 2, 5, 40):
        out = oracle.attention(q, k, v, cq, ck, H, Hkv, 0.0, causal, local_window=W)
        for b, (a, L) in enumerate(zip(lq, lkv)):
            for i in range(a):
                frontier = i + L - a
                lo, hi = max(0, frontier + 1 - W), (min(L, frontier + 1) if causal else L)
                kv0 = int(ck[b])
                for h in range(H):
                    got = out[int(cq[b]) + i, h]
                    if hi <= lo:
                        np.testing.assert_array_equal(got, 0.0)
                        continue
                    g_ = h // (H // Hkv)
                    ref = oracle.attention(q[int(cq[b]) + i: int(cq[b]) + i + 1, h:h + 1],
                                           k[kv0 + lo: kv0 + hi, g_:g_ + 1],
                                           v[kv0 + lo: kv0 + hi, g_:g_ + 1],
                                           torch.tensor([0, 1], dtype=torch.int32),
                                           torch.tensor([0, hi - lo], dtype=torch.int32), 1, 1,
                                           oracle.resolve_scale(0.0, d), False)
                    np.testing.assert_allclose(got, ref[0, 0], rtol=0, atol=1e-12)


def test_window_of_one_returns_the_value_row_at_the_causal_limit():
    q, k, v, cq, ck, lq, lkv, H, Hkv, d = _window_case(9, True)
    out = oracle.attention(q, k, v, cq, ck, H, Hkv, 0.0, True, local_window=1)
    for b, (a, L) in enumerate(zip(lq, lkv)):
        for i in range(a):
            for h in range(H):
                row = v[int(ck[b]) + i + L - a, h // (H // Hkv)].numpy()
                np.testing.assert_allclose(out[int(cq[b]) + i, h], row, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_window_wider_than_every_sequence_changes_nothing(causal):
    q, k, v, cq, ck, lq, lkv, H, Hkv, d = _window_case(3, causal)
    a = oracle.attention(q, k, v, cq, ck, H, Hkv, 0.0, causal)
    for W in (max(lkv) + max(lq), 10 ** 6):
        np.testing.assert_array_equal(oracle.attention(q, k, v, cq, ck, H, Hkv, 0.0, causal,
                                                       local_window=W), a)


def test_window_rows_api_matches_full_forward():
    q, k, v, cq, ck, lq, lkv, H, Hkv, d = _window_case(5, True)
    full = oracle.attention(q, k, v, cq, ck, H, Hkv, 0.0, True, local_window=3)
    rows = np.arange(full.shape[0] * H)[::3]
    got = oracle.attention_rows(q, k, v, cq, ck, rows, H, Hkv, 0.0, True, local_window=3)
    np.testing.assert_array_equal(got, full.reshape(-1, full.shape[-1])[rows])


# ---------------------------------------------------------------------------
# The padded form (opset-24 nonpad_kv_seqlen; attention.rs per-batch causal
# offset and padding frontier), written separately over the padded layout
# ---------------------------------------------------------------------------
def _padded_case(seed, causal=None):
    g = torch.Generator().manual_seed(700 + seed)
    B, H, Hkv, d, dv = 4, 6, 2, 8, 5
    q_seq = int(torch.randint(1, 7, (1,), generator=g))
    kv_seq = int(torch.randint(1, 12, (1,), generator=g))
    nonpad = torch.randint(0, kv_seq + 1, (B,), generator=g).tolist()
    nonpad[0] = kv_seq  # one full slot
    q = torch.randn(B, q_seq, H, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, kv_seq, Hkv, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, kv_seq, Hkv, dv, generator=g, dtype=torch.float64)
    if causal is None:
        causal = bool(seed % 2)
    return q, k, v, nonpad, H, Hkv, causal


@pytest.mark.parametrize("seed", range(6))
def test_padded_form_matches_sdpa_with_both_frontiers(seed):
    """attention_padded against torch float64 SDPA given the padded op's
    explicit mask: j < nonpad[b], and (causal) j <= i + nonpad[b] - q_seq."""
    q, k, v, nonpad, H, Hkv, causal = _padded_case(seed)
    B, q_seq, _, d = q.shape
    kv_seq = k.shape[1]
    out = oracle.attention_padded(q, k, v, nonpad, H, Hkv, 0.0, causal, softcap=0.0)
    i = torch.arange(q_seq).view(-1, 1)
    j = torch.arange(kv_seq).view(1, -1)
    for b in range(B):
        mask = (j < nonpad[b]).expand(q_seq, kv_seq)
        if causal:
            mask = mask & (j <= i + (nonpad[b] - q_seq))
        ref = torch.nan_to_num(_sdpa_seq(q[b], k[b], v[b], oracle.resolve_scale(0.0, d), mask),
                               nan=0.0)
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=0, atol=1e-12)
        assert np.all(out[b][~mask.any(dim=1).numpy()] == 0.0)


@pytest.mark.parametrize("seed", range(6))
def test_padded_form_equals_packed_form_on_the_prefix_sum(seed):
    """The two representations the module doc relates: the padded op equals
    the packed op fed cu_seqlens_kv = exclusive prefix sum of nonpad (its
    rows packed) and cu_seqlens_q of equal q_seq lengths.  Two separate loop
    nests, so this holds each against the other; softcap included."""
    q, k, v, nonpad, H, Hkv, causal = _padded_case(seed)
    B, q_seq, _, d = q.shape
    softcap = 0.0 if seed < 3 else 1.5
    out = oracle.attention_padded(q, k, v, nonpad, H, Hkv, 0.3, causal, softcap)
    kp = torch.cat([k[b, :nonpad[b]] for b in range(B)])
    vp = torch.cat([v[b, :nonpad[b]] for b in range(B)])
    packed = oracle.attention(q.reshape(B * q_seq, H, d), kp, vp,
                              workloads.cu_from_lengths([q_seq] * B),
                              workloads.cu_from_lengths(nonpad), H, Hkv, 0.3, causal, softcap)
    np.testing.assert_allclose(out.reshape(packed.shape), packed, rtol=0, atol=1e-13)


def test_padded_form_ignores_what_the_padding_holds():
    q, k, v, nonpad, H, Hkv, _ = _padded_case(11, causal=True)
    nonpad[1] = 0
    a = oracle.attention_padded(q, k, v, nonpad, H, Hkv, 0.0, True)
    k2, v2 = k.clone(), v.clone()
    for b, n in enumerate(nonpad):
        k2[b, n:] = 1e6
        v2[b, n:] = -7.0
    np.testing.assert_array_equal(oracle.attention_padded(q, k2, v2, nonpad, H, Hkv, 0.0, True), a)
    assert np.all(a[1] == 0.0)


def test_padded_form_rejects_lengths_outside_the_slot():
    q, k, v, nonpad, H, Hkv, causal = _padded_case(2)
    for bad in (-1, k.shape[1] + 1):
        with pytest.raises(ValueError):
            oracle.attention_padded(q, k, v, [bad] + nonpad[1:], H, Hkv, 0.0, causal)
