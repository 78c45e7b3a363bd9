"""Pins of the KV-cache step oracle (``oracle/gqa_cache.py``) to things other
than itself (CPU only).

* metadata: hand-derived totals, first rows and error bits of the page's
  metadata kernel (group_query_attention.rs, `gqa_prepare_metadata`);
* rotary embedding (`gqa_rope_bnsh`): exact special angles (0 and 90
  degrees), complex multiplication in float64 within the f32 rounding bound,
  interleaved and half-split layouts as one permutation of each other, the
  untouched tail dims, and the relative-position property of the rotation;
* append (`gqa_append_cache`): only rows [past, past + k_seq) change, and to
  exactly the new rows;
* the attention step against torch float64 SDPA over the valid cache rows
  with the tail-aligned causal mask (and window), independently rotated
  inputs for the rotary case, rejected and poisoned steps.

Every pin takes the oracle module as an argument so that
``test_oracle_cache_mutants.py`` can run it against planted mistakes.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import gqa_cache

pytestmark = pytest.mark.filterwarnings("ignore")


# ---------------------------------------------------------------------------
# metadata
# ---------------------------------------------------------------------------
META_CASES = [
    # (seqlens_k, q_seq, k_seq, capacity, rotary, cache_rows, position_ids) -> (total, past, first, bits)
    (([4], 1, 1, 8, False, 0, None), (5, 4, 4, 0)),
    (([0], 2, 2, 8, False, 0, None), (1, -1, -1, 2 | 4)),
    (([0], 2, 0, 8, False, 0, None), (1, 1, -1, 4)),
    (([3], 1, 0, 8, False, 0, None), (4, 4, 3, 0)),
    (([5], 1, 3, 8, False, 0, None), (6, 3, 5, 0)),
    (([7], 1, 1, 8, False, 0, None), (8, 7, 7, 0)),
    (([8], 1, 1, 8, False, 0, None), (9, 8, 8, 16)),
    (([9], 1, 1, 8, False, 0, None), (10, 9, 9, 8 | 16)),
    (([2 ** 31 - 1], 1, 1, 2 ** 31, False, 0, None), (2 ** 31, 2 ** 31 - 1, 2 ** 31 - 1, 1)),
    (([4], 2, 2, 8, True, 5, None), (5, 3, 3, 0)),
    (([4], 2, 2, 8, True, 4, None), (5, 3, 3, 32)),
    (([4], 2, 2, 8, True, 5, [[-1, 0]]), (5, 3, 3, 32)),
    (([4], 2, 2, 8, True, 5, [[4, 0]]), (5, 3, 3, 0)),
    (([4], 2, 2, 8, True, 5, [[0, 5]]), (5, 3, 3, 32)),
]


def pin_metadata(gc=gqa_cache):
    for (args, expect) in META_CASES:
        sk, qs, ks, cap, rot, rows, pid = args
        got = gc.metadata(sk, qs, ks, cap, rot, rows,
                          None if pid is None else np.array(pid, dtype=np.int64))
        assert got == [expect], (args, got, expect)


def test_metadata_worked_cases():
    pin_metadata()


# ---------------------------------------------------------------------------
# rotary embedding
# ---------------------------------------------------------------------------
def _rows(seed, n, d):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, d, generator=g) * 3).numpy().astype(np.float32)


def pin_rope_special_angles(gc=gqa_cache):
    x = _rows(1, 5, 16)
    half = 6
    for inter in (False, True):
        same = gc.rotate(x, np.ones((5, half), np.float32), np.zeros((5, half), np.float32), 12,
                         inter)
        np.testing.assert_array_equal(same, x)
        quarter = gc.rotate(x, np.zeros((5, half), np.float32), np.ones((5, half), np.float32),
                            12, inter)
        for k in range(half):
            d0, d1 = (2 * k, 2 * k + 1) if inter else (k, k + half)
            np.testing.assert_array_equal(quarter[:, d0], -x[:, d1])
            np.testing.assert_array_equal(quarter[:, d1], x[:, d0])
        np.testing.assert_array_equal(quarter[:, 12:], x[:, 12:])


def pin_rope_is_complex_multiplication(gc=gqa_cache):
    x = _rows(2, 7, 24)
    rot, half = 20, 10
    g = torch.Generator().manual_seed(3)
    ang = (torch.rand(7, half, generator=g, dtype=torch.float64) * 2 * math.pi).numpy()
    c, s = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    for inter in (False, True):
        y = gc.rotate(x, c, s, rot, inter)
        for k in range(half):
            d0, d1 = (2 * k, 2 * k + 1) if inter else (k, k + half)
            z = (x[:, d0].astype(np.float64) + 1j * x[:, d1].astype(np.float64)) * \
                (c[:, k].astype(np.float64) + 1j * s[:, k].astype(np.float64))
            # two rounded products and one rounded sum: within 3 units of
            # f32 rounding of the sum of the two terms' magnitudes
            u = 2.0 ** -24
            b0 = 3 * u * (np.abs(c[:, k] * x[:, d0]) + np.abs(s[:, k] * x[:, d1]))
            b1 = 3 * u * (np.abs(s[:, k] * x[:, d0]) + np.abs(c[:, k] * x[:, d1]))
            assert np.all(np.abs(y[:, d0] - z.real) <= b0)
            assert np.all(np.abs(y[:, d1] - z.imag) <= b1)
        np.testing.assert_array_equal(y[:, rot:], x[:, rot:])


def pin_rope_layouts_are_one_permutation(gc=gqa_cache):
    """Half-split on x equals interleaved on x with its rotated dims
    reordered (k, k + half) -> (2k, 2k + 1), output reordered back."""
    d, rot, half = 16, 12, 6
    x = _rows(4, 6, d)
    g = torch.Generator().manual_seed(5)
    c = torch.rand(6, half, generator=g).numpy().astype(np.float32)
    s = torch.rand(6, half, generator=g).numpy().astype(np.float32)
    perm = np.arange(d)
    for k in range(half):
        perm[2 * k], perm[2 * k + 1] = k, k + half
    split = gc.rotate(x, c, s, rot, False)
    inter = gc.rotate(x[:, perm], c, s, rot, True)
    np.testing.assert_array_equal(split[:, perm], inter)
    pairs = gc.rope_pairs(d, rot, False)
    assert sorted([p[0] for p in pairs] + [p[1] for p in pairs]) == list(range(d))


def pin_rope_relative_position(gc=gqa_cache):
    """With tables cos/sin(p * theta_k), the dot product of a query rotated to
    position p and a key rotated to position p' depends on p - p' only."""
    d = rot = 32
    half = rot // 2
    theta = 10000.0 ** (-np.arange(half) / half)
    table = np.arange(64)[:, None] * theta[None, :]
    C, S = np.cos(table).astype(np.float32), np.sin(table).astype(np.float32)
    q, k = _rows(6, 1, d)[0], _rows(7, 1, d)[0]
    for inter in (False, True):
        def dot(p, pp):
            a = gc.rotate_row(q, C[p], S[p], rot, inter).astype(np.float64)
            b = gc.rotate_row(k, C[pp], S[pp], rot, inter).astype(np.float64)
            return float(a @ b)
        for delta in (0, 3, 17):
            ref = dot(delta, 0)
            for shift in (5, 20, 40):
                assert abs(dot(delta + shift, shift) - ref) <= 2e-4 * (1 + abs(ref))
        assert abs(dot(9, 0) - dot(0, 0)) > 1e-2  # the rotation does act


def test_rope_special_angles():
    pin_rope_special_angles()


def test_rope_is_complex_multiplication():
    pin_rope_is_complex_multiplication()


def test_rope_layouts_are_one_permutation():
    pin_rope_layouts_are_one_permutation()


def test_rope_relative_position():
    pin_rope_relative_position()


# ---------------------------------------------------------------------------
# append and the attention step
# ---------------------------------------------------------------------------
def _case(seed, B=3, q_seq=1, k_seq=1, H=4, Hkv=2, d=16, cap=12, dtype=torch.float32,
          seqlens=None):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, q_seq, H, d, generator=g).to(dtype)
    kn = torch.randn(B, k_seq, Hkv, d, generator=g).to(dtype) if k_seq else None
    vn = torch.randn(B, k_seq, Hkv, d, generator=g).to(dtype) if k_seq else None
    kc = torch.randn(B, Hkv, cap, d, generator=g).to(dtype)
    vc = torch.randn(B, Hkv, cap, d, generator=g).to(dtype)
    if seqlens is None:
        lo = max(q_seq, k_seq)
        seqlens = (torch.randint(lo, cap + 1, (B,), generator=g) - 1).tolist()
    return q, kn, vn, kc, vc, seqlens


def _sdpa_cache(q, kc, vc, totals, H, Hkv, scale, window=0):
    """float64 SDPA of q [B, q_seq, H, d] over rows [0, total_b) of the cache,
    query row s seeing rows j <= total - q_seq + s (and the window)."""
    B, q_seq, _, d = q.shape
    out = torch.zeros(B, q_seq, H, d, dtype=torch.float64)
    for b in range(B):
        T = totals[b]
        i = torch.arange(q_seq).view(-1, 1)
        j = torch.arange(T).view(1, -1)
        limit = T - q_seq + i
        mask = j <= limit
        if window > 0:
            mask = mask & (j >= limit + 1 - window)
        qq = q[b].double().permute(1, 0, 2).unsqueeze(0)
        kk = kc[b, :, :T].double().unsqueeze(0)
        vv = vc[b, :, :T].double().unsqueeze(0)
        r = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale,
                                           enable_gqa=True)
        out[b] = torch.nan_to_num(r.squeeze(0).permute(1, 0, 2), nan=0.0)
    return out.numpy()


def pin_append_touches_only_the_new_rows(gc=gqa_cache):
    q, kn, vn, kc, vc, sk = _case(11, q_seq=1, k_seq=2, dtype=torch.bfloat16)
    out, ka, va, bits = gc.gqa_cache_step(q, kn, vn, kc, vc, sk, 4, 2)
    assert bits == 0
    for b, s in enumerate(sk):
        past = s + 1 - 2
        keep = [r for r in range(kc.shape[2]) if not past <= r < past + 2]
        assert torch.equal(ka[b][:, keep], kc[b][:, keep])
        assert torch.equal(va[b][:, keep], vc[b][:, keep])
        assert torch.equal(ka[b][:, past:past + 2], kn[b].permute(1, 0, 2))
        assert torch.equal(va[b][:, past:past + 2], vn[b].permute(1, 0, 2))
    _, ka0, va0, bits0 = gc.gqa_cache_step(q, None, None, kc, vc, sk, 4, 2)
    assert bits0 == 0 and torch.equal(ka0, kc) and torch.equal(va0, vc)


def pin_step_matches_sdpa_over_the_cache(gc=gqa_cache):
    for seed, q_seq, k_seq, window in [(12, 1, 1, 0), (13, 3, 3, 0), (14, 4, 0, 0),
                                       (15, 3, 2, 2), (16, 1, 0, 3)]:
        q, kn, vn, kc, vc, sk = _case(seed, q_seq=q_seq, k_seq=k_seq, H=6, Hkv=2)
        out, ka, va, bits = gc.gqa_cache_step(q, kn, vn, kc, vc, sk, 6, 2, scale=0.3,
                                              local_window=window)
        assert bits == 0
        ref = _sdpa_cache(q, ka, va, [s + 1 for s in sk], 6, 2, oracle.resolve_scale(0.3, 16),
                          window)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def _rotate_reference(x, pos, theta, inter):
    """Independent rotation: complex multiplication in float64 per pair."""
    y = x.double().clone()
    half = theta.shape[0]
    for k in range(half):
        d0, d1 = (2 * k, 2 * k + 1) if inter else (k, k + half)
        ang = pos.double() * theta[k]
        z = torch.complex(x[..., d0].double(), x[..., d1].double()) * torch.polar(
            torch.ones_like(ang), ang)
        y[..., d0], y[..., d1] = z.real, z.imag
    return y


def pin_rotary_step_against_independent_rotation(gc=gqa_cache):
    """f32 step with rotary tables against SDPA on queries and appended keys
    rotated by complex multiplication at the page's positions: queries at
    first + s, appended keys at past + s (k_seq = q_seq), or k_seq = 0 (the
    queries alone)."""
    rows, d, rot = 40, 16, 12
    theta = 10000.0 ** (-torch.arange(rot // 2, dtype=torch.float64) / (rot // 2))
    table = torch.arange(rows, dtype=torch.float64)[:, None] * theta[None, :]
    C, S = torch.cos(table).float(), torch.sin(table).float()
    for seed, q_seq, k_seq, inter in [(21, 2, 2, False), (22, 3, 0, True), (23, 1, 1, True)]:
        q, kn, vn, kc, vc, sk = _case(seed, q_seq=q_seq, k_seq=k_seq, d=d, cap=30)
        out, ka, va, bits = gc.gqa_cache_step(q, kn, vn, kc, vc, sk, 4, 2, C, S,
                                              interleaved=inter)
        assert bits == 0
        kexp, vexp = kc.double().clone(), vc.double().clone()
        qexp = torch.zeros(q.shape, dtype=torch.float64)
        for b, s_k in enumerate(sk):
            total = s_k + 1
            first, past = total - q_seq, total - k_seq
            qexp[b] = _rotate_reference(q[b], torch.arange(first, first + q_seq)[:, None],
                                        theta, inter)
            if k_seq:
                kr = _rotate_reference(kn[b], torch.arange(past, past + k_seq)[:, None], theta,
                                       inter)
                kexp[b, :, past:past + k_seq] = kr.permute(1, 0, 2)
                vexp[b, :, past:past + k_seq] = vn[b].double().permute(1, 0, 2)
        np.testing.assert_allclose(ka.double().numpy(), kexp.numpy(), rtol=0, atol=1e-5)
        np.testing.assert_array_equal(va.double().numpy(), vexp.numpy())
        ref = _sdpa_cache(qexp, kexp, vexp, [s + 1 for s in sk], 4, 2,
                          oracle.resolve_scale(0.0, d))
        np.testing.assert_allclose(out, ref, rtol=0, atol=2e-5)


def pin_position_ids_override(gc=gqa_cache):
    """position_ids equal to the default positions change nothing; shifted
    ones change the rotation."""
    rows, rot = 30, 8
    th = np.arange(rows)[:, None] * (10000.0 ** (-np.arange(rot // 2) / (rot // 2)))[None, :]
    C = torch.from_numpy(np.cos(th).astype(np.float32))
    S = torch.from_numpy(np.sin(th).astype(np.float32))
    q, kn, vn, kc, vc, sk = _case(31, q_seq=2, k_seq=2, cap=20, dtype=torch.bfloat16)
    a = gc.gqa_cache_step(q, kn, vn, kc, vc, sk, 4, 2, C, S)
    pid = np.array([[s + 1 - 2, s + 1 - 1] for s in sk], dtype=np.int64)
    b = gc.gqa_cache_step(q, kn, vn, kc, vc, sk, 4, 2, C, S, position_ids=pid)
    assert np.array_equal(a[0], b[0]) and torch.equal(a[1], b[1])
    c = gc.gqa_cache_step(q, kn, vn, kc, vc, sk, 4, 2, C, S, position_ids=pid + 1)
    assert not torch.equal(a[1], c[1])


def pin_rejected_and_poisoned_steps_change_nothing(gc=gqa_cache):
    q, kn, vn, kc, vc, _ = _case(41, q_seq=1, k_seq=1, cap=8)
    for sk, bits in [([3, 8, 1], 16), ([3, -1, 1], 2 | 4), ([3, 9, 1], 8 | 16)]:
        out, ka, va, got = gc.gqa_cache_step(q, kn, vn, kc, vc, sk, 4, 2)
        assert out is None and got == bits
        assert torch.equal(ka, kc) and torch.equal(va, vc)
    out, ka, va, got = gc.gqa_cache_step(q, kn, vn, kc, vc, [3, 4, 1], 4, 2, poisoned=True)
    assert out is None and got == -1 and torch.equal(ka, kc) and torch.equal(va, vc)


def test_append_touches_only_the_new_rows():
    pin_append_touches_only_the_new_rows()


def test_step_matches_sdpa_over_the_cache():
    pin_step_matches_sdpa_over_the_cache()


def test_rotary_step_against_independent_rotation():
    pin_rotary_step_against_independent_rotation()


def test_position_ids_override():
    pin_position_ids_override()


def test_rejected_and_poisoned_steps_change_nothing():
    pin_rejected_and_poisoned_steps_change_nothing()


ALL_PINS = [pin_metadata, pin_rope_special_angles, pin_rope_is_complex_multiplication,
            pin_rope_layouts_are_one_permutation, pin_rope_relative_position,
            pin_append_touches_only_the_new_rows, pin_step_matches_sdpa_over_the_cache,
            pin_rotary_step_against_independent_rotation, pin_position_ids_override,
            pin_rejected_and_poisoned_steps_change_nothing]
