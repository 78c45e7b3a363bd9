"""The benchmark's work counts (CPU): visible (query, key) pairs per the mask
rules of packed_varlen_attention.rs ("Causal alignment") and the softmax
kernels' local window, checked against brute-force enumeration; FLOPs and
K/V bytes follow from them."""
import itertools

import pytest

import bench


def brute_visible(a, b, causal, window):
    out = []
    for i in range(a):
        limit = i + b - a  # tail-aligned causal limit
        n = 0
        for j in range(b):
            if causal and j > limit:
                continue
            if window > 0 and j < limit + 1 - window:
                continue
            n += 1
        out.append(n)
    return out


@pytest.mark.parametrize("causal,window", list(itertools.product([False, True], [0, 1, 5, 64])))
def test_visible_keys_match_brute_force(causal, window):
    for a, b in [(1, 1), (1, 50), (7, 7), (7, 30), (30, 7), (64, 200), (129, 129), (0, 5),
                 (5, 0)]:
        got = [int(x) for x in bench.visible_keys(a, b, causal, window)]
        assert got == brute_visible(a, b, causal, window), (a, b, causal, window)


def test_work_units_flops_and_bytes():
    lq, lkv = [3, 1, 0, 17], [10, 40, 5, 17]
    w = {"lq": lq, "lkv": lkv, "is_causal": True, "num_heads": 8, "kv_num_heads": 2,
         "head_size": 192, "v_head_size": 128, "dtype": "bf16", "window": 6}
    pairs = sum(sum(brute_visible(a, b, True, 6)) for a, b in zip(lq, lkv))
    flops, kv_bytes = bench.work_units(w)
    assert flops == pairs * 2 * 8 * (192 + 128)
    assert kv_bytes == sum(lkv) * 2 * (192 + 128) * 2
    assert bench.unmasked_pairs(lq, lkv, True, 6) == pairs
