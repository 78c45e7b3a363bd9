"""TEST INFRASTRUCTURE ONLY: the oracle of one GroupQueryAttention step
against a fixed-capacity KV cache.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this module; the product path never does, and nothing here comes
from the product.  It follows the group_query_attention.rs page of the
"onnx-runtime-ep-cuda" source, step by step and in the page's order:

1. ``gqa_prepare_metadata``: per sequence total = seqlens_k + 1,
   past = total - k_seq, first query position = total - q_seq, and the bounds
   the page checks (bit 1 total beyond int32, 2 past < 0, 4 first < 0,
   8 past beyond the past capacity, 16 total beyond the present capacity,
   32 a rotary position outside the cos/sin tables).  In-place caches have one
   capacity for both.
2. ``gqa_append_cache``: the k_seq new rows of each (sequence, kv head) go to
   cache rows [past, past + k_seq).
3. ``gqa_rope_bnsh`` on the queries (positions first + s) and on the appended
   keys (positions past + s), or on position_ids when given: pair k of a head
   row is (2k, 2k+1) when interleaved, else (k, k + rot/2); it becomes
   (c x0 - s x1, s x0 + c x1) with each product and sum rounded to f32, as the
   page's f32 kernel writes it; the result is stored in the tensor's type.
4. ``gqa_attention_reference_f32``'s definition: query row s of sequence b
   sees cache rows j <= first + s (and, with a window W > 0, j >= first + s +
   1 - W), scores scale * q.k with the optional softcap, softmax, times V.
   This is the packed oracle (``oracle.attention``, fp64) run on the valid
   cache rows, with L_q = q_seq and L_kv = total: the tail-aligned causal
   limit i + L_kv - L_q is first + i.

A step whose metadata has any error bit, or that follows a rejected step (the
page's latch-first rule), changes nothing and produces no output.

The rotation is done with numpy float32 arithmetic (one IEEE rounding per
operation, no fused multiply-add); conversions to bf16/f16 round to nearest
even (torch).
"""
from __future__ import annotations

import numpy as np
import torch

from . import attention

INT32_MAX = 2 ** 31 - 1


def metadata(seqlens_k, q_seq: int, k_seq: int, capacity: int, rotary: bool = False,
             cache_rows: int = 0, position_ids=None):
    """Per sequence (total, past, first, error bits), the page's metadata step."""
    res = []
    pos = None if position_ids is None else np.asarray(position_ids, dtype=np.int64)
    for b, sk in enumerate(np.asarray(seqlens_k, dtype=np.int64).tolist()):
        total = sk + 1
        past = total - k_seq
        first = total - q_seq
        bits = 0
        if total > INT32_MAX:
            bits |= 1
        if past < 0:
            bits |= 2
        if first < 0:
            bits |= 4
        if past > capacity:
            bits |= 8
        if total > capacity:
            bits |= 16
        if rotary:
            for s in range(q_seq):
                p = int(pos[b, s]) if pos is not None else first + s
                if p < 0 or p >= cache_rows:
                    bits |= 32
        res.append((total, past, first, bits))
    return res


def rope_pairs(d: int, rot: int, interleaved: bool):
    """(d0, d1, rotated) for every pair k in [0, d/2) of a head row."""
    half = rot // 2
    pairs = []
    for k in range(d // 2):
        if k < half:
            pairs.append((2 * k, 2 * k + 1, True) if interleaved else (k, k + half, True))
        else:
            t = rot + 2 * (k - half)
            pairs.append((t, t + 1, False))
    return pairs


def rotate(x: np.ndarray, cos_rows: np.ndarray, sin_rows: np.ndarray, rot: int,
           interleaved: bool) -> np.ndarray:
    """Head rows x (float32 [..., d]) rotated by table rows (float32
    [..., rot/2], broadcast against x's leading axes)."""
    x = np.asarray(x, dtype=np.float32)
    pairs = [p for p in rope_pairs(x.shape[-1], rot, interleaved) if p[2]]
    i0 = np.array([p[0] for p in pairs], dtype=np.int64)
    i1 = np.array([p[1] for p in pairs], dtype=np.int64)
    c = np.asarray(cos_rows, dtype=np.float32)
    s = np.asarray(sin_rows, dtype=np.float32)
    x0, x1 = x[..., i0], x[..., i1]
    y = x.copy()
    # numpy float32: each product and each difference/sum rounded on its own
    y[..., i0] = c * x0 - s * x1
    y[..., i1] = s * x0 + c * x1
    return y


def rotate_row(x, cos_row, sin_row, rot: int, interleaved: bool) -> np.ndarray:
    """One head row (float32 [d]) rotated by one table row (float32 [rot/2])."""
    return rotate(np.asarray(x, dtype=np.float32)[None], np.asarray(cos_row)[None],
                  np.asarray(sin_row)[None], rot, interleaved)[0]


def _f32(t) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float32).numpy()


def gqa_cache_step(q, k_new, v_new, k_cache, v_cache, seqlens_k, num_heads: int,
                   kv_num_heads: int, cos_cache=None, sin_cache=None, position_ids=None,
                   interleaved: bool = False, scale: float = 0.0, softcap: float = 0.0,
                   local_window: int = 0, poisoned: bool = False, threads: int = 0):
    """One step.  q [B, q_seq, H, d]; k_new/v_new [B, k_seq, Hkv, d] or None;
    caches [B, Hkv, cap, d] (torch, any float dtype; not modified); seqlens_k
    [B]; cos/sin [rows, rot/2] or None.  Returns (out, k_after, v_after, bits):
    out float64 [B, q_seq, H, d] or None when the step is rejected; the caches
    after the step (copies, in the caches' dtype); the OR of the error bits
    (-1 for a step rejected because an earlier one was)."""
    B, q_seq, H, d = q.shape
    Hkv = int(kv_num_heads)
    assert H == num_heads and k_cache.shape[1] == Hkv
    cap = k_cache.shape[2]
    k_seq = 0 if k_new is None else k_new.shape[1]
    rot = 0 if cos_cache is None else 2 * cos_cache.shape[1]
    rows = 0 if cos_cache is None else cos_cache.shape[0]
    kc, vc = k_cache.detach().to("cpu").clone(), v_cache.detach().to("cpu").clone()
    if poisoned:
        return None, kc, vc, -1
    meta = metadata(seqlens_k, q_seq, k_seq, cap, rot > 0, rows, position_ids)
    bits = 0
    for _, _, _, e in meta:
        bits |= e
    if bits:
        return None, kc, vc, bits

    cs = None if cos_cache is None else (_f32(cos_cache), _f32(sin_cache))
    pos = None if position_ids is None else np.asarray(position_ids, dtype=np.int64)

    def positions(starts, seq):
        """[B, seq] positions of rows starting at starts[b]."""
        if pos is not None:
            return pos[:, :seq]
        return np.asarray(starts, dtype=np.int64)[:, None] + np.arange(seq)[None, :]

    # steps 2 and 3 on the keys: the appended rows, keys rotated, values as given
    if k_seq:
        kn = k_new.detach().to("cpu")
        if rot:
            P = positions([m[1] for m in meta], k_seq)
            kr = rotate(_f32(k_new), cs[0][P][:, :, None, :], cs[1][P][:, :, None, :], rot,
                        interleaved)
            kn = torch.from_numpy(kr).to(kc.dtype)
        for b, (total, past, first, _) in enumerate(meta):
            kc[b, :, past:past + k_seq] = kn[b].permute(1, 0, 2).to(kc.dtype)
            vc[b, :, past:past + k_seq] = v_new[b].to("cpu").permute(1, 0, 2).to(vc.dtype)
    # step 3 on the queries
    qr = q.detach().to("cpu")
    if rot:
        P = positions([m[2] for m in meta], q_seq)
        qr = torch.from_numpy(rotate(_f32(q), cs[0][P][:, :, None, :], cs[1][P][:, :, None, :],
                                     rot, interleaved)).to(q.dtype)
    # step 4: the valid cache rows of every sequence, as packed sequences
    totals = [m[0] for m in meta]
    kp = torch.cat([kc[b, :, :totals[b]].permute(1, 0, 2) for b in range(B)])
    vp = torch.cat([vc[b, :, :totals[b]].permute(1, 0, 2) for b in range(B)])
    cu_q = torch.tensor([0] + [q_seq * (b + 1) for b in range(B)], dtype=torch.int32)
    cu_kv = torch.tensor(np.concatenate([[0], np.cumsum(totals)]), dtype=torch.int32)
    out = attention(qr.reshape(B * q_seq, H, d), kp, vp, cu_q, cu_kv, H, Hkv, scale, True,
                    softcap, threads=threads, local_window=local_window)
    return out.reshape(B, q_seq, H, d), kc, vc, 0
