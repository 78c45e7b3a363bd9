"""The Python binding only marshals arguments (CPU, no GPU): each wrapper is
run against a recording stand-in for libpva.so and must pass exactly the
pointers, sizes and flags that include/pva.h declares, in order."""
import pytest
import torch

import gqa_attention_cu_gb300 as pva


class Recorder:
    """Stands in for the loaded library: records every call, returns 0."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append((name, args))
            return 0
        return fn


@pytest.fixture
def rec(monkeypatch):
    r = Recorder()
    monkeypatch.setattr(pva, "_lib", r)
    return r


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def test_pva_forward_marshalling(rec):
    q, k, v, o = _t(10, 8, 64), _t(12, 2, 64), _t(12, 2, 48), _t(10, 8, 48)
    cq, ck = _t(3, dtype=torch.int32), _t(3, dtype=torch.int32)
    pva.pva_forward(q, k, v, cq, ck, o, 2, 8, 2, 64, 48, 0.25, 1, 30.0, stream=7)
    name, a = rec.calls[-1]
    assert name == "pva_forward"
    assert a == (q.data_ptr(), k.data_ptr(), v.data_ptr(), cq.data_ptr(), ck.data_ptr(),
                 o.data_ptr(), 2, 8, 2, 64, 48, 0.25, 1, 30.0, 2, 7)


def test_forward_local_and_noalloc_marshalling(rec):
    q, k, v, o = _t(4, 4, 64, dtype=torch.float16), _t(4, 4, 64, dtype=torch.float16), \
        _t(4, 4, 64, dtype=torch.float16), _t(4, 4, 64, dtype=torch.float16)
    cq = _t(2, dtype=torch.int32)
    pva.pva_forward_local(q, k, v, cq, cq, o, 1, 4, 4, 64, 64, is_causal=1, local_window=9,
                          stream=0)
    name, a = rec.calls[-1]
    assert name == "pva_forward_local" and a[-3:] == (9, 1, 0) and a[12] == 1
    st = _t(1, dtype=torch.int32)
    pva.pva_forward_noalloc(q, k, v, cq, cq, o, 1, 4, 4, 64, 64, device_status=st, stream=0)
    name, a = rec.calls[-1]
    assert name == "pva_forward_noalloc" and a[-2:] == (st.data_ptr(), 0) and a[-3] == 1


def test_forward_padded_marshalling(rec):
    q, k, v, o = _t(2, 5, 8, 128), _t(2, 9, 2, 128), _t(2, 9, 2, 128), _t(2, 5, 8, 128)
    npd = _t(2, dtype=torch.int64)
    pva.pva_forward_padded(q, k, v, npd, o, 2, 5, 9, 8, 2, 128, 128, is_causal=1, stream=0)
    name, a = rec.calls[-1]
    assert name == "pva_forward_padded"
    assert a == (q.data_ptr(), k.data_ptr(), v.data_ptr(), npd.data_ptr(), o.data_ptr(), 2, 5,
                 9, 8, 2, 128, 128, 0.0, 1, 0.0, 2, 0)


def test_gqa_kvcache_marshalling_derives_shapes(rec):
    B, q_seq, H, Hkv, d, cap = 3, 2, 8, 2, 128, 40
    q, kn, vn = _t(B, q_seq, H, d), _t(B, q_seq, Hkv, d), _t(B, q_seq, Hkv, d)
    kc, vc, o = _t(B, Hkv, cap, d), _t(B, Hkv, cap, d), _t(B, q_seq, H, d)
    sk = _t(B, dtype=torch.int32)
    cos, sin = _t(50, 32, dtype=torch.float32), _t(50, 32, dtype=torch.float32)
    pid = _t(B, q_seq, dtype=torch.int64)
    pva.pva_gqa_kvcache(q, kn, vn, kc, vc, sk, o, H, Hkv, cos, sin, pid, True, 0.5, 20.0, 7,
                        stream=0)
    name, a = rec.calls[-1]
    assert name == "pva_gqa_kvcache"
    assert a == (q.data_ptr(), kn.data_ptr(), vn.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                 sk.data_ptr(), cos.data_ptr(), sin.data_ptr(), pid.data_ptr(), o.data_ptr(),
                 B, q_seq, q_seq, cap, H, Hkv, d, 64, 50, 1, 0, 0.5, 20.0, 7, 2, 0)
    # no new rows and no rotary: NULL pointers, k_seq 0, rotary_dim 0
    pva.pva_gqa_kvcache(q, None, None, kc, vc, sk, o, H, Hkv, stream=0)
    name, a = rec.calls[-1]
    assert a[1] is None and a[2] is None and a[6] is None and a[7] is None and a[8] is None
    assert a[12] == 0 and a[17] == 0 and a[18] == 0


def test_errors_raise_with_the_library_text(monkeypatch):
    class Failing(Recorder):
        def __getattr__(self, name):
            if name == "pva_status_string":
                return lambda rc: b"invalid argument"
            if name == "pva_last_error":
                return lambda: b"B must be >= 1"
            return lambda *a: -1
    monkeypatch.setattr(pva, "_lib", Failing())
    with pytest.raises(pva.PvaError, match="B must be >= 1"):
        pva.pva_forward(_t(1, 1, 64), _t(1, 1, 64), _t(1, 1, 64), _t(1, dtype=torch.int32),
                        _t(1, dtype=torch.int32), _t(1, 1, 64), 0, 1, 1, 64, 64, stream=0)


def test_forward_from_host_marshalling(rec):
    qh, kh, vh, oh = _t(10, 8, 64), _t(12, 2, 64), _t(12, 2, 48), _t(10, 8, 48)
    qd, kd, vd, od = _t(10, 8, 64), _t(12, 2, 64), _t(12, 2, 48), _t(10, 8, 48)
    cq, ck = _t(3, dtype=torch.int32), _t(3, dtype=torch.int32)
    cu = _t(4 * 2 + 34, dtype=torch.int32)
    pva.pva_forward_from_host(qh, kh, vh, cq, ck, oh, qd, kd, vd, od, cu, 2, 8, 2, 64, 48,
                              0.25, 1, 30.0, chunks=3, stream=5)
    name, a = rec.calls[-1]
    assert name == "pva_forward_from_host"
    assert a == (qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), cq.data_ptr(), ck.data_ptr(),
                 oh.data_ptr(), qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(),
                 cu.data_ptr(), 2, 8, 2, 64, 48, 0.25, 1, 30.0, 2, 3, 5)
