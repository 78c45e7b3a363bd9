"""The C-ABI library builds, loads and exports every symbol include/*.h
declares; host-side argument checks work without a GPU (CPU only)."""
import ctypes
import glob
import os
import re

import pytest

import gqa_attention_cu_gb300 as pva

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pva.build()
    return pva.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(pva_[a-z0-9_]+)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("pva_forward", "pva_get_status", "pva_schedule", "pva_status_string",
              "pva_last_error", "pva_release", "pva_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libpva.so does not export {name}"


def test_status_strings_and_version(lib):
    assert pva.pva_status_string(0) == "ok"
    assert "invalid" in pva.pva_status_string(-1)
    assert "unsupported" in pva.pva_status_string(-2)
    assert pva.pva_status_string(12345) == "unknown status"
    assert pva.pva_version() == (0 << 16) | (1 << 8)


def _call(lib, **kw):
    args = dict(q=16, k=16, v=16, cq=16, ck=16, out=16, B=1, H=4, Hkv=2, d=128, dv=128,
                scale=0.0, causal=0, softcap=0.0, dtype=2)
    args.update(kw)
    return lib.pva_forward(args["q"], args["k"], args["v"], args["cq"], args["ck"], args["out"],
                           args["B"], args["H"], args["Hkv"], args["d"], args["dv"],
                           args["scale"], args["causal"], args["softcap"], args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(cq=None), -1), (dict(ck=None), -1),
    (dict(B=0), -1), (dict(H=0), -1), (dict(Hkv=0), -1), (dict(H=6, Hkv=4), -1),
    (dict(dtype=3), -1), (dict(dtype=-1), -1),
    (dict(scale=float("nan")), -1), (dict(softcap=float("inf")), -1),
    (dict(d=80, dv=80), -2), (dict(d=128, dv=64), -2), (dict(d=192, dv=96), -2),
    (dict(dtype=0, d=512, dv=64), -2),
    (dict(H=256, Hkv=1), -2), (dict(q=24), -1),
])
def test_host_argument_checks_need_no_gpu(lib, kw, code):
    """Malformed calls are rejected on the host, before any CUDA call, with the
    codes include/pva.h documents."""
    assert _call(lib, **kw) == code
    assert pva.pva_last_error() != ""


def test_python_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(pva.PvaError):
        pva.load_library(str(tmp_path / "missing.so"))


def _call_padded(lib, **kw):
    args = dict(q=16, k=16, v=16, nonpad=16, out=16, B=2, q_seq=4, kv_seq=8, H=4, Hkv=2, d=128,
                dv=128, scale=0.0, causal=0, softcap=0.0, dtype=2)
    args.update(kw)
    return lib.pva_forward_padded(args["q"], args["k"], args["v"], args["nonpad"], args["out"],
                                  args["B"], args["q_seq"], args["kv_seq"], args["H"],
                                  args["Hkv"], args["d"], args["dv"], args["scale"],
                                  args["causal"], args["softcap"], args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(nonpad=None), -1), (dict(B=0), -1), (dict(q_seq=-1), -1), (dict(kv_seq=-3), -1),
    (dict(B=3, q_seq=1 << 30), -1), (dict(B=5, kv_seq=1 << 29), -1),
    (dict(H=6, Hkv=4), -1), (dict(d=80, dv=80), -2), (dict(dtype=7), -1),
])
def test_padded_host_argument_checks_need_no_gpu(lib, kw, code):
    """pva_forward_padded rejects malformed calls on the host, before any CUDA
    call (its extra rules: a non-null nonpad_kv_seqlen, non-negative q_seq and
    kv_seq, B * q_seq and B * kv_seq within int32)."""
    assert _call_padded(lib, **kw) == code
    assert pva.pva_last_error() != ""


def _call_kvcache(lib, **kw):
    args = dict(q=16, kn=16, vn=16, kc=16, vc=16, sk=16, cos=16, sin=16, pid=None, out=16, B=2,
                q_seq=1, k_seq=1, cap=64, H=8, Hkv=2, d=128, rot=0, rows=0, inter=0,
                rot_dtype=0, scale=0.0, softcap=0.0, window=0, dtype=2)
    args.update(kw)
    a = args
    return lib.pva_gqa_kvcache(a["q"], a["kn"], a["vn"], a["kc"], a["vc"], a["sk"], a["cos"],
                               a["sin"], a["pid"], a["out"], a["B"], a["q_seq"], a["k_seq"],
                               a["cap"], a["H"], a["Hkv"], a["d"], a["rot"], a["rows"],
                               a["inter"], a["rot_dtype"], a["scale"], a["softcap"],
                               a["window"], a["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(kc=None), -1), (dict(sk=None), -1), (dict(out=None), -1),
    (dict(B=0), -1), (dict(q_seq=0), -1), (dict(k_seq=-1), -1), (dict(cap=0), -1),
    (dict(kn=None), -1), (dict(B=3, cap=1 << 29), -1),
    (dict(d=127), -2),
    (dict(rot=3, rows=8), -1), (dict(rot=256, rows=8), -1), (dict(rot=64, rows=0), -1),
    (dict(rot=64, rows=8, cos=None), -1), (dict(rot=64, rows=8, q_seq=4, k_seq=2), -1),
    (dict(rot=64, rows=8, rot_dtype=2), -1), (dict(rot=64, rows=8, rot_dtype=1, dtype=0), -1),
    (dict(H=6, Hkv=4), -1), (dict(dtype=5), -1),
])
def test_kvcache_host_argument_checks_need_no_gpu(lib, kw, code):
    """pva_gqa_kvcache rejects malformed calls on the host, before any CUDA
    call: null pointers, counts, the cache extent, odd head sizes, rotary
    dimensions and tables, rotary with k_seq not in {0, q_seq}, table types."""
    assert _call_kvcache(lib, **kw) == code
    assert pva.pva_last_error() != ""


def _call_from_host(lib, cq, ck, **kw):
    import ctypes
    B = len(cq) - 1
    cq_a = (ctypes.c_int32 * len(cq))(*cq)
    ck_a = (ctypes.c_int32 * len(ck))(*ck)
    args = dict(buf=16, cu=16, B=B, H=4, Hkv=2, d=128, dv=128, dtype=2, chunks=0)
    args.update(kw)
    b = args["buf"]
    return lib.pva_forward_from_host(b, b, b, ctypes.addressof(cq_a), ctypes.addressof(ck_a), b,
                                     b, b, b, b, args["cu"], args["B"], args["H"], args["Hkv"],
                                     args["d"], args["dv"], 0.0, 1, 0.0, args["dtype"],
                                     args["chunks"], None)


@pytest.mark.parametrize("cq,ck,kw", [
    ([1, 3], [0, 3], {}),                 # offsets not starting at 0
    ([0, 3], [1, 3], {}),
    ([0, 3, 2], [0, 3, 4], {}),           # decreasing
    ([0, 3, 4], [0, 5, 4], {}),
    ([0, 3], [0, 3], dict(B=0)),
    ([0, 3], [0, 3], dict(cu=None)),
    ([0, 3], [0, 3], dict(buf=None)),     # null buffers with rows to move
    ([0, 3], [0, 3], dict(H=0)),
    ([0, 3], [0, 3], dict(dtype=5)),
])
def test_forward_from_host_checks_offsets_on_the_host(lib, cq, ck, kw):
    """pva_forward_from_host sizes its copies from the host offsets, so it
    rejects malformed ones (and missing buffers) before any CUDA call."""
    assert _call_from_host(lib, cq, ck, **kw) == -1
    assert pva.pva_last_error() != ""
