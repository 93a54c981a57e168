"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol include/qkv.h declares, agrees with the oracle on row geometry,
computes the same Lloyd-Max table independently, and rejects invalid
arguments before touching the device."""

import ctypes as C
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qlib():
    from quantized_paged_kv_append_gb300 import build, _lib
    build.build()
    return _lib


def _header_functions():
    src = open(os.path.join(ROOT, "include", "qkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*QKV_API\s+(?:const\s+)?\w+\*?\s+\**(\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(qlib):
    L = qlib.lib()
    names = _header_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(L, n), f"libqkv.so does not export {n}"
    assert set(names) == set(qlib.EXPORTS)


def test_row_bytes_match_oracle(qlib, orc):
    import quantized_paged_kv_append_gb300 as qkv
    for fmt, dims in ((0, (128, 256)), (1, (256,)), (2, (128, 256)), (3, (128, 256))):
        for d in dims:
            for st in (0, 1):
                assert qkv.row_bytes(fmt, st, d) == orc.row_bytes(fmt, st, d)


def test_iso_levels_independent_of_oracle_agree(qlib, orc):
    import quantized_paged_kv_append_gb300 as qkv
    for bits in (3, 4):
        ours = qkv.iso_levels(bits)
        ref, _ = orc.iso_table(bits)
        assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def _desc(qlib, fmt=0, d=256, hkv=2, pages=4, page_size=16, ptr=1 << 20):
    x = qlib.CacheDesc()
    x.format, x.num_pages, x.page_size, x.num_kv_heads, x.head_dim = fmt, pages, page_size, hkv, d
    x.k_codes = x.k_scales = x.v_codes = x.v_scales = ptr
    return x


def test_validation_rejects_before_launch(qlib):
    L = qlib.lib()
    P = C.c_void_p
    good = P(1 << 20)
    # append
    assert L.iso_kv_append(None, good, good, 1, good, good, good, 1, 1, None) == -1
    assert L.iso_kv_append(C.byref(_desc(qlib, fmt=7)), good, good, 1, good, good, good, 1, 1, None) == -5
    assert L.iso_kv_append(C.byref(_desc(qlib, d=192)), good, good, 1, good, good, good, 1, 1, None) == -2
    assert L.iso_kv_append(C.byref(_desc(qlib, fmt=1, d=128)), good, good, 1, good, good, good, 1, 1, None) == -2
    assert L.iso_kv_append(C.byref(_desc(qlib, fmt=2, d=64)), good, good, 1, good, good, good, 1, 1, None) == -2
    assert L.iso_kv_append(C.byref(_desc(qlib, page_size=32)), good, good, 1, good, good, good, 1, 1, None) == -1
    assert L.iso_kv_append(C.byref(_desc(qlib)), None, good, 1, good, good, good, 1, 1, None) == -1
    assert L.iso_kv_append(C.byref(_desc(qlib)), good, good, -1, good, good, good, 1, 1, None) == -1
    assert L.iso_kv_append(C.byref(_desc(qlib, ptr=(1 << 20) + 8)), good, good, 1, good, good, good, 1, 1, None) == -1
    assert L.iso_kv_append(C.byref(_desc(qlib)), good, good, 0, None, None, None, 0, 0, None) == 0  # no-op
    # decode
    d = C.byref(_desc(qlib))
    args = lambda **kw: dict(dict(q=good, B=1, Hq=16, pt=good, mp=4, sl=good, msl=64, scale=0.0625, out=good,
                                  odt=0, ws=good, wsb=1 << 30), **kw)

    def call(desc=d, **kw):
        a = args(**kw)
        return L.kv_decode_attn(desc, a["q"], a.get("kn"), a.get("vn"), a["B"], a["Hq"], a["pt"], a["mp"], a["sl"],
                                a["msl"], a["scale"], a["out"], a["odt"], a["ws"], a["wsb"], None)

    assert call(desc=None) == -1
    assert call(B=-1) == -1
    assert call(B=0) == 0
    assert call(q=None) == -1
    assert call(odt=5) == -1
    assert call(scale=float("nan")) == -1
    assert call(B=5000) == -8
    assert call(kn=good) == -1            # k_new without v_new


def test_gather_validation_rejects_before_launch(qlib):
    L = qlib.lib()
    P = C.c_void_p
    good = P(1 << 20)
    g = lambda desc, row=good, n=16, k=good, v=good: L.kv_gather_dequant(desc, row, n, k, v, None)
    assert g(None) == -1
    assert g(C.byref(_desc(qlib, fmt=9))) == -5
    assert g(C.byref(_desc(qlib, fmt=1, d=128))) == -2
    assert g(C.byref(_desc(qlib)), n=-1) == -1
    assert g(C.byref(_desc(qlib)), n=0, row=None, k=None, v=None) == 0   # no-op
    assert g(C.byref(_desc(qlib)), row=None) == -1
    assert g(C.byref(_desc(qlib)), k=P((1 << 20) + 4)) == -1            # fp32 rows must be 16-byte aligned


def test_verify_validation_rejects_before_launch(qlib):
    L = qlib.lib()
    P = C.c_void_p
    good = P(1 << 20)
    v = lambda desc, B=1, tq=2, q=good, cu=good: L.kv_verify_attn(desc, q, B, 16, cu, good, tq, good, 4, 64, 0.0625,
                                                                  good, 0, good, 1 << 30, None)
    assert v(None) == -1
    assert v(C.byref(_desc(qlib, fmt=7))) == -5
    assert v(C.byref(_desc(qlib)), B=-1) == -1
    assert v(C.byref(_desc(qlib)), B=0) == 0          # no-op
    assert v(C.byref(_desc(qlib)), tq=0) == 0         # no-op
    assert v(C.byref(_desc(qlib)), tq=2000) == -8     # more query rows than one decode call takes
    assert v(C.byref(_desc(qlib)), cu=None) == -1


def test_verify_fixed_validation_rejects_before_launch(qlib):
    L = qlib.lib()
    P = C.c_void_p
    good = P(1 << 20)
    v = lambda desc, B=1, W=2, q=good: L.kv_verify_attn_fixed(desc, q, B, W, 16, good, good, 4, 64, 0.0625, good, 0,
                                                              good, 1 << 30, None)
    assert v(None) == -1
    assert v(C.byref(_desc(qlib, fmt=7))) == -5
    assert v(C.byref(_desc(qlib)), W=0) == -1          # a window of at least one query
    assert v(C.byref(_desc(qlib)), B=-1) == -1
    assert v(C.byref(_desc(qlib)), B=0) == 0           # no-op
    assert v(C.byref(_desc(qlib, fmt=1)), B=0) == 0    # no-op (the expanded path)
    assert v(C.byref(_desc(qlib)), B=600, W=2) == -8   # more query rows than one decode call takes
    assert L.kv_verify_fixed_workspace_size(C.byref(_desc(qlib)), 1, 0, 16, 4) == 0
    assert L.kv_verify_fixed_workspace_size(C.byref(_desc(qlib)), 1, 2, 16, 0) == 0


def test_strerror_covers_codes(qlib):
    L = qlib.lib()
    for code in range(-8, 1):
        assert L.qkv_strerror(code)
    assert b"unknown" in L.qkv_strerror(-99)
