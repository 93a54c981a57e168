"""CPU oracle for the quantized paged KV-cache path (ctypes wrapper).

TEST INFRASTRUCTURE. Only the test suite, `__graft_entry__.smoke()` and the
benchmark's CPU-baseline leg may import this package. The product library never
does, and shares no code with `qkv_oracle.cpp`.

`build()` compiles qkv_oracle.cpp with g++ (-O2 -ffp-contract=off, no fast
math) into oracle/_build/libqkv_oracle.so.
"""

from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qkv_oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libqkv_oracle.so")

FMT_INT8, FMT_K8V4, FMT_ISO3, FMT_ISO4 = 0, 1, 2, 3
FMT_Q4, FMT_K8, FMT_V8 = 4, 5, 6   # q4_0 both stores (rotated); int8 K + bf16 V; bf16 K + int8 V

_lib = None


def build(force: bool = False) -> str:
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = C.CDLL(_LIB_PATH)
        _declare(_lib)
    return _lib


P = C.c_void_p
I = C.c_int
I64 = C.c_int64
F = C.c_float
D = C.c_double


def _declare(L):
    sig = {
        "orc_half_from_f64_array": (None, [P, P, I64, I]),
        "orc_f64_from_half_array": (None, [P, P, I64]),
        "orc_f32_from_bf16_array": (None, [P, P, I64]),
        "orc_row_bytes": (I, [I, I, I, P, P]),
        "orc_lloyd_max": (I, [I, D, P, P, P]),
        "orc_iso_table": (I, [I, P, P]),
        "orc_quant_int8": (None, [P, I, P, P]),
        "orc_fwht256": (None, [P]),
        "orc_fwht256_f64": (None, [P]),
        "orc_quant_q4": (None, [P, I, P, P]),
        "orc_qmul": (None, [P, P, P]),
        "orc_sumsq128": (F, [P]),
        "orc_quant_iso_block": (I, [I, P, P, P, P, P, P, P]),
        "orc_pack_iso": (None, [I, P, P]),
        "orc_unpack_iso": (None, [I, P, P]),
        "orc_quant_vector": (I, [I, I, I, P, P, P, P]),
        "orc_dequant_vector": (I, [I, I, I, P, P, P, P]),
        "orc_append": (I, [I, I, I, I, I, P, P, P, P, P, P, I, P, P, P, I, P]),
        "orc_gather_dequant": (I, [I, I, I, I, I, P, P, P, P, P, I, I, I, P, P, P]),
        "orc_decode": (I, [I, I, I, I, I, P, P, P, P, P, I, I, P, I, P, F, P, P]),
        "orc_verify": (I, [I, I, I, I, I, P, P, P, P, P, I, I, P, P, I, P, F, P, P]),
        "orc_decode_split": (I, [I, I, I, I, I, P, P, P, P, P, I, P, I, I, F, P, P, I, P]),
        "orc_extend": (I, [I, I, I, I, I, P, P, P, P, P, P, P, I, P, P, I, P, I, F, I, P, P, I, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


_IDQ = np.array([1, 0, 0, 0], dtype=np.float32)


# ---- number formats -------------------------------------------------------
def half_bits(x, sat=False):
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().orc_half_from_f64_array(_p(x), _p(out), x.size, int(sat))
    return out


def half_value(h):
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float64)
    lib().orc_f64_from_half_array(_p(h), _p(out), h.size)
    return out


def bf16_value(b):
    b = _c(b, np.uint16)
    out = np.empty(b.shape, np.float32)
    lib().orc_f32_from_bf16_array(_p(b), _p(out), b.size)
    return out


# ---- geometry -------------------------------------------------------------
def row_bytes(fmt, store, head_dim):
    cb, sb = C.c_int(), C.c_int()
    if lib().orc_row_bytes(fmt, store, head_dim, C.byref(cb), C.byref(sb)) != 0:
        raise ValueError("bad format")
    return cb.value, sb.value


def plane_shapes(fmt, num_pages, num_kv_heads, head_dim, page_size=16):
    """[(k_codes bytes, k_scales bytes, v_codes bytes, v_scales bytes)] per-row
    sizes expanded to full plane byte counts."""
    kcb, ksb = row_bytes(fmt, 0, head_dim)
    vcb, vsb = row_bytes(fmt, 1, head_dim)
    rows = num_pages * num_kv_heads * page_size
    return rows * kcb, rows * ksb, rows * vcb, rows * vsb


# ---- Lloyd-Max --------------------------------------------------------------
def lloyd_max(n_levels, sigma):
    lv = np.empty(n_levels, np.float64)
    r, it = C.c_double(), C.c_int()
    if lib().orc_lloyd_max(n_levels, sigma, _p(lv), C.byref(r), C.byref(it)) != 0:
        raise ValueError
    return lv, r.value, it.value


def iso_table(bits):
    lv = np.empty(16, np.float32)
    mid = np.empty(15, np.float32)
    n = lib().orc_iso_table(bits, _p(lv), _p(mid))
    return lv[:n].copy(), mid[:n - 1].copy()


# ---- primitives -------------------------------------------------------------
def quant_int8(x):
    x = _c(x, np.float32)
    codes = np.empty(x.size, np.int8)
    scales = np.empty(x.size // 64, np.uint16)
    lib().orc_quant_int8(_p(x), x.size, _p(codes), _p(scales))
    return codes, scales


def fwht256(x):
    x = _c(x, np.float32).copy()
    lib().orc_fwht256(_p(x))
    return x


def fwht256_f64(x):
    x = _c(x, np.float64).copy()
    lib().orc_fwht256_f64(_p(x))
    return x


def quant_q4(x):
    x = _c(x, np.float32)
    nib = np.empty(x.size // 2, np.uint8)
    d = np.empty(x.size // 32, np.uint16)
    lib().orc_quant_q4(_p(x), x.size, _p(nib), _p(d))
    return nib, d


def qmul(p, v):
    p, v = _c(p, np.float32), _c(v, np.float32)
    y = np.empty(4, np.float32)
    lib().orc_qmul(_p(p), _p(v), _p(y))
    return y


def sumsq128(v):
    v = _c(v, np.float32)
    return lib().orc_sumsq128(_p(v))


def quant_iso_block(bits, x, quat):
    x, quat = _c(x, np.float32), _c(quat, np.float32)
    codes = np.empty(128, np.int32)
    s16 = np.empty(1, np.uint16)
    y = np.empty(128, np.float32)
    n, cn = C.c_float(), C.c_float()
    lib().orc_quant_iso_block(bits, _p(x), _p(quat), _p(codes), _p(s16), _p(y), C.byref(n), C.byref(cn))
    return codes, s16[0], y, n.value, cn.value


def pack_iso(bits, codes):
    codes = _c(codes, np.int32)
    out = np.empty(48 if bits == 3 else 64, np.uint8)
    lib().orc_pack_iso(bits, _p(codes), _p(out))
    return out


def unpack_iso(bits, packed):
    packed = _c(packed, np.uint8)
    out = np.empty(128, np.int32)
    lib().orc_unpack_iso(bits, _p(packed), _p(out))
    return out


def quant_vector(fmt, store, x, quat=None):
    x = _c(x, np.float32)
    quat = _IDQ if quat is None else _c(quat, np.float32)
    cb, sb = row_bytes(fmt, store, x.size)
    code = np.empty(cb, np.uint8)
    scale = np.empty(sb, np.uint8)
    lib().orc_quant_vector(fmt, store, x.size, _p(x), _p(quat), _p(code), _p(scale))
    return code, scale


def dequant_vector(fmt, store, head_dim, code, scale, quat=None):
    code, scale = _c(code, np.uint8), _c(scale, np.uint8)
    quat = _IDQ if quat is None else _c(quat, np.float32)
    out = np.empty(head_dim, np.float64)
    lib().orc_dequant_vector(fmt, store, head_dim, _p(code), _p(scale), _p(quat), _p(out))
    return out


# ---- paged operations -------------------------------------------------------
class Pool:
    """Byte planes of a paged KV pool: [num_pages, Hkv, page_size, row bytes]."""

    def __init__(self, fmt, num_pages, num_kv_heads, head_dim, page_size=16, quat=None):
        self.fmt, self.num_pages, self.hkv, self.d, self.p = fmt, num_pages, num_kv_heads, head_dim, page_size
        self.quat = _IDQ.copy() if quat is None else _c(quat, np.float32)
        kc, ks, vc, vs = plane_shapes(fmt, num_pages, num_kv_heads, head_dim, page_size)
        self.kc = np.zeros(kc, np.uint8)
        self.ks = np.zeros(ks, np.uint8)
        self.vc = np.zeros(vc, np.uint8)
        self.vs = np.zeros(vs, np.uint8)

    def planes(self):
        return self.kc, self.ks, self.vc, self.vs

    def _head(self):
        return (self.fmt, self.num_pages, self.hkv, self.d, self.p,
                _p(self.kc), _p(self.ks), _p(self.vc), _p(self.vs))

    def append(self, k_bf16, v_bf16, seq_id, pos, page_table):
        k, v = _c(k_bf16, np.uint16), _c(v_bf16, np.uint16)
        seq_id, pos, pt = _c(seq_id, np.int32), _c(pos, np.int32), _c(page_table, np.int32)
        n = seq_id.size
        return lib().orc_append(*self._head(), _p(k), _p(v), n, _p(seq_id), _p(pos), _p(pt),
                                pt.shape[1], _p(self.quat))

    def gather_dequant(self, page_table, b, length):
        pt = _c(page_table, np.int32)
        k = np.empty((length, self.hkv, self.d), np.float64)
        v = np.empty((length, self.hkv, self.d), np.float64)
        rc = lib().orc_gather_dequant(*self._head(), _p(pt), pt.shape[1], b, length, _p(self.quat), _p(k), _p(v))
        if rc != 0:
            raise ValueError("page table entry out of range")
        return k, v

    def decode(self, q_bf16, page_table, seq_lens, scale):
        q = _c(q_bf16, np.uint16)
        pt, sl = _c(page_table, np.int32), _c(seq_lens, np.int32)
        B, Hq, Dh = q.shape
        out = np.empty((B, Hq, Dh), np.float64)
        rc = lib().orc_decode(*self._head(), _p(q), B, Hq, _p(pt), pt.shape[1], _p(sl), scale,
                              _p(self.quat), _p(out))
        if rc != 0:
            raise ValueError(f"orc_decode failed ({rc})")
        return out

    def verify(self, q_bf16, page_table, seq_lens, cu_seqlens, scale):
        """Verify window: rows cu[b] .. cu[b+1]-1 of q are the last W_b positions of
        sequence b, query j attending [0, seq_lens[b] - W_b + j + 1)."""
        q = _c(q_bf16, np.uint16)
        pt, sl, cu = _c(page_table, np.int32), _c(seq_lens, np.int32), _c(cu_seqlens, np.int32)
        T, Hq, Dh = q.shape
        out = np.empty((T, Hq, Dh), np.float64)
        rc = lib().orc_verify(*self._head(), _p(q), sl.size, Hq, _p(cu), _p(pt), pt.shape[1], _p(sl), scale,
                              _p(self.quat), _p(out))
        if rc != 0:
            raise ValueError(f"orc_verify failed ({rc})")
        return out

    def decode_split(self, q_bf16, page_table, length, scale, bounds):
        q = _c(q_bf16, np.uint16)
        pt, bd = _c(page_table, np.int32), _c(bounds, np.int32)
        Hq, Dh = q.shape[-2], q.shape[-1]
        out = np.empty((Hq, Dh), np.float64)
        rc = lib().orc_decode_split(*self._head(), _p(q), Hq, _p(pt), pt.shape[1], length, scale,
                                    _p(self.quat), _p(bd), bd.size - 1, _p(out))
        if rc != 0:
            raise ValueError
        return out

    def extend(self, q_bf16, k_new, v_new, cu_seqlens, prefix_lens, page_table, scale, causal=True, rows=None):
        q, kn, vn = _c(q_bf16, np.uint16), _c(k_new, np.uint16), _c(v_new, np.uint16)
        cu, pl, pt = _c(cu_seqlens, np.int32), _c(prefix_lens, np.int32), _c(page_table, np.int32)
        T, Hq, Dh = q.shape
        r = None if rows is None else _c(rows, np.int32)
        nrows = T if r is None else r.size
        out = np.empty((nrows, Hq, Dh), np.float64)
        rc = lib().orc_extend(*self._head(), _p(q), _p(kn), _p(vn), Hq, _p(cu), _p(pl), pl.size,
                              _p(pt), pt.shape[1], scale, int(causal), _p(self.quat), _p(r), nrows, _p(out))
        if rc != 0:
            raise ValueError(f"orc_extend failed ({rc})")
        return out
