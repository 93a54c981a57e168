"""Pins of the oracle's dequantization (orc_dequant_vector and the pool gather)
against values fixed outside the oracle: codes and scales packed by hand in
this file, numpy's fp16 decoding, scipy's Sylvester Hadamard matrix, a 4x4
left-multiplication matrix written here from Hamilton's rules, and the
reconstruction error that the Lloyd-Max distortion (Max 1960, pinned in
test_oracle_iso.py) allows.

Sources: "feat(kvcache): add ISO3/ISO4 KV-cache quantization", section "What"
(per 128-value block: normalise, rotate each 4-D group by one unit quaternion,
nearest Lloyd-Max level, corrected norm; the dequantization undoes the
rotation); "--kv k8v4: hybrid KV cache", sections "What" and "How" (q4_0 V in
the FWHT-256-rotated domain, rotated back on the way out); "qwen35/q36: --kv -
int8 K/V caches", section "What it does" (code times the group's fp16 scale).
"""

import json
import os

import numpy as np
import pytest

from quantized_paged_kv_append_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_inputs(seed, n, scale=1.0):
    return synth.bf16_to_f32(synth.bf16_bits(synth.normals_f32(seed, "misc", n) * np.float32(scale)))


def _f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def _left_matrix(w, x, y, z):
    """Matrix of v -> p (x) v for p = w + xi + yj + zk, written from i^2 = j^2 =
    k^2 = ijk = -1 (component order: real, i, j, k)."""
    return np.array([[w, -x, -y, -z],
                     [x, w, -z, y],
                     [y, z, w, -x],
                     [z, -y, x, w]], np.float64)


# ------------------------------------------------------------------ int8
def test_int8_dequant_is_code_times_fp16_scale(orc):
    x = _bf16_inputs(11, 256 * 30, 1.5)
    x[5::256] *= 20.0                                 # outlier channel
    for v in x.reshape(30, 256):
        code, scale = orc.quant_vector(orc.FMT_INT8, 0, v)
        deq = orc.dequant_vector(orc.FMT_INT8, 0, 256, code, scale)
        d16 = _f16(scale.view(np.uint16))            # numpy decodes the stored scales
        want = code.view(np.int8).reshape(4, 64).astype(np.float64) * d16[:, None]
        assert np.array_equal(deq, want.ravel())
        assert np.all(np.abs(v.astype(np.float64) - deq).reshape(4, 64) <= d16[:, None] / 2 + 1e-12)


def test_int8_dequant_hand_packed(orc):
    # codes -127..127 in a known order, scale 2^-5 in group 0, 0.75 in group 1
    codes = np.concatenate([np.arange(-32, 32), np.arange(127, 63, -1)]).astype(np.int8)
    scale = np.array([0x2800, 0x3A00], np.uint16)     # fp16 bit patterns of 2^-5 and 0.75
    deq = orc.dequant_vector(orc.FMT_INT8, 0, 128, codes.view(np.uint8), scale.view(np.uint8))
    want = np.concatenate([np.arange(-32, 32) * 2.0 ** -5, np.arange(127, 63, -1) * 0.75])
    assert np.array_equal(deq, want)


# ------------------------------------------------------------------ q4_0 V (k8v4)
def test_q4_dequant_hand_packed_nibble_order(orc):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(256).astype(np.float64)
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, size=(8, 32))
    q[:, :16] = np.arange(16)                          # element j and j + 16 always differ:
    q[:, 16:] = 15 - np.arange(16)                     # a swapped nibble order changes every value
    q[3] = rng.integers(0, 16, 32)
    packed = (q[:, :16] | (q[:, 16:] << 4)).astype(np.uint8).ravel()   # byte j: j low, j + 16 high
    dbits = np.array([0x3C00, 0xBC00, 0x3800, 0x4000, 0x2E66, 0xB555, 0x0001, 0x7BFF], np.uint16)
    r = (q - 8).astype(np.float64) * _f16(dbits)[:, None]              # rotated-domain values
    want = H @ r.ravel() / 16                                          # back to the original domain
    deq = orc.dequant_vector(orc.FMT_K8V4, 1, 256, packed, dbits.view(np.uint8))
    assert np.max(np.abs(deq - want)) <= 1e-12 * np.max(np.abs(want))
    swapped = (q[:, 16:] | (q[:, :16] << 4)).astype(np.uint8).ravel()
    other = orc.dequant_vector(orc.FMT_K8V4, 1, 256, swapped, dbits.view(np.uint8))
    assert np.max(np.abs(other - want)) > 0.1 * np.max(np.abs(want)), "the test sees the nibble order"


@pytest.mark.parametrize("fmt,store", [(1, 1), (4, 0), (4, 1)])
def test_q4_reconstruction_within_half_step(orc, fmt, store):
    """k8v4 V and both stores of the q4_0 format (K rotated like V: "rotate K after RoPE
    and V", qwen35/q36 page, "Not in this PR")."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(256).astype(np.float64)
    x = _bf16_inputs(12, 256 * 20, 1.0).reshape(20, 256)
    x[:, [3, 77]] *= 20.0
    for v in x:
        code, scale = orc.quant_vector(fmt, store, v)
        deq = orc.dequant_vector(fmt, store, 256, code, scale)
        ds = _f16(scale.view(np.uint16))
        d = np.abs(ds)
        # the error, seen in the rotated domain (H/16 is orthonormal), is at most half a
        # step d per element, and at most a whole step for values clamped at code 15
        # (x / d > 7.5, on the side opposite the block's extreme)
        r = (H @ v.astype(np.float64) / 16).reshape(8, 32)
        err_rot = (H @ (v.astype(np.float64) - deq) / 16).reshape(8, 32)
        top = r / ds[:, None] > 7.5
        bound = np.where(top, d[:, None], d[:, None] / 2) * (1 + 1e-5)
        assert np.all(np.abs(err_rot) <= bound)
        # and the norm of the error is the same in both domains
        assert abs(np.linalg.norm(err_rot) - np.linalg.norm(v - deq)) < 1e-9 * np.linalg.norm(v)


# ------------------------------------------------------------------ ISO3 / ISO4
def _hand_pack(bits, codes):
    """Reading of the pages' block layout: ISO3 = 32 B of low 2-bit fields (value i
    at byte i/4, bits 2(i%4)) + 16 B of high bits (byte 32 + i/8, bit i%8); ISO4 =
    value i at byte i/2, low nibble when i is even."""
    if bits == 3:
        out = np.zeros(48, np.uint8)
        for i, c in enumerate(codes):
            out[i // 4] |= (c & 3) << (2 * (i % 4))
            out[32 + i // 8] |= ((c >> 2) & 1) << (i % 8)
        return out
    out = np.zeros(64, np.uint8)
    for i, c in enumerate(codes):
        out[i // 2] |= c << (4 * (i % 2))
    return out


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("quat", [(1.0, 0.0, 0.0, 0.0), (0.0, 1.0, 0.0, 0.0), (0.5, -0.5, 0.5, 0.5), "seeded"])
def test_iso_dequant_hand_computed(orc, bits, quat):
    quat = synth.unit_quaternion(3) if isinstance(quat, str) else np.array(quat, np.float32)
    lv, _ = orc.iso_table(bits)
    n = len(lv)
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, n, size=256)
    codes[:n] = np.arange(n)                           # every level appears
    packed = np.concatenate([_hand_pack(bits, codes[:128]), _hand_pack(bits, codes[128:])])
    s = np.array([0x3E00, 0xC500], np.uint16)          # norm scales 1.5 and -5.0
    if bits == 3:
        scale = s.view(np.uint8)
    else:                                              # ISO4: norm then a reserved fp16 per block
        scale = np.array([s[0], 0, s[1], 0], np.uint16).view(np.uint8)
    fmt = orc.FMT_ISO3 if bits == 3 else orc.FMT_ISO4
    deq = orc.dequant_vector(fmt, 0, 256, packed, scale, quat)
    w, x, y, z = (float(t) for t in quat)
    conj = _left_matrix(w, -x, -y, -z)                 # conj(q) (x) c undoes q (x) .
    c = lv.astype(np.float64)[codes].reshape(64, 4)
    want = (c @ conj.T).ravel() * np.repeat(_f16(s), 128)
    assert np.max(np.abs(deq - want)) <= 1e-6 * np.max(np.abs(want))


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("quat", [(0.0, 1.0, 0.0, 0.0), "seeded"])
def test_iso_reconstruction_within_lloyd_max_distortion(orc, bits, quat):
    """dequant(quant(x)) ~ x: the relative error of a block is the error of coding
    the rotated unit vector, whose coordinates are ~N(0, 1/128), so its square is
    about the Lloyd-Max MSE of a unit Gaussian (0.0345 for 8 levels, 0.0095 for
    16; Max 1960). A rotation that is not undone (a missing conjugate) leaves an
    error near sqrt(2) (near 2 for q = i)."""
    g = json.load(open(os.path.join(GOLDEN, "lloyd_max_gaussian.json")))
    mse = g["mse"]["8" if bits == 3 else "16"]
    quat = synth.unit_quaternion(4) if isinstance(quat, str) else np.array(quat, np.float32)
    fmt = orc.FMT_ISO3 if bits == 3 else orc.FMT_ISO4
    x = _bf16_inputs(13, 128 * 200, 1.0).reshape(200, 128)
    x[::3] *= 40.0
    rel = []
    for v in x:
        code, scale = orc.quant_vector(fmt, 0, v, quat)
        deq = orc.dequant_vector(fmt, 0, 128, code, scale, quat)
        rel.append(np.linalg.norm(v - deq) / np.linalg.norm(v))
        cos = float(np.dot(v, deq) / (np.linalg.norm(v) * np.linalg.norm(deq)))
        assert cos > 1.0 - 3.0 * mse, "direction kept to within the coding distortion"
    rel = np.array(rel)
    # the mean squared relative error estimates the MSE (plus the norm correction's
    # small share); every block stays well inside twice the expected error
    assert abs(np.mean(rel ** 2) / mse - 1.0) < 0.25
    assert np.max(rel) < 2.0 * np.sqrt(mse)


def test_pool_gather_reads_the_hand_packed_planes(orc):
    """The pool's gather goes through the page table and returns the same values as
    the hand-computed int8 dequantization of the planes it reads."""
    D, hkv, npages = 128, 2, 3
    pool = orc.Pool(orc.FMT_INT8, npages, hkv, D)
    rng = np.random.default_rng(9)
    kc = rng.integers(-127, 128, size=(npages, hkv, 16, D)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(npages, hkv, 16, D)).astype(np.int8)
    ks = rng.integers(0x2000, 0x3C00, size=(npages, hkv, 16, D // 64)).astype(np.uint16)
    vs = rng.integers(0x2000, 0x3C00, size=(npages, hkv, 16, D // 64)).astype(np.uint16)
    pool.kc[:] = kc.view(np.uint8).ravel()
    pool.vc[:] = vc.view(np.uint8).ravel()
    pool.ks[:] = ks.view(np.uint8).ravel()
    pool.vs[:] = vs.view(np.uint8).ravel()
    table = np.array([[2, 0, 1]], np.int32)
    L = 40
    k, v = pool.gather_dequant(table, 0, L)
    for t in range(L):
        pg, sl = table[0, t // 16], t % 16
        for h in range(hkv):
            wk = kc[pg, h, sl].astype(np.float64) * np.repeat(_f16(ks[pg, h, sl]), 64)
            wv = vc[pg, h, sl].astype(np.float64) * np.repeat(_f16(vs[pg, h, sl]), 64)
            assert np.array_equal(k[t, h], wk) and np.array_equal(v[t, h], wv)


@pytest.mark.parametrize("fmt,store", [(5, 1), (6, 0)])
def test_unquantized_store_returns_the_bf16_input(orc, fmt, store):
    """The one-store formats keep the other store as the bf16 input bits: two bytes
    per value, little-endian bf16, no scale row; reading it back is exact."""
    x = _bf16_inputs(14, 128 * 8, 30.0)
    x[:4] = [0.0, -0.0, 2.0 ** -130, -(2.0 ** 100)]
    for v in x.reshape(8, 128):
        code, scale = orc.quant_vector(fmt, store, v)
        assert code.size == 256 and scale.size == 0
        assert np.array_equal(code.view(np.uint16), synth.bf16_bits(v))
        deq = orc.dequant_vector(fmt, store, 128, code, scale)
        assert np.array_equal(deq, v.astype(np.float64))
