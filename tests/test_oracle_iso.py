"""Pins of the oracle's ISO3/ISO4 block quantizer and its Lloyd-Max table."""

import json
import os

import numpy as np
import pytest

from quantized_paged_kv_append_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SIGMA = 1.0 / np.sqrt(128.0)


def test_lloyd_max_matches_max_1960(orc):
    g = json.load(open(os.path.join(GOLDEN, "lloyd_max_gaussian.json")))
    for n in (8, 16):
        lv, resid, iters = orc.lloyd_max(n, 1.0)
        pos = lv[n // 2:]
        assert np.max(np.abs(pos - np.array(g["levels"][str(n)]))) < g["tolerance_levels"]
        assert np.allclose(lv, -lv[::-1], atol=1e-14), "symmetric levels"
        assert resid < 1e-12, "centroid condition at the fixed point"


def test_lloyd_max_conditions_by_quadrature(orc):
    stats = pytest.importorskip("scipy.stats")
    integrate = pytest.importorskip("scipy.integrate")
    g = json.load(open(os.path.join(GOLDEN, "lloyd_max_gaussian.json")))
    for n in (8, 16):
        lv, _, _ = orc.lloyd_max(n, 1.0)
        b = np.concatenate([[-np.inf], 0.5 * (lv[1:] + lv[:-1]), [np.inf]])
        mse = 0.0
        for j in range(n):
            mass = stats.norm.cdf(b[j + 1]) - stats.norm.cdf(b[j])
            mean = integrate.quad(lambda z: z * stats.norm.pdf(z), b[j], b[j + 1])[0] / mass
            assert abs(mean - lv[j]) < 1e-8, "each level is the mean of its cell"
            mse += integrate.quad(lambda z: (z - lv[j]) ** 2 * stats.norm.pdf(z), b[j], b[j + 1])[0]
        assert abs(mse - g["mse"][str(n)]) / g["mse"][str(n)] < g["tolerance_mse_rel"]


def test_iso_table_is_fp16_rounded_sigma_levels(orc):
    for bits, n in ((3, 8), (4, 16)):
        lv, mids = orc.iso_table(bits)
        raw, _, _ = orc.lloyd_max(n, SIGMA)
        assert np.array_equal(lv.astype(np.float16).astype(np.float32), lv), "levels are fp16 values"
        assert np.all(np.abs(lv - raw) <= np.abs(raw) * 2.0 ** -11), "within half an fp16 ulp"
        assert np.array_equal(mids, (lv[1:] + lv[:-1]) * np.float32(0.5))
        assert np.all(np.diff(lv) > 0)


def _block(seed, scale=1.0):
    return synth.bf16_to_f32(synth.bf16_bits(synth.normals_f32(seed, "misc", 128) * np.float32(scale)))


@pytest.mark.parametrize("bits", [3, 4])
def test_iso_codes_nearest_centroid(orc, bits):
    quat = synth.unit_quaternion(7)
    lv, mids = orc.iso_table(bits)
    for seed in range(20):
        x = _block(seed, 0.5 + seed)
        codes, s16, y, n, cn = orc.quant_iso_block(bits, x, quat)
        dist = np.abs(y[:, None].astype(np.float64) - lv[None, :].astype(np.float64))
        best = np.argmin(dist, axis=1)
        tie = np.sort(dist, axis=1)
        clear = (tie[:, 1] - tie[:, 0]) > 1e-7
        assert np.array_equal(codes[clear], best[clear])
        # y is the rotated unit vector: its norm is 1 (fp32)
        assert abs(np.linalg.norm(y.astype(np.float64)) - 1.0) < 1e-5


@pytest.mark.parametrize("bits", [3, 4])
def test_iso_norm_preservation(orc, bits):
    quat = synth.unit_quaternion(8)
    lv, _ = orc.iso_table(bits)
    fmt = orc.FMT_ISO3 if bits == 3 else orc.FMT_ISO4
    for seed in range(20):
        x = _block(100 + seed, 0.1 * (seed + 1))
        codes, s16, y, n, cn = orc.quant_iso_block(bits, x, quat)
        xn = np.linalg.norm(x.astype(np.float64))
        # before fp16 rounding the corrected norm reproduces ||x|| to 1e-5 rel
        s32 = np.float32(n) / np.float32(cn)
        assert abs(float(s32) * cn - xn) <= 1e-5 * xn
        # dequantized vector: ||xhat|| = s16 * ||c|| (rotation is orthogonal)
        code, scale = orc.quant_vector(fmt, 0, x, quat)
        xh = orc.dequant_vector(fmt, 0, 128, code, scale, quat)
        s = orc.half_value(np.frombuffer(scale[:2].tobytes(), np.uint16))[0]
        assert abs(np.linalg.norm(xh) - s * cn) <= 1e-5 * s * cn
        # and ||x|| up to the fp16 rounding of the stored norm
        assert abs(np.linalg.norm(xh) - xn) <= (2.0 ** -11 + 1e-5) * xn


@pytest.mark.parametrize("bits", [3, 4])
def test_iso_symmetric_input_symmetric_codes(orc, bits):
    quat = synth.unit_quaternion(9)
    n_lv = 8 if bits == 3 else 16
    x = _block(200)
    c1, s1, _, _, _ = orc.quant_iso_block(bits, x, quat)
    c2, s2, _, _, _ = orc.quant_iso_block(bits, -x, quat)
    y1 = orc.quant_iso_block(bits, x, quat)[2]
    away = np.abs(y1) > 1e-6
    assert np.array_equal(c2[away], (n_lv - 1) - c1[away])
    assert s1 == s2


@pytest.mark.parametrize("bits", [3, 4])
def test_iso_pack_roundtrip_and_sizes(orc, bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 2 ** bits, 128)
    packed = orc.pack_iso(bits, codes)
    assert packed.size == (48 if bits == 3 else 64)
    assert np.array_equal(orc.unpack_iso(bits, packed), codes)
    # bit placement of the spec: element 5 of ISO3 -> low bits of byte 1 at 2..3, high bit of byte 32 bit 5
    if bits == 3:
        one = np.zeros(128, int)
        one[5] = 0b111
        p = orc.pack_iso(3, one)
        assert p[1] == 0b1100 and p[32] == 0b100000 and p.sum() == 0b1100 + 0b100000
    else:
        one = np.zeros(128, int)
        one[5] = 0xA
        p = orc.pack_iso(4, one)
        assert p[2] == 0xA0 and p.sum() == 0xA0


@pytest.mark.parametrize("bits", [3, 4])
def test_iso_zero_block(orc, bits):
    quat = synth.unit_quaternion(10)
    codes, s16, y, n, cn = orc.quant_iso_block(bits, np.zeros(128, np.float32), quat)
    assert n == 0 and s16 == 0 and np.all(y == 0)
    fmt = orc.FMT_ISO3 if bits == 3 else orc.FMT_ISO4
    code, scale = orc.quant_vector(fmt, 0, np.zeros(128, np.float32), quat)
    assert np.all(orc.dequant_vector(fmt, 0, 128, code, scale, quat) == 0)


def test_iso_identity_quaternion_codes_the_unrotated_vector(orc):
    one = np.array([1, 0, 0, 0], np.float32)
    lv, mids = orc.iso_table(4)
    x = _block(300)
    codes, s16, y, n, cn = orc.quant_iso_block(4, x, one)
    assert np.array_equal(y, (x / np.float32(n)).astype(np.float32))


def test_sumsq_tree_is_exact_on_integers(orc):
    v = np.arange(128, dtype=np.float32)
    assert orc.sumsq128(v) == float(np.sum(np.arange(128) ** 2))
