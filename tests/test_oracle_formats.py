"""Pins of the CPU oracle's number formats and quantizers against facts that do
not come from the oracle: IEEE conversions done by numpy/torch, closed-form
bounds, brute force over every code, and the pages' byte counts."""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

from quantized_paged_kv_append_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fp16 / bf16
@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_half_rounding_matches_numpy(orc):
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11,
                  1.0 + 3 * 2.0 ** -11, np.inf, -np.inf]),
    ])
    ours = orc.half_bits(x)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    # saturating variant: identical except overflow goes to +-65504
    sat = orc.half_bits(x, sat=True)
    ovf = np.isinf(x.astype(np.float16))
    assert np.array_equal(sat[~ovf], ref[~ovf])
    assert np.all(orc.half_value(sat[ovf]) == np.sign(x[ovf]) * 65504.0)


def test_half_decode_matches_numpy(orc):
    h = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    v = orc.half_value(h)
    ref = h.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    assert np.array_equal(v[finite], ref[finite])
    assert np.array_equal(np.isnan(v), np.isnan(ref))


def test_bf16_decode_matches_torch(orc):
    torch = pytest.importorskip("torch")
    b = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.bf16_value(b)
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_synth_bf16_narrowing_matches_torch():
    torch = pytest.importorskip("torch")
    x = synth.normals_f32(3, "misc", 50000) * np.float32(37.0)
    ours = synth.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------- int8 groups
def _bf16_inputs(seed, n, scale=1.0):
    return synth.bf16_to_f32(synth.bf16_bits(synth.normals_f32(seed, "misc", n) * np.float32(scale)))


def test_int8_error_bound_and_extreme_code(orc):
    x = _bf16_inputs(1, 64 * 400, 1.0)
    x[::64] *= 40.0  # an outlier in every group
    codes, scales = orc.quant_int8(x)
    d = orc.half_value(scales).astype(np.float64)
    xd = codes.reshape(-1, 64).astype(np.float64) * d[:, None]
    err = np.abs(xd - x.reshape(-1, 64))
    assert np.all(err <= d[:, None] / 2 + 1e-12), "|x - xhat| <= d16/2"
    amax_idx = np.argmax(np.abs(x.reshape(-1, 64)), axis=1)
    ext = codes.reshape(-1, 64)[np.arange(len(d)), amax_idx]
    assert np.all(np.abs(ext) >= 126), "the group maximum codes at (or next to, after fp16 rounding) +-127"
    assert np.all(np.abs(codes.astype(np.int32)) <= 127)


def test_int8_brute_force_nearest_ties_even(orc):
    # every code equals argmin_q |x - q*d16| over q in [-127, 127], ties to the
    # even q, whenever x/d16 is not within fp32 rounding of a half-integer
    x = _bf16_inputs(2, 64 * 60, 3.0)
    # plant exact ties: values that are (k + 1/2) * d16 exactly
    codes, scales = orc.quant_int8(x)
    for g in range(60):
        d16 = Fraction(float(orc.half_value(scales[g:g + 1])[0]))
        for i in range(64):
            xi = Fraction(float(x[64 * g + i]))
            best = min(range(-127, 128), key=lambda q: (abs(xi - q * d16), q % 2))
            r = xi / d16
            near_tie = abs(abs(r - int(r)) - Fraction(1, 2)) < Fraction(1, 1 << 18)
            if not near_tie:
                assert int(codes[64 * g + i]) == best


def test_int8_exact_ties_go_to_even(orc):
    # group: one value 127*d (sets d16 = d exactly representable), others (k+1/2)*d
    d = 2.0 ** -4
    x = np.zeros(64, np.float32)
    x[0] = 127 * d
    ks = np.arange(-30, 33)
    x[1:] = ((ks + 0.5) * d).astype(np.float32)
    codes, scales = orc.quant_int8(x)
    assert orc.half_value(scales)[0] == d
    expect = [k if k % 2 == 0 else k + 1 for k in ks]   # nearest even of k + 1/2
    assert list(codes[1:].astype(int)) == expect


def test_int8_zero_group(orc):
    codes, scales = orc.quant_int8(np.zeros(64, np.float32))
    assert np.all(codes == 0) and scales[0] == 0


# ---------------------------------------------------------------- FWHT-256
def test_fwht_matches_sylvester_hadamard(orc):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(256).astype(np.float64)
    # columns of the oracle transform times 16 are exactly the +-1 Hadamard matrix
    cols = np.stack([orc.fwht256(np.eye(256, dtype=np.float32)[j]) for j in range(256)], axis=1) * 16
    assert np.array_equal(cols, H)
    assert np.array_equal(H @ H.T, 256 * np.eye(256))
    x = _bf16_inputs(3, 256, 2.0)
    y = orc.fwht256(x).astype(np.float64)
    dense = H @ x.astype(np.float64) / 16
    assert np.max(np.abs(y - dense)) <= 1e-6 * np.max(np.abs(dense))
    twice = orc.fwht256(orc.fwht256(x))
    assert np.max(np.abs(twice - x)) <= 1e-6 * np.max(np.abs(x))
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) <= 1e-6 * np.linalg.norm(x)
    assert np.allclose(orc.fwht256_f64(orc.fwht256_f64(x.astype(np.float64))), x, atol=1e-12)


# ---------------------------------------------------------------- q4_0
def test_q4_codes_brute_force_and_bounds(orc):
    x = np.concatenate([orc.fwht256(v) for v in _bf16_inputs(4, 256 * 40, 1.0).reshape(40, 256)])
    nib, d = orc.quant_q4(x)
    dv = orc.half_value(d)
    q = np.empty(x.size, np.int64)
    blk = nib.reshape(-1, 16)
    qb = q.reshape(-1, 32)
    qb[:, :16] = blk & 15
    qb[:, 16:] = blk >> 4
    assert q.min() >= 0 and q.max() <= 15
    xb = x.reshape(-1, 32).astype(np.float64)
    for g in range(xb.shape[0]):
        # the extreme element: sign of d opposite to it, decodes to -8*d16
        m_idx = int(np.argmax(np.abs(xb[g])))
        assert qb[g, m_idx] == 0
        assert np.sign(dv[g]) == -np.sign(xb[g, m_idx])
        for i in range(32):
            r = Fraction(float(x[32 * g + i])) / Fraction(float(dv[g])) + Fraction(17, 2)
            expect = min(15, int(r))  # trunc of a positive value
            frac = r - int(r)
            if frac > Fraction(1, 1 << 16) and frac < 1 - Fraction(1, 1 << 16):
                assert qb[g, i] == expect
    xd = (qb - 8) * dv[:, None]
    err = np.abs(xd - xb)
    top = (xb / dv[:, None]) > 7.5           # values clamped at code 15
    assert np.all(err[~top] <= np.abs(dv[:, None]).repeat(32, 1)[~top] / 2 * (1 + 1e-6))
    assert np.all(err[top] <= np.abs(dv[:, None]).repeat(32, 1)[top] * (1 + 1e-6))


def test_q4_first_index_tie_and_zero(orc):
    x = np.zeros(32, np.float32)
    x[3], x[7] = -2.0, 2.0      # equal magnitude: the first one (-2) is the signed max
    nib, d = orc.quant_q4(x)
    assert orc.half_value(d)[0] == 0.25      # -2 / -8
    nib0, d0 = orc.quant_q4(np.zeros(32, np.float32))
    # m = +0 gives d = 0 / -8 = -0: the stored scale is the fp16 negative zero
    assert d0[0] == 0x8000 and np.all(nib0 == 0x88)


# ---------------------------------------------------------------- quaternion
def test_quaternion_hamilton_rules(orc):
    one, i, j, k = np.eye(4, dtype=np.float32)
    neg = lambda v: (-v).astype(np.float32)
    assert np.array_equal(orc.qmul(i, j), k)
    assert np.array_equal(orc.qmul(j, k), i)
    assert np.array_equal(orc.qmul(k, i), j)
    assert np.array_equal(orc.qmul(j, i), neg(k))
    for u in (i, j, k):
        assert np.array_equal(orc.qmul(u, u), neg(one))
    ijk = orc.qmul(orc.qmul(i, j), k)
    assert np.array_equal(ijk, neg(one))
    rng = np.random.default_rng(5)
    for _ in range(50):
        p, v, w = rng.standard_normal((3, 4)).astype(np.float32)
        pv = orc.qmul(p, v).astype(np.float64)
        # |p v| = |p| |v|
        assert abs(np.linalg.norm(pv) - np.linalg.norm(p) * np.linalg.norm(v)) < 1e-5 * np.linalg.norm(pv)
        # associativity
        a = orc.qmul(orc.qmul(p, v), w).astype(np.float64)
        b = orc.qmul(p, orc.qmul(v, w)).astype(np.float64)
        assert np.allclose(a, b, rtol=1e-5, atol=1e-5)
        # conjugate undoes a unit rotation
        u = (p / np.linalg.norm(p)).astype(np.float32)
        uc = np.array([u[0], -u[1], -u[2], -u[3]], np.float32)
        back = orc.qmul(uc, orc.qmul(u, v))
        assert np.allclose(back, v, atol=1e-5)
    assert np.array_equal(orc.qmul(one, v), v)


def test_left_multiplication_matrix_orthogonal(orc):
    u = synth.unit_quaternion(0)
    Lm = np.stack([orc.qmul(u, e) for e in np.eye(4, dtype=np.float32)], axis=1).astype(np.float64)
    assert np.allclose(Lm.T @ Lm, np.eye(4), atol=1e-6)
