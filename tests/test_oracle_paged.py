"""Pins of the oracle's paged append, gather, decode and extend attention:
closed forms, brute force in 50-digit arithmetic, invariants (page-table
permutation, split-K merge), and the pages' byte accounting."""

import json
import os

import numpy as np
import pytest

from quantized_paged_kv_append_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMTS = [0, 1, 2, 3, 4, 5, 6]
DIMS = {0: 256, 1: 256, 2: 128, 3: 128, 4: 256, 5: 128, 6: 256}


def _pool(orc, fmt, L, hkv, d, seed=0, shuffle=True, outliers=True, B=1):
    P = 16
    pages = [(L + P - 1) // P] * B
    table, npages = synth.page_table(seed, pages, shuffle=shuffle)
    quat = synth.unit_quaternion(seed)
    pool = orc.Pool(fmt, npages, hkv, d, quat=quat)
    k = synth.tensor_bf16(seed, "k", (B * L, hkv, d), outlier_scale=20.0 if outliers else 0.0)
    v = synth.tensor_bf16(seed, "v", (B * L, hkv, d))
    seq = np.repeat(np.arange(B), L).astype(np.int32)
    pos = np.tile(np.arange(L), B).astype(np.int32)
    assert pool.append(k, v, seq, pos, table) == 0
    return pool, table, k, v


@pytest.mark.parametrize("fmt", FMTS)
def test_append_gather_equals_direct_quantization(orc, fmt):
    d = DIMS[fmt]
    pool, table, k, v = _pool(orc, fmt, 37, 2, d)
    kg, vg = pool.gather_dequant(table, 0, 37)
    for t in (0, 15, 16, 36):
        for h in range(2):
            for st, src, got in ((0, k, kg), (1, v, vg)):
                x = synth.bf16_to_f32(src[t, h])
                code, scale = orc.quant_vector(fmt, st, x, pool.quat)
                ref = orc.dequant_vector(fmt, st, d, code, scale, pool.quat)
                assert np.array_equal(got[t, h], ref)


@pytest.mark.parametrize("fmt", FMTS)
def test_page_table_permutation_invariance(orc, fmt):
    d = DIMS[fmt]
    L = 70
    a, ta, _, _ = _pool(orc, fmt, L, 2, d, seed=1, shuffle=False)
    b, tb, _, _ = _pool(orc, fmt, L, 2, d, seed=1, shuffle=True)
    assert not np.array_equal(ta, tb)
    # the planes hold the same rows, only at permuted pages
    rows_a = a.kc.reshape(a.num_pages, -1)
    rows_b = b.kc.reshape(b.num_pages, -1)
    for lp in range(ta.shape[1]):
        assert np.array_equal(rows_a[ta[0, lp]], rows_b[tb[0, lp]])
    q = synth.tensor_bf16(1, "q", (1, 4, d))
    oa = a.decode(q, ta, np.array([L], np.int32), 1 / np.sqrt(d))
    ob = b.decode(q, tb, np.array([L], np.int32), 1 / np.sqrt(d))
    assert np.array_equal(oa, ob)


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_brute_force_mpmath(orc, fmt):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    d = DIMS[fmt]
    L, hkv, hq = 21, 2, 4
    pool, table, _, _ = _pool(orc, fmt, L, hkv, d, seed=3)
    q = synth.tensor_bf16(3, "q", (1, hq, d))
    scale = float(np.float32(1 / np.sqrt(d)))   # the softmax scale is an fp32 argument
    out = pool.decode(q, table, np.array([L], np.int32), scale)
    K, V = pool.gather_dequant(table, 0, L)
    qf = synth.bf16_to_f32(q)[0].astype(np.float64)
    for h in range(hq):
        g = h // (hq // hkv)
        s = [mp.mpf(float(scale)) * mp.fsum(mp.mpf(float(a)) * mp.mpf(float(b)) for a, b in zip(qf[h], K[t, g]))
             for t in range(L)]
        w = [mp.e ** si for si in s]
        Z = mp.fsum(w)
        for i in (0, d // 3, d - 1):
            ref = mp.fsum(wi * mp.mpf(float(V[t, g, i])) for t, wi in enumerate(w)) / Z
            assert abs(float(ref) - out[0, h, i]) < 1e-12


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_closed_forms(orc, fmt):
    d = DIMS[fmt]
    hkv, hq = 2, 8
    pool, table, _, _ = _pool(orc, fmt, 16, hkv, d, seed=4)
    K, V = pool.gather_dequant(table, 0, 16)
    q = synth.tensor_bf16(4, "q", (1, hq, d))
    # one cached token: the output is that token's dequantized V, per KV head
    o1 = pool.decode(q, table, np.array([1], np.int32), 0.0625)
    for h in range(hq):
        assert np.array_equal(o1[0, h], V[0, h // (hq // hkv)])
    # scale 0: uniform softmax -> mean of the dequantized V rows
    o0 = pool.decode(q, table, np.array([16], np.int32), 0.0)
    for h in range(hq):
        assert np.allclose(o0[0, h], V[:, h // (hq // hkv)].mean(axis=0), rtol=0, atol=1e-13)
    # two tokens: weights are the logistic function of the score difference
    o2 = pool.decode(q, table, np.array([2], np.int32), 0.05)
    qf = synth.bf16_to_f32(q)[0].astype(np.float64)
    for h in range(hq):
        g = h // (hq // hkv)
        ds = float(np.float32(0.05)) * (qf[h] @ K[0, g] - qf[h] @ K[1, g])
        w0 = 1 / (1 + np.exp(-ds))
        assert np.allclose(o2[0, h], w0 * V[0, g] + (1 - w0) * V[1, g], atol=1e-12)


def test_decode_gqa_head_mapping(orc):
    # K all equal -> uniform weights; V of KV head g is the constant (g+1)*0.5.
    # Query head h must read KV head h // (Hq/Hkv).
    d, hkv, hq, L = 256, 4, 8, 5
    table, npages = synth.page_table(0, [1], shuffle=False)
    pool = orc.Pool(0, npages, hkv, d)
    k = np.tile(synth.bf16_bits(np.full(d, 0.5, np.float32)), (L, hkv, 1))
    v = np.stack([np.stack([synth.bf16_bits(np.full(d, (g + 1) * 0.5, np.float32)) for g in range(hkv)])] * L)
    pool.append(k, v, np.zeros(L, np.int32), np.arange(L, dtype=np.int32), table)
    q = synth.tensor_bf16(0, "q", (1, hq, d))
    out = pool.decode(q, table, np.array([L], np.int32), 0.1)
    for h in range(hq):
        # int8 codes the constant to within half a scale step (c/254)
        assert np.allclose(out[0, h], (h // 2 + 1) * 0.5, atol=(h // 2 + 1) * 0.5 / 254)


@pytest.mark.parametrize("fmt", FMTS)
def test_split_merge_equals_unsplit(orc, fmt):
    d = DIMS[fmt]
    L = 100
    pool, table, _, _ = _pool(orc, fmt, L, 2, d, seed=5)
    q = synth.tensor_bf16(5, "q", (1, 4, d))
    full = pool.decode(q, table, np.array([L], np.int32), 1 / np.sqrt(d))[0]
    for bounds in ([0, 100], [0, 1, 100], [0, 16, 17, 64, 99, 100], list(range(0, 101, 10))):
        sp = pool.decode_split(q[0], table, L, 1 / np.sqrt(d), bounds)
        assert np.max(np.abs(sp - full)) <= 1e-12


def test_decode_empty_sequence_is_zero(orc):
    pool, table, _, _ = _pool(orc, 0, 16, 2, 256, seed=6)
    q = synth.tensor_bf16(6, "q", (1, 2, 256))
    out = pool.decode(q, table, np.array([0], np.int32), 0.0625)
    assert np.all(out == 0)


@pytest.mark.parametrize("fmt", FMTS)
def test_extend_reduces_to_decode_and_dense(orc, fmt):
    d = DIMS[fmt]
    hkv, hq, L0, T = 2, 4, 40, 6
    pool, table, kpre, vpre = _pool(orc, fmt, L0 + T, hkv, d, seed=7)
    # a fresh pool holding only the prefix
    pre = orc.Pool(fmt, pool.num_pages, hkv, d, quat=pool.quat)
    pre.append(kpre[:L0], vpre[:L0], np.zeros(L0, np.int32), np.arange(L0, dtype=np.int32), table)
    q = synth.tensor_bf16(7, "q", (T, hq, d))
    kn, vn = kpre[L0:], vpre[L0:]
    cu = np.array([0, T], np.int32)
    ext = pre.extend(q, kn, vn, cu, np.array([L0], np.int32), table, 1 / np.sqrt(d), causal=True)
    # token 0 of the chunk with an empty... compare against dense attention over
    # [dequantized prefix ; raw bf16 new tokens j <= i]
    K, V = pre.gather_dequant(table, 0, L0)
    knf = synth.bf16_to_f32(kn).astype(np.float64)
    vnf = synth.bf16_to_f32(vn).astype(np.float64)
    qf = synth.bf16_to_f32(q).astype(np.float64)
    for i in range(T):
        for h in range(hq):
            g = h // (hq // hkv)
            keys = np.concatenate([K[:, g], knf[:i + 1, g]])
            vals = np.concatenate([V[:, g], vnf[:i + 1, g]])
            s = keys @ qf[i, h] * float(np.float32(1 / np.sqrt(d)))
            p = np.exp(s - s.max())
            ref = (p @ vals) / p.sum()
            assert np.allclose(ext[i, h], ref, atol=1e-12, rtol=0)
    # non-causal: every token sees all T new tokens
    nc = pre.extend(q, kn, vn, cu, np.array([L0], np.int32), table, 1 / np.sqrt(d), causal=False)
    assert np.allclose(nc[T - 1], ext[T - 1], atol=1e-13)
    # rows subset gives the same rows
    sub = pre.extend(q, kn, vn, cu, np.array([L0], np.int32), table, 1 / np.sqrt(d), rows=np.array([4, 1], np.int32))
    assert np.array_equal(sub[0], ext[4]) and np.array_equal(sub[1], ext[1])


def test_extend_with_empty_prefix_is_dense_causal(orc):
    d, hkv, hq, T = 256, 2, 4, 9
    table, npages = synth.page_table(8, [1], shuffle=False)
    pool = orc.Pool(0, npages, hkv, d)
    q = synth.tensor_bf16(8, "q", (T, hq, d))
    kn = synth.tensor_bf16(8, "k_new", (T, hkv, d))
    vn = synth.tensor_bf16(8, "v_new", (T, hkv, d))
    out = pool.extend(q, kn, vn, np.array([0, T], np.int32), np.array([0], np.int32), table, 0.0625)
    vnf = synth.bf16_to_f32(vn).astype(np.float64)
    for h in range(hq):
        assert np.array_equal(out[0, h], vnf[0, h // 2])   # first token attends only itself


def test_byte_accounting_matches_pages(orc):
    g = json.load(open(os.path.join(GOLDEN, "byte_accounting.json")))
    int8_k = sum(orc.row_bytes(0, 0, 256))
    int8_v = sum(orc.row_bytes(0, 1, 256))
    q4_v = sum(orc.row_bytes(1, 1, 256))
    assert 2 * int8_k == g["int8_cell_bytes_head_dim_256"]["value"]
    assert 2 * (int8_k + int8_v) == g["int8_pair_cell_bytes"]["value"]
    assert 2 * (int8_k + q4_v) == g["k8v4_cell_bytes"]["value"]
    assert q4_v == g["q4_v_bytes_per_head_cell"]["value"]
    assert orc.row_bytes(0, 1, 256)[0] == g["int8_v_bytes_per_head_cell"]["value"]
    assert 2 * 2 * 256 * 4 == g["fp32_cell_bytes_head_dim_256"]["value"] * 2
    # q4_0 for both stores (the q4_0 format): 18 B per 32 values, K and V
    q4_k4, q4_v4 = sum(orc.row_bytes(orc.FMT_Q4, 0, 256)), sum(orc.row_bytes(orc.FMT_Q4, 1, 256))
    assert 2 * 2 * q4_v == g["q4_0_pair_cell_bytes"]["value"] == 2 * (q4_k4 + q4_v4)
    # one store quantized: int8 on one side, the bf16 input values (no scale row) on the other
    assert orc.row_bytes(orc.FMT_K8, 0, 256) == orc.row_bytes(0, 0, 256)
    assert orc.row_bytes(orc.FMT_K8, 1, 256) == (512, 0) == orc.row_bytes(orc.FMT_V8, 0, 256)
    assert orc.row_bytes(orc.FMT_V8, 1, 256) == orc.row_bytes(0, 1, 256)
    iso3 = sum(orc.row_bytes(2, 0, 128))
    iso4 = sum(orc.row_bytes(3, 0, 128))
    assert iso3 == g["iso3_block_bytes"]["value"] and iso4 == g["iso4_block_bytes"]["value"]
    assert iso3 * 8 / 128 == g["iso3_block_bytes"]["bits_per_value"]
    assert iso4 * 8 / 128 == g["iso4_block_bytes"]["bits_per_value"]
    e = g["bf16_vs_iso3_bytes_per_token_10_layers"]
    per_layer_iso3 = 2 * e["kv_heads"] * sum(orc.row_bytes(2, 0, e["head_dim"]))
    assert e["layers"] * per_layer_iso3 == e["iso3"]
    assert e["layers"] * 2 * e["kv_heads"] * e["head_dim"] * 2 == e["bf16"]
    c = g["compression_vs_bf16"]
    assert round(256 / iso3, 1) == c["iso3"] and round(256 / iso4, 1) == c["iso4"]
    kv = g["kv_bytes_131k_ctx_gb"]
    for name, per_tok in (("int8", 2 * (int8_k + int8_v)), ("k8v4", 2 * (int8_k + q4_v))):
        assert round(per_tok * kv["layers_reading"] * kv["tokens"] / 1e9, 2) == kv[name]


def test_append_reports_bad_page_entries(orc):
    table, npages = synth.page_table(0, [2], shuffle=False)
    pool = orc.Pool(0, npages, 2, 256)
    bad = table.copy()
    bad[0, 1] = npages + 5
    k = synth.tensor_bf16(0, "k", (20, 2, 256))
    skipped = pool.append(k, k, np.zeros(20, np.int32), np.arange(20, dtype=np.int32), bad)
    assert skipped == 4   # positions 16..19 fall on the bad page


@pytest.mark.parametrize("fmt", FMTS)
def test_verify_window_of_one_is_decode(orc, fmt):
    """A verify window of one query per sequence is plain decode."""
    d = DIMS[fmt]
    pool, table, _, _ = _pool(orc, fmt, 90, 2, d, seed=11, B=3)
    q = synth.tensor_bf16(11, "q", (3, 8, d))
    lens = np.array([90, 17, 64], np.int32)
    cu = np.arange(4, dtype=np.int32)
    ver = pool.verify(q, table, lens, cu, float(np.float32(1 / np.sqrt(d))))
    dec = pool.decode(q, table, lens, float(np.float32(1 / np.sqrt(d))))
    assert np.array_equal(ver, dec)


def test_verify_equals_extend_on_a_lossless_window(orc):
    """Window tokens whose int8 packing is lossless (values c / 8 with |c| <= 127
    and one |c| = 127 per 64-value group, so the scale is exactly 1/8): reading
    them back from the pool (verify) must give what extend gives when it takes
    them as raw bf16 new tokens after the same packed prefix."""
    d, hkv, hq, L0, W = 256, 2, 8, 70, 5
    rng = np.random.default_rng(3)
    codes = rng.integers(-127, 128, size=(W, 2, hkv, d))
    codes[..., ::64] = 127 * np.where(rng.random(codes[..., ::64].shape) < 0.5, -1, 1)
    win = (codes / 8.0).astype(np.float32)
    win_bits = (win.view(np.uint32) >> 16).astype(np.uint16)      # exact in bf16
    assert np.array_equal(synth.bf16_to_f32(win_bits), win)
    pre_k = synth.tensor_bf16(3, "k", (L0, hkv, d), outlier_scale=20.0)
    pre_v = synth.tensor_bf16(3, "v", (L0, hkv, d))
    table, npages = synth.page_table(3, [(L0 + W + 15) // 16])
    full = orc.Pool(0, npages, hkv, d)
    full.append(np.concatenate([pre_k, win_bits[:, 0]]), np.concatenate([pre_v, win_bits[:, 1]]),
                np.zeros(L0 + W, np.int32), np.arange(L0 + W, dtype=np.int32), table)
    pre = orc.Pool(0, npages, hkv, d)
    pre.append(pre_k, pre_v, np.zeros(L0, np.int32), np.arange(L0, dtype=np.int32), table)
    q = synth.tensor_bf16(3, "q", (W, hq, d))
    scale = 0.0625
    ver = full.verify(q, table, np.array([L0 + W], np.int32), np.array([0, W], np.int32), scale)
    ext = pre.extend(q, win_bits[:, 0], win_bits[:, 1], np.array([0, W], np.int32), np.array([L0], np.int32),
                     table, scale, causal=True)
    assert np.allclose(ver, ext, rtol=0, atol=1e-12)


def test_verify_rejects_window_longer_than_sequence(orc):
    pool, table, _, _ = _pool(orc, 0, 10, 2, 256, seed=12)
    q = synth.tensor_bf16(12, "q", (4, 2, 256))
    with pytest.raises(ValueError):
        pool.verify(q, table, np.array([3], np.int32), np.array([0, 4], np.int32), 0.0625)
