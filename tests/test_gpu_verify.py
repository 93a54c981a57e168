"""GPU parity of kv_verify_attn (several decode queries per sequence, query j
of a window of W at position L - W + j) against the oracle's verify window.
Tolerance as for decode: fp32 output within max-abs 2e-3, cosine > 0.9999."""

import numpy as np
import pytest

from _workload import Workload, bf16_dev, compare_attention, gpu_cache, to_dev
from quantized_paged_kv_append_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_paged_kv_append_gb300 as qkv
    from quantized_paged_kv_append_gb300 import build
    build.build()
    return torch, qkv


def _run(torch, qkv, w, pool, windows, out_dtype=None, seed=61):
    cu = np.concatenate([[0], np.cumsum(windows)]).astype(np.int32)
    q = synth.tensor_bf16(seed, "q_verify", (int(cu[-1]), w.hq, w.d))
    ref = pool.verify(q, w.table, w.lens, cu, w.scale)
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    got = qkv.verify(cache, bf16_dev(q, torch), to_dev(cu, torch), to_dev(w.lens, torch), to_dev(w.table, torch),
                     w.max_len(), scale=w.scale, out_dtype=out_dtype or torch.float32)
    torch.cuda.synchronize()
    return got.float().cpu().numpy(), ref


@pytest.mark.parametrize("fmt,d,hkv,hq", [("int8", 256, 2, 16), ("k8v4", 256, 2, 16), ("iso3", 128, 4, 16),
                                          ("iso4", 128, 4, 16), ("int8", 128, 2, 4), ("q4", 256, 2, 16),
                                          ("k8vbf16", 256, 2, 16), ("kbf16v8", 128, 4, 16)])
def test_verify_matches_oracle(env, orc, fmt, d, hkv, hq):
    torch, qkv = env
    w = Workload(fmt, [300, 45, 1000, 17], hkv, hq, d, seed=61)
    pool = w.oracle_pool(orc)
    got, ref = _run(torch, qkv, w, pool, [2, 1, 4, 3])
    assert qkv.device_error() == 0
    r = compare_attention(got, ref)
    assert r["ok"], r


def test_verify_128k_window_and_bf16(env, orc):
    """A window of 3 at the 128K int8 benchmark length, bf16 output."""
    torch, qkv = env
    w = Workload("int8", [131072], 2, 16, 256, seed=0)
    pool = w.oracle_pool(orc)
    got, ref = _run(torch, qkv, w, pool, [3], out_dtype=torch.bfloat16)
    assert qkv.device_error() == 0
    r = compare_attention(got, ref, bf16=True)
    assert r["ok"], r


def test_verify_window_longer_than_sequence_flags(env, orc):
    """W = 5 over a 3-token sequence: the position bit is set, the two queries
    that would sit before position 0 give zero rows, the other three attend as
    usual."""
    torch, qkv = env
    w = Workload("int8", [3, 40], 2, 16, 256, seed=62)
    pool = w.oracle_pool(orc)
    cu = np.array([0, 5, 6], np.int32)
    q = synth.tensor_bf16(62, "q_verify", (6, 16, 256))
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    qkv.device_error(clear=True)
    got = qkv.verify(cache, bf16_dev(q, torch), to_dev(cu, torch), to_dev(w.lens, torch), to_dev(w.table, torch),
                     w.max_len(), scale=w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert qkv.device_error() & 2
    got = got.cpu().numpy()
    assert np.all(got[:2] == 0)
    ref_ok = pool.verify(q[2:], w.table, w.lens, np.array([0, 3, 4], np.int32), w.scale)
    r = compare_attention(got[2:], ref_ok)
    assert r["ok"], r


# ---- the fixed-window verify (kv_verify_attn_fixed): the window's queries as columns of one
# tile pass; expected values from the oracle's verify window with cu_seqlens = b * W ----

def _run_fixed(torch, qkv, w, pool, window, out_dtype=None, seed=63):
    cu = (np.arange(w.B + 1) * window).astype(np.int32)
    q = synth.tensor_bf16(seed, "q_verify_fixed", (w.B * window, w.hq, w.d))
    ref = pool.verify(q, w.table, w.lens, cu, w.scale)
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    qkv.device_error(clear=True)
    got = qkv.verify_fixed(cache, bf16_dev(q, torch), to_dev(w.lens, torch), to_dev(w.table, torch), w.max_len(),
                           window, scale=w.scale, out_dtype=out_dtype or torch.float32)
    torch.cuda.synchronize()
    return got.float().cpu().numpy(), ref


@pytest.mark.parametrize("fmt,d,hkv,hq,window", [
    # int8: 16 query columns a tile pass (window x heads per KV head = 16, 32, 8, 48)
    ("int8", 256, 2, 16, 2), ("int8", 256, 2, 16, 4), ("int8", 256, 2, 16, 1), ("int8", 128, 2, 4, 4),
    ("int8", 256, 1, 16, 3), ("int8", 128, 4, 8, 2),
    # the other formats: 8 columns a pass
    ("k8v4", 256, 2, 16, 2), ("iso3", 128, 4, 16, 3), ("iso4", 128, 4, 16, 2), ("q4", 256, 2, 16, 2),
    ("k8vbf16", 256, 2, 16, 4), ("kbf16v8", 128, 4, 16, 2)])
def test_verify_fixed_matches_oracle(env, orc, fmt, d, hkv, hq, window):
    torch, qkv = env
    w = Workload(fmt, [300, 45, 1000, 17, 129], hkv, hq, d, seed=63)
    pool = w.oracle_pool(orc)
    got, ref = _run_fixed(torch, qkv, w, pool, window)
    assert qkv.device_error() == 0
    r = compare_attention(got, ref)
    assert r["ok"], r


def test_verify_fixed_128k_window_and_bf16(env, orc):
    """A window of 4 at the 128K int8 benchmark length (two 16-column passes), bf16 output."""
    torch, qkv = env
    w = Workload("int8", [131072], 2, 16, 256, seed=0)
    pool = w.oracle_pool(orc)
    got, ref = _run_fixed(torch, qkv, w, pool, 4, out_dtype=torch.bfloat16)
    assert qkv.device_error() == 0
    r = compare_attention(got, ref, bf16=True)
    assert r["ok"], r


def test_verify_fixed_equals_expanded(env, orc):
    """The one-pass window and the expanded one (one decode row per query) agree
    within the fp32 rounding of their different merge orders."""
    torch, qkv = env
    w = Workload("int8", [700, 33, 4096], 2, 16, 256, seed=64)
    pool = w.oracle_pool(orc)
    window = 3
    cu = (np.arange(w.B + 1) * window).astype(np.int32)
    q = bf16_dev(synth.tensor_bf16(64, "q_verify_fixed", (w.B * window, 16, 256)), torch)
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    a = qkv.verify_fixed(cache, q, to_dev(w.lens, torch), to_dev(w.table, torch), w.max_len(), window, scale=w.scale,
                         out_dtype=torch.float32)
    b = qkv.verify(cache, q, to_dev(cu, torch), to_dev(w.lens, torch), to_dev(w.table, torch), w.max_len(),
                   scale=w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert qkv.device_error() == 0
    assert float((a - b).abs().max()) < 2e-3


def test_verify_fixed_window_longer_than_sequence_flags(env, orc):
    """W = 5 over a 3-token sequence (and a 40-token one): the position bit is set,
    the two queries that would sit before position 0 give zero rows, the rest
    attend as the oracle's window does."""
    torch, qkv = env
    w = Workload("int8", [3, 40], 2, 16, 256, seed=65)
    pool = w.oracle_pool(orc)
    window = 5
    q = synth.tensor_bf16(65, "q_verify_fixed", (2 * window, 16, 256))
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    qkv.device_error(clear=True)
    got = qkv.verify_fixed(cache, bf16_dev(q, torch), to_dev(w.lens, torch), to_dev(w.table, torch), w.max_len(),
                           window, scale=w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert qkv.device_error() & 2
    got = got.cpu().numpy()
    assert np.all(got[:2] == 0)
    ref_ok = pool.verify(q[2:], w.table, w.lens, np.array([0, 3, 8], np.int32), w.scale)
    r = compare_attention(got[2:], ref_ok)
    assert r["ok"], r
