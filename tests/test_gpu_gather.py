"""GPU parity of kv_gather_dequant (pool -> dense fp32 K and V of one sequence)
against the oracle's gather and dequantization (double precision).

int8 rows (c * d16, exact in fp32) must match bit for bit; k8v4 V (rotated back
by an fp32 FWHT-256) and ISO rows (fp32 quaternion products) within 1e-6 of the
row's largest magnitude."""

import numpy as np
import pytest

from _workload import Workload, gpu_cache, to_dev

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


def _check(got, ref, exact):
    got = np.asarray(got, np.float64)
    if exact:
        assert np.array_equal(got, ref.astype(np.float32).astype(np.float64))
    else:
        scale = np.maximum(np.abs(ref).max(axis=-1, keepdims=True), 1e-30)
        assert np.all(np.abs(got - ref) <= 1e-6 * scale), np.abs(got - ref).max()


@pytest.mark.parametrize("fmt,lens,hkv,d", [
    ("int8", [37, 300], 2, 256),
    ("int8", [129], 4, 128),
    ("k8v4", [200, 17], 2, 256),
    ("iso3", [150], 4, 128),
    ("iso4", [61], 4, 128),
    ("iso3", [90], 2, 256),
    ("iso4", [45], 2, 256),
    ("q4", [200, 17], 2, 256),
    ("k8vbf16", [37, 300], 2, 256),
    ("kbf16v8", [129], 4, 128),
])
def test_gather_matches_oracle(env, orc, fmt, lens, hkv, d):
    torch, qkv = env
    w = Workload(fmt, lens, hkv, 16, d, seed=51)
    pool = w.oracle_pool(orc)
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    table = to_dev(w.table, torch)
    for b, L in enumerate(lens):
        k, v = qkv.gather_dequant(cache, table[b], L)
        torch.cuda.synchronize()
        kr, vr = pool.gather_dequant(w.table, b, L)
        _check(k.cpu().numpy(), kr, exact=fmt in ("int8", "k8v4", "k8vbf16", "kbf16v8"))
        _check(v.cpu().numpy(), vr, exact=fmt in ("int8", "k8vbf16", "kbf16v8"))
    assert qkv.device_error() == 0


def test_gather_k8v4_full_size(env, orc):
    """The k8v4 benchmark length (118750 tokens, Hkv 2, D 256)."""
    torch, qkv = env
    w = Workload("k8v4", [118750], 2, 16, 256, seed=0)
    pool = w.oracle_pool(orc)
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    k, v = qkv.gather_dequant(cache, to_dev(w.table, torch)[0], 118750)
    torch.cuda.synchronize()
    kr, vr = pool.gather_dequant(w.table, 0, 118750)
    _check(k.cpu().numpy(), kr, exact=True)
    _check(v.cpu().numpy(), vr, exact=False)


def test_gather_bad_page_entry_gives_zero_rows(env, orc):
    torch, qkv = env
    w = Workload("int8", [40], 2, 16, 256, seed=52)
    pool = w.oracle_pool(orc)
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    row = np.array(w.table[0], np.int32)
    row[1] = w.num_pages + 5   # positions 16..31
    qkv.device_error(clear=True)
    k, v = qkv.gather_dequant(cache, to_dev(row, torch), 40)
    torch.cuda.synchronize()
    assert qkv.device_error() & 1
    kr, vr = pool.gather_dequant(w.table, 0, 40)
    k, v = k.cpu().numpy(), v.cpu().numpy()
    assert np.all(k[16:32] == 0) and np.all(v[16:32] == 0)
    _check(k[:16], kr[:16], exact=True)
    _check(v[32:], vr[32:], exact=True)
