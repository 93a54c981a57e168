"""kv_decode_attn_noalloc: decode attention for callers that cannot allocate
device memory (stream capture, memory owned by another pool, allocation-free
loops). It runs the regular decode kernel on a fixed static scratch array, so
its output must match kv_decode_attn with a caller workspace, call after call.

This file sorts last so that a run stopping at the first failure has already
run every other test."""

import ctypes as C

import numpy as np
import pytest

from _workload import Workload, bf16_dev, compare_attention, gpu_cache, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_paged_kv_append_gb300 as qkv
    from quantized_paged_kv_append_gb300 import _lib, build
    build.build()
    return torch, qkv, _lib


def _noalloc(_lib, cache, q, table, lens, max_len, scale, out, torch, k_new=None, v_new=None):
    p = lambda t: C.c_void_p(t.data_ptr()) if t is not None else C.c_void_p(0)
    rc = _lib.lib().kv_decode_attn_noalloc(C.byref(cache.desc), p(q), p(k_new), p(v_new), q.shape[0], q.shape[1],
                                           p(table), int(table.shape[1]), p(lens), int(max_len), float(scale), p(out),
                                           1 if out.dtype == torch.float32 else 0,
                                           C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


@pytest.mark.parametrize("fmt,d,hkv,hq,lens", [("int8", 256, 2, 16, [3000, 17, 450]),
                                               ("k8v4", 256, 2, 16, [1200]),
                                               ("iso3", 128, 4, 16, [700, 64])])
def test_noalloc_matches_workspace_entry_point_twice(env, orc, fmt, d, hkv, hq, lens):
    torch, qkv, _lib = env
    # a larger call first leaves partial slots and merge records all over the scratch
    big = Workload("int8", [20000, 9000, 5000, 3000], 2, 16, 256, seed=52)
    bpool = big.oracle_pool(orc)
    bcache = gpu_cache(qkv, big, torch, planes=bpool.planes())
    bout = torch.empty((big.B, 16, 256), dtype=torch.float32, device="cuda")
    rc = _noalloc(_lib, bcache, bf16_dev(big.q, torch), to_dev(big.table, torch), to_dev(big.lens, torch),
                  big.max_len(), big.scale, bout, torch)
    assert rc == 0, _lib.lib().qkv_strerror(rc)

    w = Workload(fmt, lens, hkv, hq, d, seed=51)
    pool = w.oracle_pool(orc)
    oracle_out = pool.decode(w.q, w.table, w.lens, w.scale)
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    q, table, sl = bf16_dev(w.q, torch), to_dev(w.table, torch), to_dev(w.lens, torch)
    ref = qkv.decode(cache, q, table, sl, w.max_len(), scale=w.scale, out_dtype=torch.float32).cpu().numpy()
    for _ in range(2):
        out = torch.full((w.B, hq, d), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(_lib, cache, q, table, sl, w.max_len(), w.scale, out, torch)
        assert rc == 0, _lib.lib().qkv_strerror(rc)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        # the same kernels over the same inputs in the same order: identical bits
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
        r = compare_attention(got, oracle_out)
        assert r["ok"], r
    assert qkv.device_error() == 0


def test_noalloc_rejects_requests_beyond_the_static_scratch(env):
    torch, qkv, _lib = env
    cache = qkv.PagedKVCache("int8", 64, 8, 256)
    z = torch.zeros((1024, 64, 256), dtype=torch.bfloat16, device="cuda")   # batch 1024 x 8 KV heads
    table = torch.zeros((1024, 4), dtype=torch.int32, device="cuda")
    lens = torch.ones(1024, dtype=torch.int32, device="cuda")
    out = torch.zeros((1024, 64, 256), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(_lib, cache, z, table, lens, 64, 0.0625, out, torch) == -4
