"""GPU parity of extend (prefill-chunk) attention over a packed prefix plus
bf16 new tokens, against the CPU oracle (double precision). Tolerance as for
decode: fp32 output within max-abs 2e-3 and cosine > 0.9999."""

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


def _case(orc, prefix, chunk, hkv, hq, d, seed, spare_pages=2, fmt="int8"):
    """Pool of format `fmt` holding `prefix[b]` packed tokens per sequence (table
    sized for prefix + chunk), plus the chunk's bf16 q / k_new / v_new."""
    total_pages = [max(1, (p + c + 15) // 16) for p, c in zip(prefix, chunk)]
    w = Workload(fmt, prefix, hkv, hq, d, seed=seed)
    table, npages = synth.page_table(seed, total_pages, num_pages=sum(total_pages) + spare_pages)
    w.table, w.num_pages = table, npages
    pool = orc.Pool(w.fmt, npages, hkv, d, quat=w.quat)
    if w.seq_id.size:
        pool.append(w.k, w.v, w.seq_id, w.pos, table)
    T = int(sum(chunk))
    q = synth.tensor_bf16(seed, "q", (T, hq, d))
    kn = synth.tensor_bf16(seed, "k_new", (T, hkv, d), outlier_scale=20.0)
    vn = synth.tensor_bf16(seed, "v_new", (T, hkv, d))
    cu = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    return w, pool, table, q, kn, vn, cu, np.asarray(prefix, np.int32)


def _run(torch, qkv, w, pool, table, q, kn, vn, cu, pre, causal=True, out_dtype=None, scale=None):
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    chunk = np.diff(cu)
    out = qkv.extend(cache, bf16_dev(q, torch), bf16_dev(kn, torch), bf16_dev(vn, torch), to_dev(cu, torch),
                     to_dev(pre, torch), to_dev(table, torch), int(chunk.max()), scale=scale, causal=causal,
                     out_dtype=out_dtype or torch.float32)
    torch.cuda.synchronize()
    assert qkv.device_error() == 0
    return out.float().cpu().numpy()


@pytest.mark.parametrize("prefix,chunk,hkv,hq,d", [
    ([100], [37], 2, 16, 256),
    ([0], [45], 2, 16, 256),
    ([64], [64], 2, 16, 256),
    ([0, 200, 33], [20, 70, 1], 2, 16, 256),
    ([150], [40], 2, 8, 256),
    ([90], [33], 4, 4, 128),
    ([77], [19], 2, 32, 128),
    ([130], [50], 1, 2, 256),
])
def test_extend_small(env, orc, prefix, chunk, hkv, hq, d):
    torch, qkv = env
    w, pool, table, q, kn, vn, cu, pre = _case(orc, prefix, chunk, hkv, hq, d, seed=41)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    ref = pool.extend(q, kn, vn, cu, pre, table, scale, causal=True)
    got = _run(torch, qkv, w, pool, table, q, kn, vn, cu, pre, scale=scale)
    r = compare_attention(got, ref)
    assert r["ok"], r


@pytest.mark.parametrize("fmt,prefix,chunk,hkv,hq,d", [
    ("k8v4", [100], [37], 2, 16, 256),
    ("k8v4", [0, 200, 33], [20, 70, 1], 2, 16, 256),
    ("iso3", [90], [33], 4, 16, 128),
    ("iso4", [90], [33], 4, 16, 128),
    ("iso3", [0, 150, 64], [17, 40, 64], 4, 16, 128),
    ("iso4", [130], [50], 2, 16, 128),
    ("iso3", [77], [19], 2, 32, 128),
    ("iso4", [60], [25], 4, 4, 128),
    ("q4", [100], [37], 2, 16, 256),
    ("q4", [0, 200, 33], [20, 70, 1], 2, 16, 256),
    ("k8vbf16", [100], [37], 2, 16, 256),
    ("k8vbf16", [90], [33], 4, 4, 128),
    ("kbf16v8", [0, 150, 64], [17, 40, 64], 2, 16, 256),
    ("kbf16v8", [77], [19], 2, 32, 128),
])
def test_extend_formats(env, orc, fmt, prefix, chunk, hkv, hq, d):
    """k8v4 (V rotated back from the FWHT domain) and ISO3 / ISO4 (raw levels as
    keys against the rotated query; V rotated back by the conjugate quaternion)
    prefixes, with the x20 K outlier channels."""
    torch, qkv = env
    w, pool, table, q, kn, vn, cu, pre = _case(orc, prefix, chunk, hkv, hq, d, seed=44, fmt=fmt)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    ref = pool.extend(q, kn, vn, cu, pre, table, scale, causal=True)
    got = _run(torch, qkv, w, pool, table, q, kn, vn, cu, pre, scale=scale)
    r = compare_attention(got, ref)
    assert r["ok"], r


@pytest.mark.parametrize("fmt,hkv,d", [("k8v4", 2, 256), ("iso3", 4, 128), ("iso4", 4, 128), ("q4", 2, 256),
                                       ("k8vbf16", 2, 256), ("kbf16v8", 2, 256)])
def test_extend_formats_long_prefix_sampled(env, orc, fmt, hkv, d):
    """A 256-token chunk over an 8192-token prefix (Hq 16); the oracle computes a
    sample of rows one by one."""
    torch, qkv = env
    w, pool, table, q, kn, vn, cu, pre = _case(orc, [8192], [256], hkv, 16, d, seed=45, fmt=fmt)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    got = _run(torch, qkv, w, pool, table, q, kn, vn, cu, pre, scale=scale)
    rows = np.array([0, 1, 63, 64, 200, 255], np.int32)
    ref = pool.extend(q, kn, vn, cu, pre, table, scale, causal=True, rows=rows)
    r = compare_attention(got[rows], ref)
    assert r["ok"], r


def test_extend_non_causal_and_bf16(env, orc):
    torch, qkv = env
    w, pool, table, q, kn, vn, cu, pre = _case(orc, [120, 5], [30, 66], 2, 16, 256, seed=42)
    scale = float(np.float32(1.0 / 16))
    ref = pool.extend(q, kn, vn, cu, pre, table, scale, causal=False)
    got = _run(torch, qkv, w, pool, table, q, kn, vn, cu, pre, causal=False, scale=scale)
    assert compare_attention(got, ref)["ok"]
    refc = pool.extend(q, kn, vn, cu, pre, table, scale, causal=True)
    gotb = _run(torch, qkv, w, pool, table, q, kn, vn, cu, pre, out_dtype=torch.bfloat16, scale=scale)
    r = compare_attention(gotb, refc, bf16=True)
    assert r["ok"], r


def test_extend_serving_chunk_sampled(env, orc):
    """The serving-step chunk: 2048 new tokens over a 32768-token prefix,
    Hq 16 / Hkv 2, D 256; the oracle computes a sample of rows one by one."""
    torch, qkv = env
    w, pool, table, q, kn, vn, cu, pre = _case(orc, [32768], [2048], 2, 16, 256, seed=0)
    scale = float(np.float32(1.0 / 16))
    got = _run(torch, qkv, w, pool, table, q, kn, vn, cu, pre, scale=scale)
    rows = np.array([0, 1, 15, 16, 127, 128, 1000, 2046, 2047], np.int32)
    ref = pool.extend(q, kn, vn, cu, pre, table, scale, causal=True, rows=rows)
    r = compare_attention(got[rows], ref)
    assert r["ok"], r


def test_extend_then_deferred_pack_matches_oracle(env, orc):
    """After extend, the chunk is packed with append (deferred packing): the
    planes equal the oracle's append of prefix + chunk."""
    torch, qkv = env
    w, pool, table, q, kn, vn, cu, pre = _case(orc, [40], [30], 2, 16, 256, seed=43)
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    qkv.extend(cache, bf16_dev(q, torch), bf16_dev(kn, torch), bf16_dev(vn, torch), to_dev(cu, torch),
               to_dev(pre, torch), to_dev(table, torch), 30)
    seq = np.zeros(30, np.int32)
    pos = (40 + np.arange(30)).astype(np.int32)
    qkv.append(cache, bf16_dev(kn, torch), bf16_dev(vn, torch), to_dev(seq, torch), to_dev(pos, torch),
               to_dev(table, torch))
    torch.cuda.synchronize()
    pool.append(kn, vn, seq, pos, table)
    for g, r in zip([p.cpu().numpy() for p in cache.planes()], pool.planes()):
        assert np.array_equal(g, r)


def test_extend_rejects_unsupported_gqa(env):
    """num_q_heads / num_kv_heads = 3 is outside {1, 2, 4, 8k}: QKV_ERR_GQA, nothing launched."""
    torch, qkv = env
    c = qkv.PagedKVCache("k8v4", 4, 2, 256)
    z = torch.zeros((4, 6, 256), dtype=torch.bfloat16, device="cuda")
    zk = torch.zeros((4, 2, 256), dtype=torch.bfloat16, device="cuda")
    i32 = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    with pytest.raises(qkv.QkvError) as e:
        qkv.extend(c, z, zk, zk, i32([0, 4]), i32([0]), i32([[0, 1, 2, 3]]), 4)
    assert e.value.code == -3


@pytest.mark.parametrize("fmt,prefix,chunk,hkv,hq", [
    ("iso3", [100], [37], 2, 16),
    ("iso4", [0, 150, 64], [17, 40, 64], 2, 16),
    ("iso3", [0], [45], 2, 16),
    ("iso4", [77], [19], 1, 8),
    ("iso3", [130], [50], 2, 4),
])
def test_extend_iso_head_dim_256(env, orc, fmt, prefix, chunk, hkv, hq):
    """ISO extend at head_dim 256 (two 128-value blocks per head, as in the pages'
    model): the rotated query's hi tile shares the query region with the plain
    query, which replaces it once the prefix tiles are done."""
    torch, qkv = env
    w, pool, table, q, kn, vn, cu, pre = _case(orc, prefix, chunk, hkv, hq, 256, seed=46, fmt=fmt)
    scale = float(np.float32(1.0 / 16))
    ref = pool.extend(q, kn, vn, cu, pre, table, scale, causal=True)
    got = _run(torch, qkv, w, pool, table, q, kn, vn, cu, pre, scale=scale)
    r = compare_attention(got, ref)
    assert r["ok"], r


@pytest.mark.parametrize("fmt", ["iso3", "iso4"])
def test_extend_iso_head_dim_256_long_prefix_sampled(env, orc, fmt):
    """A 256-token chunk over an 8192-token ISO prefix at head_dim 256 (Hq 16 / Hkv 2),
    sampled rows against the oracle, fp32 and bf16 output."""
    torch, qkv = env
    w, pool, table, q, kn, vn, cu, pre = _case(orc, [8192], [256], 2, 16, 256, seed=47, fmt=fmt)
    scale = float(np.float32(1.0 / 16))
    got = _run(torch, qkv, w, pool, table, q, kn, vn, cu, pre, scale=scale)
    rows = np.array([0, 1, 63, 64, 200, 255], np.int32)
    ref = pool.extend(q, kn, vn, cu, pre, table, scale, causal=True, rows=rows)
    r = compare_attention(got[rows], ref)
    assert r["ok"], r
    gotb = _run(torch, qkv, w, pool, table, q, kn, vn, cu, pre, scale=scale, out_dtype=torch.bfloat16)
    rb = compare_attention(gotb[rows], ref, bf16=True)
    assert rb["ok"], rb
