"""GPU parity of paged split-K decode attention against the CPU oracle.

The GPU reads the oracle's own packed planes (so decode is tested independently
of append). Tolerance: fp32 output within max-abs 2e-3 and cosine > 0.9999 of
the oracle's double-precision attention over the same dequantized K/V."""

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
    from quantized_paged_kv_append_gb300 import build
    build.build()
    return torch, qkv


def _run(torch, qkv, w, pool, out_dtype=None, table=None, lens=None, workspace=None, repeat=1):
    out_dtype = out_dtype or torch.float32
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    t = to_dev(w.table if table is None else table, torch)
    sl = to_dev(w.lens if lens is None else lens, torch)
    q = bf16_dev(w.q, torch)
    outs = []
    for _ in range(repeat):
        o = qkv.decode(cache, q, t, sl, max(1, w.max_len()), scale=w.scale, out_dtype=out_dtype, workspace=workspace)
        outs.append(o.float().cpu().numpy())
    torch.cuda.synchronize()
    assert qkv.device_error() == 0
    return outs if repeat > 1 else outs[0]


SMALL = [
    # fmt, D, Hkv, Hq
    ("int8", 256, 2, 16), ("int8", 128, 2, 8), ("int8", 256, 4, 4), ("int8", 256, 1, 2),
    ("int8", 256, 2, 32), ("int8", 128, 1, 16), ("k8v4", 256, 2, 16), ("k8v4", 256, 1, 4),
    ("iso3", 128, 4, 16), ("iso4", 128, 4, 16), ("iso3", 256, 2, 16), ("iso4", 256, 2, 4),
    ("iso4", 128, 2, 2),
    ("q4", 256, 2, 16), ("q4", 256, 1, 4), ("k8vbf16", 256, 2, 16), ("k8vbf16", 128, 4, 16),
    ("kbf16v8", 256, 2, 16), ("kbf16v8", 128, 2, 2),
]


@pytest.mark.parametrize("fmt,d,hkv,hq", SMALL)
def test_decode_small_ragged(env, orc, fmt, d, hkv, hq):
    torch, qkv = env
    w = Workload(fmt, [1, 37, 300, 16, 1000], hkv, hq, d, seed=21)
    pool = w.oracle_pool(orc)
    ref = pool.decode(w.q, w.table, w.lens, w.scale)
    got = _run(torch, qkv, w, pool)
    r = compare_attention(got, ref)
    assert r["ok"], r


@pytest.mark.parametrize("fmt,d,hkv,hq,L", [
    ("int8", 256, 2, 16, 2048),      # tiny config
    ("int8", 256, 2, 16, 131072),    # 128K
    ("k8v4", 256, 2, 16, 118750),
    ("iso3", 128, 4, 16, 81920),
    ("iso4", 128, 4, 16, 81920),
    ("q4", 256, 2, 16, 131072),
    ("k8vbf16", 256, 2, 16, 65536),
    ("kbf16v8", 256, 2, 16, 65536),
    ("int8", 256, 2, 32, 65536),     # 16 query heads per KV head: one 16-column pass (V scales folded)
])
def test_decode_full_size(env, orc, fmt, d, hkv, hq, L):
    torch, qkv = env
    w = Workload(fmt, [L], hkv, hq, d, seed=0)
    pool = w.oracle_pool(orc)
    ref = pool.decode(w.q, w.table, w.lens, w.scale)
    got = _run(torch, qkv, w, pool)
    r = compare_attention(got, ref)
    assert r["ok"], r
    gotb = _run(torch, qkv, w, pool, out_dtype=torch.bfloat16)
    rb = compare_attention(gotb, ref, bf16=True)
    assert rb["ok"], rb


def test_decode_mixed_batch_subset(env, orc):
    """32 sequences, lengths uniform in [4096, 65536] (the serving mix); the
    oracle checks a subset of 6 sequences against the full GPU batch."""
    torch, qkv = env
    from quantized_paged_kv_append_gb300 import synth
    lens = synth.seq_lengths(0, 32, 4096, 65536)
    w = Workload("int8", lens, 2, 16, 256, seed=0, spare=0)
    pool = w.oracle_pool(orc)
    got = _run(torch, qkv, w, pool)
    pick = np.array([0, 5, 11, 17, 26, 31])
    ref = pool.decode(w.q[pick], w.table[pick], w.lens[pick], w.scale)
    r = compare_attention(got[pick], ref)
    assert r["ok"], r


@pytest.mark.parametrize("B,lo,hi", [(200, 1, 700), (1024, 0, 40)])
def test_decode_many_sequences(env, orc, B, lo, hi):
    """More (sequence, head group) segments than CTAs: the merge records are
    kept per CTA instead of per segment. B = 1024 is the largest batch a call
    takes; empty sequences are mixed in when lo = 0."""
    torch, qkv = env
    rng = np.random.default_rng(B)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    w = Workload("int8", lens, 2, 16, 256, seed=8, spare=0)
    pool = w.oracle_pool(orc)
    got = _run(torch, qkv, w, pool)
    pick = np.unique(np.concatenate([np.arange(0, B, max(1, B // 24)), [B - 1], np.argmax(lens)[None]]))
    ref = pool.decode(w.q[pick], w.table[pick], w.lens[pick], w.scale)
    r = compare_attention(got[pick], ref)
    assert r["ok"], r
    assert np.all(got[lens == 0] == 0)


def test_decode_empty_and_single_token(env, orc):
    torch, qkv = env
    w = Workload("int8", [0, 1, 17, 0], 2, 16, 256, seed=4)
    pool = w.oracle_pool(orc)
    got = _run(torch, qkv, w, pool)
    ref = pool.decode(w.q, w.table, w.lens, w.scale)
    assert np.all(got[0] == 0) and np.all(got[3] == 0)
    r = compare_attention(got, ref)
    assert r["ok"], r


def test_decode_page_table_permutation_bitwise(env, orc):
    """Moving the same pages to other physical slots changes nothing: the
    output is bit-identical."""
    torch, qkv = env
    w = Workload("k8v4", [900, 333], 2, 16, 256, seed=8, spare=10)
    pool = w.oracle_pool(orc)
    a = _run(torch, qkv, w, pool)
    # relocate every page of the pool by a seeded permutation
    from quantized_paged_kv_append_gb300 import synth
    perm = synth.permutation(99, w.num_pages)
    planes2 = []
    for pl in pool.planes():
        rows = pl.reshape(w.num_pages, -1)
        moved = np.empty_like(rows)
        moved[perm] = rows
        planes2.append(moved.reshape(-1))
    table2 = np.where(w.table >= 0, perm[np.maximum(w.table, 0)], -1).astype(np.int32)

    class P2:
        def planes(self):
            return planes2
    b = _run(torch, qkv, w, P2(), table=table2)
    assert np.array_equal(a, b)


def test_decode_deterministic_and_workspace_reuse(env, orc):
    """Repeated calls with one workspace give identical bits (the counters are
    returned to zero by each call)."""
    torch, qkv = env
    w = Workload("int8", [5000, 20000, 70], 2, 16, 256, seed=9)
    pool = w.oracle_pool(orc)
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    ws = qkv.decode_workspace(cache, w.B, w.hq, w.max_len())
    outs = _run(torch, qkv, w, pool, workspace=ws, repeat=3)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    ref = pool.decode(w.q, w.table, w.lens, w.scale)
    assert compare_attention(outs[0], ref)["ok"]


def test_decode_bad_page_entry_flags_without_fault(env, orc):
    torch, qkv = env
    w = Workload("int8", [64], 2, 16, 256, seed=10)
    pool = w.oracle_pool(orc)
    bad = w.table.copy()
    bad[0, 2] = 10 ** 6
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    qkv.decode(cache, bf16_dev(w.q, torch), to_dev(bad, torch), to_dev(w.lens, torch), 64, scale=w.scale)
    torch.cuda.synchronize()
    assert qkv.device_error() & 1


@pytest.mark.parametrize("fmt,d,hkv,hq,lens", [
    ("int8", 256, 2, 16, [1, 37, 300, 16, 1000]), ("k8v4", 256, 2, 16, [1, 37, 300, 16, 1000]),
    ("iso3", 128, 4, 16, [1, 37, 300, 16, 1000]), ("iso4", 128, 4, 16, [1, 37, 300, 16, 1000]),
    ("int8", 256, 2, 32, [1, 37, 300, 16, 1000]), ("iso4", 256, 2, 4, [1, 37, 300, 16, 1000]),
    ("int8", 256, 2, 16, [131072]),   # the benchmark step: quantize-on-write + decode at 128K
    ("q4", 256, 2, 16, [1, 37, 300, 16, 1000]), ("k8vbf16", 256, 2, 16, [1, 37, 300, 16, 1000]),
    ("kbf16v8", 256, 2, 16, [1, 37, 300, 16, 1000]), ("kbf16v8", 128, 4, 16, [1, 37, 300, 16, 1000]),
])
def test_decode_fused_quantize_on_write(env, orc, fmt, d, hkv, hq, lens):
    """kv_decode_attn with k_new/v_new: the newest token (position L - 1) is
    quantized inside the decode launch. The pool bytes must equal the oracle's
    append of all tokens, and the output the oracle's decode over them."""
    torch, qkv = env
    w = Workload(fmt, lens, hkv, hq, d, seed=31)
    full = w.oracle_pool(orc)
    ref = full.decode(w.q, w.table, w.lens, w.scale)
    # the pool before the step: every token except each sequence's last one
    last = np.cumsum(w.lens) - 1
    keep = np.ones(w.seq_id.size, bool)
    keep[last] = False
    pre = orc.Pool(w.fmt, w.num_pages, w.hkv, w.d, quat=w.quat)
    pre.append(w.k[keep], w.v[keep], w.seq_id[keep], w.pos[keep], w.table)
    cache = gpu_cache(qkv, w, torch, planes=pre.planes())
    out = qkv.decode(cache, bf16_dev(w.q, torch), to_dev(w.table, torch), to_dev(w.lens, torch), w.max_len(),
                     scale=w.scale, out_dtype=torch.float32, k_new=bf16_dev(w.k[last], torch),
                     v_new=bf16_dev(w.v[last], torch))
    torch.cuda.synchronize()
    assert qkv.device_error() == 0
    for got, want, nm in zip([p.cpu().numpy() for p in cache.planes()], full.planes(), ["kc", "ks", "vc", "vs"]):
        assert np.array_equal(got, want), nm
    r = compare_attention(out.cpu().numpy(), ref)
    assert r["ok"], r


def test_decode_seq_lens_changed_in_stream(env, orc):
    """The kernel works out its share of the units from seq_lens before its dependency wait
    and keeps it only if a read after the wait finds seq_lens unchanged. Here a kernel
    earlier in the same stream rewrites seq_lens before every decode call (and one call
    follows another decode directly): each call must attend exactly its own lengths."""
    torch, qkv = env
    full = [900, 37, 2100, 16]
    w = Workload("int8", full, 2, 16, 256, seed=23)
    pool = w.oracle_pool(orc)
    cache = gpu_cache(qkv, w, torch, planes=pool.planes())
    t = to_dev(w.table, torch)
    q = bf16_dev(w.q, torch)
    steps = [np.array(full, np.int32) - d for d in (0, 5, 15, 9)]
    sl = to_dev(steps[0], torch)
    outs = []
    for i, lens in enumerate(steps):
        if i % 2 == 1:
            # a device-side rewrite of seq_lens in the same stream just before the call
            sl.copy_(torch.from_numpy(lens).cuda(non_blocking=False))
        else:
            sl.sub_(torch.from_numpy(steps[i - 1] - lens if i else np.zeros_like(lens)).cuda())
        outs.append(qkv.decode(cache, q, t, sl, max(full), scale=w.scale, out_dtype=torch.float32))
        outs.append(qkv.decode(cache, q, t, sl, max(full), scale=w.scale, out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert qkv.device_error() == 0
    for i, lens in enumerate(steps):
        ref = pool.decode(w.q, w.table, lens, w.scale)
        for o in outs[2 * i:2 * i + 2]:
            r = compare_attention(o.cpu().numpy(), ref)
            assert r["ok"], (i, r)
