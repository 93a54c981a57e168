"""GPU parity of quantize-on-write append: the packed code and scale planes
written by the CUDA path must equal the oracle's byte for byte."""

import numpy as np
import pytest

from _workload import Workload, bf16_dev, gpu_cache, to_dev

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


def _append_gpu(torch, qkv, w, chunks=1):
    cache = gpu_cache(qkv, w, torch)
    table = to_dev(w.table, torch)
    n = w.seq_id.size
    bounds = np.linspace(0, n, chunks + 1).astype(int)
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b > a:
            qkv.append(cache, bf16_dev(w.k[a:b], torch), bf16_dev(w.v[a:b], torch),
                       to_dev(w.seq_id[a:b], torch), to_dev(w.pos[a:b], torch), table)
    torch.cuda.synchronize()
    assert qkv.device_error() == 0
    return [p.cpu().numpy() for p in cache.planes()]


def _assert_planes_equal(got, ref, label):
    names = ["k_codes", "k_scales", "v_codes", "v_scales"]
    for g, r, nm in zip(got, ref, names):
        if not np.array_equal(g, r):
            diff = np.flatnonzero(g != r)
            raise AssertionError(f"{label} {nm}: {diff.size} bytes differ, first at {diff[:8]}")


CASES = [
    ("int8", 256, 2), ("int8", 128, 4), ("k8v4", 256, 2),
    ("iso3", 128, 4), ("iso4", 128, 4), ("iso3", 256, 2), ("iso4", 256, 2),
    ("q4", 256, 2), ("k8vbf16", 256, 2), ("k8vbf16", 128, 4), ("kbf16v8", 256, 2), ("kbf16v8", 128, 4),
]


@pytest.mark.parametrize("fmt,d,hkv", CASES)
def test_append_bytes_small_ragged(env, orc, fmt, d, hkv):
    torch, qkv = env
    w = Workload(fmt, [1, 37, 300, 16], hkv, hkv, d, seed=11)
    ref = w.oracle_pool(orc).planes()
    got = _append_gpu(torch, qkv, w, chunks=3)
    _assert_planes_equal(got, ref, f"{fmt} D={d}")


@pytest.mark.parametrize("fmt,d,hkv,L", [("int8", 256, 2, 2048), ("int8", 256, 2, 131072),
                                         ("k8v4", 256, 2, 118750), ("iso3", 128, 4, 81920),
                                         ("iso4", 128, 4, 81920), ("q4", 256, 2, 131072),
                                         ("k8vbf16", 256, 2, 65536), ("kbf16v8", 256, 2, 65536)])
def test_append_bytes_full_size(env, orc, fmt, d, hkv, L):
    """The configurations the benchmark runs: every token of the pool."""
    torch, qkv = env
    w = Workload(fmt, [L], hkv, 16, d, seed=0)
    ref = w.oracle_pool(orc).planes()
    got = _append_gpu(torch, qkv, w)
    _assert_planes_equal(got, ref, f"{fmt} L={L}")


def test_append_edge_values(env, orc):
    """Zero vectors, huge/tiny magnitudes, exact ties and sign patterns."""
    torch, qkv = env
    from quantized_paged_kv_append_gb300 import synth
    for fmt, d in (("int8", 256), ("k8v4", 256), ("iso3", 128), ("iso4", 128)):
        w = Workload(fmt, [64], 2, 2, d, seed=5)
        x = synth.bf16_to_f32(w.k).copy()
        x[0] = 0.0                                   # all-zero vectors
        x[1, 0, 5] = np.float32(3e4)                 # one huge value in a group
        x[2] *= np.float32(1e-6)                     # tiny (fp16 subnormal scales)
        x[3, :, ::2] = np.float32(0.5) * np.arange(d // 2)[None]   # exact multiples -> ties
        x[4] = -np.abs(x[4])
        x[5, :, :] = np.float32(1.0)                 # constant vector (q4 first-index tie)
        w.k = synth.bf16_bits(x)
        w.v = synth.bf16_bits(x[::-1].copy())
        ref = w.oracle_pool(orc).planes()
        got = _append_gpu(torch, qkv, w)
        _assert_planes_equal(got, ref, f"{fmt} edge")


def test_append_bad_entries_flag_and_skip(env, orc):
    torch, qkv = env
    w = Workload("int8", [40], 2, 2, 256, seed=3)
    bad = w.table.copy()
    bad[0, 1] = w.num_pages + 7          # tokens 16..31 land on an out-of-range page
    cache = gpu_cache(qkv, w, torch)
    pos = w.pos.copy()
    pos[39] = 10 ** 6                    # position past the table
    qkv.append(cache, bf16_dev(w.k, torch), bf16_dev(w.v, torch), to_dev(w.seq_id, torch), to_dev(pos, torch),
               to_dev(bad, torch))
    torch.cuda.synchronize()
    err = qkv.device_error()
    assert err & 1 and err & 2
    assert qkv.device_error() == 0       # cleared
    # the oracle with the same bad table skips the same tokens (pos 39 is dropped by hand)
    pool = orc.Pool(w.fmt, w.num_pages, w.hkv, w.d)
    keep = np.arange(40) != 39
    skipped = pool.append(w.k[keep], w.v[keep], w.seq_id[keep], w.pos[keep], bad)
    assert skipped == 16
    _assert_planes_equal([p.cpu().numpy() for p in cache.planes()], pool.planes(), "bad entries")
