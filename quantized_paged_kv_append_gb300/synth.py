"""Seeded synthetic inputs for the quantized paged KV-cache path.

This module is the one piece shared by the CPU oracle's tests and the CUDA
path's tests and benchmark: it only draws numbers. It holds none of the
method's arithmetic (no quantization, rotation or attention).

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) over a counter, 53-bit uniforms, Box-Muller
normals; bf16 values are the round-to-nearest-even narrowing of the fp32
normals. Each named stream gets its own seed derived from (seed, stream id).
"""

from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

_STREAMS = {"q": 1, "k": 2, "v": 3, "outlier": 4, "perm": 5, "quat": 6, "lens": 7,
            "k_new": 8, "v_new": 9, "misc": 10, "q_ext": 11, "k_ext": 12, "v_ext": 13, "q_verify": 14, "q_verify_fixed": 15}


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _stream_seed(seed: int, stream: str) -> np.uint64:
    base = np.array([(seed * 1000003 + _STREAMS[stream]) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix(base * _GOLDEN + _GOLDEN)[0]


def uint64s(seed: int, stream: str, n: int, offset: int = 0) -> np.ndarray:
    s = _stream_seed(seed, stream)
    idx = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(s + idx * _GOLDEN)


def uniforms(seed: int, stream: str, n: int, offset: int = 0) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    return (uint64s(seed, stream, n, offset) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normals_f32(seed: int, stream: str, n: int, chunk: int = 1 << 22) -> np.ndarray:
    """n standard normals (fp32) by Box-Muller on consecutive uniform pairs."""
    out = np.empty(n, dtype=np.float32)
    done = 0
    while done < n:
        m = min(chunk, n - done)
        pairs = (m + 1) // 2
        u = uniforms(seed, stream, 2 * pairs, offset=done + (done & 1))
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))
        z = np.empty(2 * pairs, dtype=np.float64)
        z[0::2] = r * np.cos(2.0 * np.pi * u2)
        z[1::2] = r * np.sin(2.0 * np.pi * u2)
        out[done:done + m] = z[:m].astype(np.float32)
        done += m
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def outlier_channels(seed: int, head_dim: int, count: int = 4) -> np.ndarray:
    """`count` distinct channel indices, the same for every head and token."""
    keys = uint64s(seed, "outlier", head_dim)
    return np.sort(np.argsort(keys, kind="stable")[:count]).astype(np.int64)


def tensor_bf16(seed: int, stream: str, shape, outlier_scale: float = 0.0, n_outliers: int = 4) -> np.ndarray:
    """bf16 bits of N(0,1) draws of `shape`; if outlier_scale > 0, the last-axis
    channels chosen by `outlier_channels` are multiplied by it before rounding."""
    n = int(np.prod(shape))
    x = normals_f32(seed, stream, n).reshape(shape)
    if outlier_scale:
        ch = outlier_channels(seed, shape[-1], n_outliers)
        x[..., ch] *= np.float32(outlier_scale)
    return bf16_bits(x)


def permutation(seed: int, n: int, stream: str = "perm") -> np.ndarray:
    """Fisher-Yates shuffle of range(n) driven by the seeded stream."""
    p = np.arange(n, dtype=np.int64)
    r = uint64s(seed, stream, max(n - 1, 0))
    for i in range(n - 1, 0, -1):
        j = int(r[n - 1 - i] % np.uint64(i + 1))
        p[i], p[j] = p[j], p[i]
    return p


def permutation_fast(seed: int, n: int, stream: str = "perm") -> np.ndarray:
    """A seeded random permutation for large n (argsort of random keys)."""
    return np.argsort(uint64s(seed, stream, n), kind="stable").astype(np.int64)


def page_table(seed: int, pages_per_seq, page_size: int = 16, max_pages: int | None = None,
               num_pages: int | None = None, shuffle: bool = True):
    """Assign each sequence its pages out of one shuffled pool.

    Returns (table int32 [B, max_pages], num_pages). Unused entries are -1.
    """
    pages_per_seq = [int(p) for p in pages_per_seq]
    total = sum(pages_per_seq)
    if num_pages is None:
        num_pages = total
    if max_pages is None:
        max_pages = max(pages_per_seq) if pages_per_seq else 0
    if shuffle:
        perm = permutation(seed, num_pages) if num_pages <= 4096 else permutation_fast(seed, num_pages)
    else:
        perm = np.arange(num_pages, dtype=np.int64)
    table = np.full((len(pages_per_seq), max(max_pages, 1)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(pages_per_seq):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, num_pages


def unit_quaternion(seed: int) -> np.ndarray:
    """One unit quaternion (w, x, y, z) in fp32: four N(0,1) draws normalised
    in double, then rounded to fp32."""
    z = normals_f32(seed, "quat", 4).astype(np.float64)
    return (z / np.sqrt(np.sum(z * z))).astype(np.float32)


def seq_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """Integer lengths uniform on [lo, hi]."""
    u = uniforms(seed, "lens", batch)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int32)
