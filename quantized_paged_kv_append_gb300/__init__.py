"""GB300-native quantized paged KV cache.

The path: quantize-on-write append (`append`), paged split-K decode attention
with on-the-fly dequantization (`decode`), and extend attention over a packed
prefix plus bf16 new tokens. All compute runs in libqkv.so (hand-written CUDA
for sm_103a behind the C ABI of include/qkv.h); this module only hands torch
tensors and streams to it.
"""

from __future__ import annotations

import ctypes as C
import math

from . import _lib
from ._lib import (FORMATS, QKV_INT8, QKV_K8V4, QKV_ISO3, QKV_ISO4, QKV_Q4, QKV_K8_VBF16, QKV_KBF16_V8,  # noqa: F401
                   QkvError)

__all__ = ["PagedKVCache", "append", "decode", "decode_workspace", "extend", "extend_workspace", "row_bytes", "iso_levels",
           "device_error"]


def _torch():
    import torch
    return torch


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else C.c_void_p(0)


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def row_bytes(fmt: int, store: int, head_dim: int):
    cb, sb = C.c_int(), C.c_int()
    _lib.check(_lib.lib().qkv_row_bytes(fmt, store, head_dim, C.byref(cb), C.byref(sb)), "qkv_row_bytes")
    return cb.value, sb.value


def iso_levels(bits: int):
    import numpy as np
    out = np.zeros(16, np.float32)
    n = _lib.lib().qkv_iso_levels(bits, out.ctypes.data_as(C.c_void_p))
    if n < 0:
        raise QkvError(n, "qkv_iso_levels")
    return out[:n].copy()


def device_error(clear: bool = True) -> int:
    rc = _lib.lib().qkv_device_error(int(clear))
    if rc < 0:
        raise QkvError(rc, "qkv_device_error")
    return rc


class PagedKVCache:
    """A paged pool: four caller-owned uint8 planes on the GPU,
    [num_pages, num_kv_heads, 16, row bytes] each."""

    def __init__(self, fmt, num_pages, num_kv_heads, head_dim, device="cuda", quat=None, planes=None):
        torch = _torch()
        self.fmt = FORMATS[fmt] if isinstance(fmt, str) else int(fmt)
        self.num_pages, self.num_kv_heads, self.head_dim, self.page_size = num_pages, num_kv_heads, head_dim, 16
        self.quat = [1.0, 0.0, 0.0, 0.0] if quat is None else [float(x) for x in quat]
        kcb, ksb = row_bytes(self.fmt, 0, head_dim)
        vcb, vsb = row_bytes(self.fmt, 1, head_dim)
        rows = num_pages * num_kv_heads * 16
        if planes is None:
            planes = [torch.zeros(rows * n, dtype=torch.uint8, device=device) for n in (kcb, ksb, vcb, vsb)]
        self.k_codes, self.k_scales, self.v_codes, self.v_scales = planes
        d = self._desc = _lib.CacheDesc()
        d.format, d.num_pages, d.page_size = self.fmt, num_pages, 16
        d.num_kv_heads, d.head_dim = num_kv_heads, head_dim
        d.k_codes, d.k_scales = self.k_codes.data_ptr(), self.k_scales.data_ptr()
        d.v_codes, d.v_scales = self.v_codes.data_ptr(), self.v_scales.data_ptr()
        for i in range(4):
            d.quat[i] = self.quat[i]

    @property
    def desc(self):
        return self._desc

    def planes(self):
        return self.k_codes, self.k_scales, self.v_codes, self.v_scales


def append(cache: PagedKVCache, k, v, seq_id, pos, page_table, stream=None):
    """Quantize-on-write: k, v bf16 [n, Hkv, D]; seq_id, pos int32 [n];
    page_table int32 [B, max_pages]."""
    n = int(seq_id.numel())
    rc = _lib.lib().iso_kv_append(C.byref(cache.desc), _ptr(k), _ptr(v), n, _ptr(seq_id), _ptr(pos),
                                  _ptr(page_table), int(page_table.shape[0]), int(page_table.shape[1]),
                                  _stream(stream))
    _lib.check(rc, "iso_kv_append")


def decode_workspace(cache: PagedKVCache, batch: int, num_q_heads: int, max_seq_len: int, device="cuda"):
    """Workspace for `decode`: partial results and merge records (no initialization needed)."""
    torch = _torch()
    n = _lib.lib().kv_decode_workspace_size(C.byref(cache.desc), batch, num_q_heads, max_seq_len)
    if n == 0 and batch > 0:
        raise QkvError(-1, "kv_decode_workspace_size")
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def decode(cache: PagedKVCache, q, page_table, seq_lens, max_seq_len: int, scale=None, out=None,
           out_dtype=None, workspace=None, stream=None, k_new=None, v_new=None):
    """Decode attention: q bf16 [B, Hq, D] -> out [B, Hq, D] (bf16 or fp32).

    With k_new / v_new (bf16 [B, Hkv, D]) the step's own token is quantized and
    written at position seq_lens[b] - 1 inside the same kernel launch
    (quantize-on-write) before it is attended."""
    torch = _torch()
    B, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype or torch.bfloat16, device=q.device)
    odt = _lib.QKV_OUT_F32 if out.dtype == torch.float32 else _lib.QKV_OUT_BF16
    if workspace is None:
        workspace = decode_workspace(cache, B, Hq, max_seq_len, device=q.device)
    rc = _lib.lib().kv_decode_attn(C.byref(cache.desc), _ptr(q), _ptr(k_new), _ptr(v_new), B, Hq, _ptr(page_table),
                                   int(page_table.shape[1]),
                                   _ptr(seq_lens), int(max_seq_len), float(scale), _ptr(out), odt, _ptr(workspace),
                                   workspace.numel(), _stream(stream))
    _lib.check(rc, "kv_decode_attn")
    return out


def extend_workspace(cache: PagedKVCache, batch: int, max_q_len: int, max_pages_per_seq: int, device="cuda"):
    """Scratch for extend (the dequantized prefix and chunk); no initialization needed."""
    torch = _torch()
    n = _lib.lib().kv_extend_workspace_size(C.byref(cache.desc), batch, max_q_len, max_pages_per_seq)
    if n == 0:
        raise QkvError(-1, "kv_extend_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def extend(cache: PagedKVCache, q, k_new, v_new, cu_seqlens, prefix_lens, page_table, max_q_len: int, scale=None,
           causal=True, out=None, out_dtype=None, stream=None, workspace=None):
    """Extend attention: q bf16 [total, Hq, D], k_new / v_new bf16 [total, Hkv, D]
    (rows of sequence b are cu_seqlens[b]..cu_seqlens[b+1]) over the packed
    prefix [0, prefix_lens[b]) plus the new tokens. Returns out [total, Hq, D]."""
    torch = _torch()
    total, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((total, Hq, D), dtype=out_dtype or torch.bfloat16, device=q.device)
    odt = _lib.QKV_OUT_F32 if out.dtype == torch.float32 else _lib.QKV_OUT_BF16
    B, maxp = int(prefix_lens.numel()), int(page_table.shape[1])
    if workspace is None and B > 0 and max_q_len > 0:
        workspace = extend_workspace(cache, B, int(max_q_len), maxp, device=q.device)
    ws_ptr, ws_bytes = (_ptr(workspace), workspace.numel() * workspace.element_size()) if workspace is not None else (None, 0)
    rc = _lib.lib().kv_extend_attn(C.byref(cache.desc), _ptr(q), _ptr(k_new), _ptr(v_new), Hq, _ptr(cu_seqlens),
                                   _ptr(prefix_lens), B, int(max_q_len), _ptr(page_table), maxp, float(scale),
                                   int(bool(causal)), _ptr(out), odt, ws_ptr, ws_bytes, _stream(stream))
    _lib.check(rc, "kv_extend_attn")
    return out


def gather_dequant(cache: PagedKVCache, page_row, length: int, stream=None):
    """The dequantized K and V of one sequence (fp32 [length, Hkv, D] each, in
    the original domain), read through its page-table row (int32 device)."""
    torch = _torch()
    dev = page_row.device
    k = torch.empty((length, cache.desc.num_kv_heads, cache.desc.head_dim), dtype=torch.float32, device=dev)
    v = torch.empty_like(k)
    rc = _lib.lib().kv_gather_dequant(C.byref(cache.desc), _ptr(page_row), int(length), _ptr(k), _ptr(v),
                                      _stream(stream))
    _lib.check(rc, "kv_gather_dequant")
    return k, v


def verify_workspace(cache: PagedKVCache, num_q_heads: int, total_q: int, max_pages_per_seq: int, device="cuda"):
    """Scratch for verify (expanded page-table rows, per-query lengths, decode partials)."""
    torch = _torch()
    n = _lib.lib().kv_verify_workspace_size(C.byref(cache.desc), num_q_heads, total_q, max_pages_per_seq)
    if n == 0:
        raise QkvError(-1, "kv_verify_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def verify(cache: PagedKVCache, q, cu_seqlens, seq_lens, page_table, max_seq_len: int, scale=None, out=None,
           out_dtype=None, workspace=None, stream=None):
    """Verify window: q bf16 [total_q, Hq, D]; rows cu_seqlens[b]..cu_seqlens[b+1] are the
    last W_b positions of sequence b (query j attends [0, seq_lens[b] - W_b + j + 1)).
    Returns out [total_q, Hq, D]."""
    torch = _torch()
    total, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((total, Hq, D), dtype=out_dtype or torch.bfloat16, device=q.device)
    odt = _lib.QKV_OUT_F32 if out.dtype == torch.float32 else _lib.QKV_OUT_BF16
    B, maxp = int(seq_lens.numel()), int(page_table.shape[1])
    if workspace is None and total > 0 and B > 0:
        workspace = verify_workspace(cache, Hq, total, maxp, device=q.device)
    ws_ptr, ws_bytes = (_ptr(workspace), workspace.numel() * workspace.element_size()) if workspace is not None else (None, 0)
    rc = _lib.lib().kv_verify_attn(C.byref(cache.desc), _ptr(q), B, Hq, _ptr(cu_seqlens), _ptr(seq_lens), int(total),
                                   _ptr(page_table), maxp, int(max_seq_len), float(scale), _ptr(out), odt, ws_ptr,
                                   ws_bytes, _stream(stream))
    _lib.check(rc, "kv_verify_attn")
    return out


def verify_fixed_workspace(cache: PagedKVCache, batch: int, window: int, num_q_heads: int, max_pages_per_seq: int,
                           device="cuda"):
    """Scratch for the fixed-window verify (partial results of the split tiles; for the
    formats other than int8 also the expanded page-table rows)."""
    torch = _torch()
    n = _lib.lib().kv_verify_fixed_workspace_size(C.byref(cache.desc), int(batch), int(window), int(num_q_heads),
                                                  int(max_pages_per_seq))
    if n == 0:
        raise QkvError(-1, "kv_verify_fixed_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def verify_fixed(cache: PagedKVCache, q, seq_lens, page_table, max_seq_len: int, window: int, scale=None, out=None,
                 out_dtype=None, workspace=None, stream=None):
    """Verify window of the same length in every sequence, in one pass: q bf16
    [batch * window, Hq, D]; row b * window + w sits at position seq_lens[b] - window + w
    and attends [0, seq_lens[b] - window + w + 1). Returns out [batch * window, Hq, D]."""
    torch = _torch()
    total, Hq, D = q.shape
    B, maxp = int(seq_lens.numel()), int(page_table.shape[1])
    if total != B * int(window):
        raise QkvError(-1, "verify_fixed: q rows must be batch * window")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((total, Hq, D), dtype=out_dtype or torch.bfloat16, device=q.device)
    odt = _lib.QKV_OUT_F32 if out.dtype == torch.float32 else _lib.QKV_OUT_BF16
    if workspace is None and B > 0:
        workspace = verify_fixed_workspace(cache, B, int(window), Hq, maxp, device=q.device)
    ws_ptr, ws_bytes = (_ptr(workspace), workspace.numel() * workspace.element_size()) if workspace is not None else (None, 0)
    rc = _lib.lib().kv_verify_attn_fixed(C.byref(cache.desc), _ptr(q), B, int(window), Hq, _ptr(seq_lens),
                                         _ptr(page_table), maxp, int(max_seq_len), float(scale), _ptr(out), odt,
                                         ws_ptr, ws_bytes, _stream(stream))
    _lib.check(rc, "kv_verify_attn_fixed")
    return out

