"""Seeded workloads shared by the parity tests: inputs come from the synth
module; expected values come from the CPU oracle only."""

from __future__ import annotations

import math

import numpy as np

from quantized_paged_kv_append_gb300 import synth

FMT = {"int8": 0, "k8v4": 1, "iso3": 2, "iso4": 3, "q4": 4, "k8vbf16": 5, "kbf16v8": 6}


class Workload:
    """Decode workload: pool contents for B sequences of lengths `lens`, one
    query per sequence, a shuffled page table with `spare` unused pages."""

    def __init__(self, fmt, lens, hkv, hq, d, seed=0, outliers=True, spare=3, max_pages=None):
        self.fmt = FMT[fmt] if isinstance(fmt, str) else fmt
        self.lens = np.asarray(lens, np.int32)
        self.B, self.hkv, self.hq, self.d, self.seed = len(lens), hkv, hq, d, seed
        pages = [max(1, (int(L) + 15) // 16) for L in lens]
        self.table, self.num_pages = synth.page_table(seed, pages, num_pages=sum(pages) + spare,
                                                      max_pages=max_pages or max(pages))
        iso = self.fmt in (2, 3)
        self.quat = synth.unit_quaternion(seed) if iso else np.array([1, 0, 0, 0], np.float32)
        n = int(self.lens.sum())
        self.k = synth.tensor_bf16(seed, "k", (n, hkv, d), outlier_scale=20.0 if outliers else 0.0)
        self.v = synth.tensor_bf16(seed, "v", (n, hkv, d))
        self.seq_id = np.repeat(np.arange(self.B), self.lens).astype(np.int32)
        self.pos = np.concatenate([np.arange(L) for L in self.lens]).astype(np.int32) if n else np.zeros(0, np.int32)
        self.q = synth.tensor_bf16(seed, "q", (self.B, hq, d))
        self.scale = float(np.float32(1.0 / math.sqrt(d)))

    def oracle_pool(self, orc):
        pool = orc.Pool(self.fmt, self.num_pages, self.hkv, self.d, quat=self.quat)
        if self.seq_id.size:
            assert pool.append(self.k, self.v, self.seq_id, self.pos, self.table) == 0
        return pool

    def max_len(self):
        return int(self.lens.max()) if self.B else 0


def to_dev(a, torch, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_dev(bits, torch):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def gpu_cache(qkv, w, torch, planes=None):
    """A PagedKVCache on the GPU; planes (numpy) are uploaded if given."""
    dev = None
    if planes is not None:
        dev = [torch.from_numpy(np.ascontiguousarray(p)).cuda() for p in planes]
    return qkv.PagedKVCache(w.fmt, w.num_pages, w.hkv, w.d, quat=w.quat.tolist(), planes=dev)


def _log_metrics(res):
    import json
    import os
    path = os.environ.get("QKV_PARITY_LOG")
    if path:
        test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
        with open(path, "a") as f:
            f.write(json.dumps(dict(res, test=test, ok=bool(res["ok"]))) + "\n")


def compare_attention(gpu, ref, atol=2e-3, cos_min=0.9999, bf16=False):
    """max-abs and cosine against the double-precision oracle. fp32 output is
    held to |err| <= atol; bf16 output to atol + 2^-8 |ref| (half a bf16 ulp
    of the output plus the kernel tolerance)."""
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    err = np.abs(g - r)
    bound = atol + (2.0 ** -8) * np.abs(r) if bf16 else atol
    worst = float(np.max(err - bound)) if err.size else 0.0
    rows_g = g.reshape(-1, g.shape[-1])
    rows_r = r.reshape(-1, r.shape[-1])
    num = np.sum(rows_g * rows_r, axis=1)
    den = np.linalg.norm(rows_g, axis=1) * np.linalg.norm(rows_r, axis=1)
    nz = den > 0
    cos = num[nz] / den[nz]
    res = {"max_abs": float(err.max()) if err.size else 0.0, "excess": worst,
           "min_cos": float(cos.min()) if cos.size else 1.0, "ok": worst <= 0 and (cos.size == 0 or cos.min() > cos_min)}
    _log_metrics(res)
    return res
