"""Benchmark: decode attention over an int8 paged KV cache at 128K context on
one GB300 (batch 1, 16 query heads / 2 KV heads, head_dim 256, page 16,
shuffled page table, bf16 N(0,1) inputs with four x20 K outlier channels).

One step = quantize-on-write of the step's new token (K and V, position
131071) into the cache + split-K decode attention over all 131072 cached
tokens, both inside one kv_decode_attn launch. Eight
independent layer caches (1.1 GB, well above the 129 MB L2) are cycled so no
step reads another's data from L2.

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle on the
same workload instead (the reference arm).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn packed-KV HBM GB/s (% of peak) and steps/s at 128K ctx, 1 GB300"
B, HQ, HKV, D, L = 1, 16, 2, 256, 131072
LAYERS = 8   # default; --layers overrides
LAUNCHES_PER_STEP = 2   # int8 decode: the tensor-core kernel and the split-merge (combine) kernel
KV_BYTES_PER_TOKEN = 2 * HKV * (D + 2 * D // 64)        # int8 codes + fp16 scales, K and V: 1056
# dram__bytes_read.sum + dram__bytes_write.sum of one decode_tc_kernel<256,8,0,false> launch at this
# workload, from an ncu capture of the current kernel build (138.59 MB read + 2.97 MB written)
NCU_TRAFFIC_BYTES = 141_555_456
# the same counters for the other decode workloads where a capture of the current kernel exists
WORKLOAD_NCU_TRAFFIC = {}
DECODE_BYTES = L * KV_BYTES_PER_TOKEN                     # 138,412,032 packed bytes read per step
WORKLOAD = ("int8 KV decode at 128K context: batch 1, 16 q heads / 2 KV heads, head_dim 256, "
            "131072 cached tokens, page 16, shuffled page table; step = quantize-on-write of 1 token + decode")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _clock_sampler():
    f = tempfile.NamedTemporaryFile(prefix="qkv_clk", suffix=".csv", delete=False)
    q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    try:
        p = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "100"],
                             stdout=f, stderr=subprocess.DEVNULL)
    except OSError:
        return None, f.name
    return p, f.name


def _clock_summary(proc, path, gpu_index):
    if proc is None:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
    proc.terminate()
    try:
        proc.wait(timeout=5)
    except subprocess.TimeoutExpired:
        proc.kill()
    sm, smax, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in open(path):
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9 or not parts[0].isdigit() or int(parts[0]) != gpu_index:
            continue
        try:
            sm.append(float(parts[1]))
            smax = float(parts[2])
        except ValueError:
            continue
        for nm, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(nm)
    os.unlink(path)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
            "samples": len(sm)}


def rank_env():
    """(world, rank, local_rank) from the torchrun environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value, world, device="cpu"):
    """The largest `value` over all ranks (identity when alone)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step, steps_per_rank, world, elapsed_ms):
    """Whole-job GB/s: every rank's steps over the slowest rank's time."""
    return bytes_per_step * steps_per_rank * world / (elapsed_ms / 1e3) / 1e9


_INPUT_CACHE = {}


def _inputs(seed=0):
    if seed in _INPUT_CACHE:
        return _INPUT_CACHE[seed]
    from quantized_paged_kv_append_gb300 import synth
    pages = (L + 15) // 16
    k = synth.tensor_bf16(seed, "k", (L, HKV, D), outlier_scale=20.0)
    v = synth.tensor_bf16(seed, "v", (L, HKV, D))
    q = synth.tensor_bf16(seed, "q", (LAYERS, B, HQ, D))
    kn = synth.tensor_bf16(seed, "k_new", (LAYERS, 1, HKV, D), outlier_scale=20.0)
    vn = synth.tensor_bf16(seed, "v_new", (LAYERS, 1, HKV, D))
    tables = [synth.page_table(seed * 100 + layer, [pages])[0] for layer in range(LAYERS)]
    _INPUT_CACHE[seed] = (pages, k, v, q, kn, vn, tables)
    return _INPUT_CACHE[seed]


# ---------------------------------------------------------------------------
# CUDA arm
# ---------------------------------------------------------------------------
def run_gpu(args):
    import torch
    import torch.distributed as dist

    import quantized_paged_kv_append_gb300 as qkv
    from quantized_paged_kv_append_gb300 import build as qbuild

    world, rank, local = rank_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0:
        qbuild.build()
    if world > 1:
        dist.barrier()
    qbuild.build()  # no-op when up to date
    dev = torch.device("cuda", local)

    pages, k, v, q, kn, vn, tables = _inputs(args.seed)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    k_d, v_d = bf(k), bf(v)
    seq_all = i32(np.zeros(L, np.int32))
    pos_all = i32(np.arange(L, dtype=np.int32))
    caches, tabs = [], []
    for layer in range(LAYERS):
        c = qkv.PagedKVCache("int8", pages, HKV, D, device=dev)
        t = i32(tables[layer])
        qkv.append(c, k_d, v_d, seq_all, pos_all, t)   # fill the cache (quantize-on-write of all tokens)
        caches.append(c)
        tabs.append(t)
    del k_d, v_d
    q_d = bf(q)                       # [LAYERS, 1, HQ, D]
    kn_d, vn_d = bf(kn), bf(vn)       # [LAYERS, 1, HKV, D]
    seq1 = i32(np.zeros(1, np.int32))
    pos1 = i32(np.array([L - 1], np.int32))
    lens = i32(np.array([L], np.int32))
    out = torch.empty((B, HQ, D), dtype=torch.bfloat16, device=dev)
    ws = qkv.decode_workspace(caches[0], B, HQ, L, device=dev)
    scale = 1.0 / math.sqrt(D)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    assert qkv.device_error() == 0

    def step(i, ev=None):
        layer = i % LAYERS
        if ev is not None:
            ev[0].record(stream)
        qkv.decode(caches[layer], q_d[layer], tabs[layer], lens, L, scale=scale, out=out, workspace=ws, stream=stream,
                   k_new=kn_d[layer, 0], v_new=vn_d[layer, 0])
        if ev is not None:
            ev[1].record(stream)

    # warm-up (eager), then capture K steps into one graph with per-decode events
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()
    def timing_event():
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return torch.cuda.Event(enable_timing=True)

    # the timed graph: K steps back to back (nothing between the launches, so each
    # step's kernels may overlap the previous step's drain as the library allows)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(args.steps):
            step(i)
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    # a second graph of the same K steps, each bracketed by event-record nodes: the
    # duration of one launch of the decode path, for the roofline
    evs = [(timing_event(), timing_event()) for _ in range(args.steps)]
    per_launch = True
    try:
        egraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(egraph, stream=stream):
            for i in range(args.steps):
                step(i, evs[i])
        with torch.cuda.stream(stream):
            egraph.replay()
        torch.cuda.synchronize()
        _ = evs[0][0].elapsed_time(evs[0][1])
    except Exception:
        per_launch = False
        torch.cuda.synchronize()

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    proc, cpath = _clock_sampler()
    time.sleep(0.3)
    reps = max(1, args.reps)
    with torch.cuda.stream(stream):     # CUDAGraph.replay launches on the current stream
        t0.record(stream)
        for _ in range(reps):
            graph.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    if per_launch:
        with torch.cuda.stream(stream):
            egraph.replay()
        torch.cuda.synchronize()
        dec_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    else:
        dec_ms = None
    torch.cuda.synchronize()
    clocks = _clock_summary(proc, cpath, local)
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, device=dev)
    nsteps = args.steps * reps
    ms_per_step = total_ms / nsteps
    value = job_throughput(DECODE_BYTES, nsteps, world, total_ms)
    if dec_ms is None:
        dec_ms = ms_per_step

    e2e = None
    if not args.no_e2e:
        # end to end through the public API with host buffers (pinned), copies inside the timed region
        # the step's inputs (q, the new token's K and V, its sequence length) packed into one
        # pinned host buffer, so each step issues one host->device copy: q at byte 0, K at
        # nq, V at nq + nkv, the length at nq + 2 nkv (all 16-byte aligned)
        nq, nkv = B * HQ * D * 2, B * HKV * D * 2
        h_in = torch.empty(nq + 2 * nkv + 16, dtype=torch.uint8).pin_memory()
        h_in[:nq].copy_(torch.from_numpy(np.ascontiguousarray(q[0]).view(np.uint8).ravel()))
        h_in[nq:nq + nkv].copy_(torch.from_numpy(np.ascontiguousarray(kn[0]).view(np.uint8).ravel()))
        h_in[nq + nkv:nq + 2 * nkv].copy_(torch.from_numpy(np.ascontiguousarray(vn[0]).view(np.uint8).ravel()))
        h_in[nq + 2 * nkv:].copy_(torch.from_numpy(np.array([L, 0, 0, 0], np.int32).view(np.uint8)))
        h_out = torch.empty((B, HQ, D), dtype=torch.bfloat16).pin_memory()
        d_in = torch.empty_like(h_in, device=dev)
        d_q = d_in[:nq].view(torch.bfloat16).view(B, HQ, D)
        d_kn = d_in[nq:nq + nkv].view(torch.bfloat16).view(HKV, D)
        d_vn = d_in[nq + nkv:nq + 2 * nkv].view(torch.bfloat16).view(HKV, D)
        d_len = d_in[nq + 2 * nkv:nq + 2 * nkv + 4].view(torch.int32)
        h2d = h_in.numel()
        d2h = h_out.numel() * 2

        def e2e_step(i):
            layer = i % LAYERS
            d_in.copy_(h_in, non_blocking=True)
            qkv.decode(caches[layer], d_q, tabs[layer], d_len, L, scale=scale, out=out, workspace=ws,
                       stream=stream, k_new=d_kn, v_new=d_vn)
            h_out.copy_(out, non_blocking=True)

        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                e2e_step(i)
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            w0 = time.perf_counter()
            e0.record(stream)
            for i in range(args.steps):
                e2e_step(i)
            e1.record(stream)
            e1.synchronize()
            wall = time.perf_counter() - w0
        e2e_ms = max(e0.elapsed_time(e1), wall * 1e3) / args.steps
        assert qkv.device_error() == 0
        e2e = {"value": round(DECODE_BYTES / (e2e_ms / 1e3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = peaks()
    # roofline: the decode path's algorithmic bytes over the graph step time. One step is the
    # main kernel plus the merge kernel, overlapped by programmatic dependent launch, so the
    # step time is the duration of the decode path; an event pair around one call breaks that
    # overlap and reads longer than the step itself (reported below as decode_us_bracketed)
    dec_gbs = DECODE_BYTES / (ms_per_step / 1e3) / 1e9
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": nsteps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded splitmix64 + Box-Muller, bf16)",
        "config": {"workload": WORKLOAD, "batch": B, "q_heads": HQ, "kv_heads": HKV, "head_dim": D,
                   "context": L, "page_size": 16, "format": "int8", "layer_copies": LAYERS,
                   "l2": f"inputs larger than L2: {LAYERS} layer caches ({LAYERS * DECODE_BYTES / 1e9:.2f} GB) cycled",
                   "parallelism": f"replicas x{world}"},
        "steps_per_s": round(1e3 / ms_per_step, 1),
        "pct_of_peak": round(100.0 * value / peak, 2),
        "decode_us": round(ms_per_step * 1e3, 2),
        "decode_us_bracketed": round(dec_ms * 1e3, 2) if per_launch else None,
        "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(dec_gbs / peak, 4), "traffic": NCU_TRAFFIC_BYTES, "peak_kind": peak_kind,
                     "kernel": "decode_tc_kernel<256,8,0> + decode_tc_combine<256,8> (one decode call)",
                     "bytes_per_launch": DECODE_BYTES,
                     "timing": "graph step time: K decode calls back to back in a CUDA graph, CUDA events around "
                               "the replays, divided by K (main + merge launch per call, overlapped by "
                               "programmatic dependent launch)"},
        "e2e": e2e,
        "gpu_launches": nsteps * LAUNCHES_PER_STEP,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        res["cpu_baseline"] = cpu_baseline(args, quick=True)
    print(json.dumps(res))
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------
def _oracle_workload(seed):
    import oracle
    oracle.build()
    pages, k, v, q, kn, vn, tables = _inputs(seed)
    pool = oracle.Pool(0, pages, HKV, D)
    seq = np.zeros(L, np.int32)
    pos = np.arange(L, dtype=np.int32)
    pool.append(k, v, seq, pos, tables[0])
    return oracle, pool, q, kn, vn, tables


def _oracle_step(pool, q, kn, vn, table, layer):
    pool.append(kn[layer], vn[layer], np.zeros(1, np.int32), np.array([L - 1], np.int32), table)
    return pool.decode(q[layer], table, np.array([L], np.int32), float(np.float32(1 / math.sqrt(D))))


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(args, quick=False, steps=None, warmup=0):
    """The oracle as it stands on the host cores: first one thread, then one step per
    thread on every core at once (ctypes releases the GIL inside the oracle's C++, and
    each thread works on its own copy of the pool's planes, so the threads share
    nothing). The line's value is the all-core throughput."""
    import threading

    oracle, pool, q, kn, vn, tables = _oracle_workload(args.seed)
    for i in range(warmup):
        _oracle_step(pool, q, kn, vn, tables[0], i % LAYERS)
    n = steps if steps is not None else (2 if quick else 3)
    t0 = time.perf_counter()
    for i in range(n):
        _oracle_step(pool, q, kn, vn, tables[0], i % LAYERS)
    dt = time.perf_counter() - t0
    single = DECODE_BYTES * n / dt / 1e9
    cores = _host_cores()
    pools = []
    for _ in range(cores):
        pc = oracle.Pool(0, pool.num_pages, HKV, D)
        for dst, src in zip(pc.planes(), pool.planes()):
            dst[:] = src
        pools.append(pc)
    def work(j):
        _oracle_step(pools[j], q, kn, vn, tables[0], j % LAYERS)
    threads = [threading.Thread(target=work, args=(j,)) for j in range(cores)]
    t0 = time.perf_counter()
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    dtm = time.perf_counter() - t0
    del pools
    multi = DECODE_BYTES * cores / dtm / 1e9
    return {"value": round(multi, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "single_thread_value": round(single, 4),
            "sample": f"{cores} full steps (append 1 token + decode over 131072 tokens), one per host core at "
                      f"once, {dtm:.2f} s; single thread: {n} steps, {dt / n:.2f} s per step"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    oracle, pool, q, kn, vn, tables = _oracle_workload(args.seed)
    for i in range(args.warmup):
        _oracle_step(pool, q, kn, vn, tables[0], i % LAYERS)
    t0 = time.perf_counter()
    for i in range(args.steps):
        _oracle_step(pool, q, kn, vn, tables[0], i % LAYERS)
    dt = time.perf_counter() - t0
    ms = dt * 1e3 / args.steps
    value = DECODE_BYTES / (ms / 1e3) / 1e9
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded splitmix64 + Box-Muller, bf16)",
           "config": {"workload": WORKLOAD, "batch": B, "q_heads": HQ, "kv_heads": HKV, "head_dim": D,
                      "context": L, "page_size": 16, "format": "int8", "parallelism": "none (host CPU)"},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                            "sample": f"{args.steps} full steps (append 1 token + decode over 131072 tokens)"},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


# ---------------------------------------------------------------------------
# the other workloads (--workload): one JSON line each, same timing rules
# ---------------------------------------------------------------------------
DECODE_CONFIGS = {
    "int8_2k": dict(fmt="int8", HQ=16, HKV=2, D=256, L=2048),
    "k8v4_119k": dict(fmt="k8v4", HQ=16, HKV=2, D=256, L=118750),
    "iso3_82k": dict(fmt="iso3", HQ=16, HKV=4, D=128, L=81920),
    "iso4_82k": dict(fmt="iso4", HQ=16, HKV=4, D=128, L=81920),
    # the other formats at the 128K int8 shape
    "q4_128k": dict(fmt="q4", HQ=16, HKV=2, D=256, L=131072),
    "k8vbf16_128k": dict(fmt="k8vbf16", HQ=16, HKV=2, D=256, L=131072),
    "kbf16v8_128k": dict(fmt="kbf16v8", HQ=16, HKV=2, D=256, L=131072),
    # 16 query heads per KV head: one 16-column pass over the int8 cache
    "int8_128k_hq32": dict(fmt="int8", HQ=32, HKV=2, D=256, L=131072),
}


def kv_bytes_per_token(fmt, hkv, d):
    """Packed bytes read per cached token by decode (K and V codes + scales; for
    ISO4 the 2 reserved bytes per block are not counted)."""
    if fmt == "int8":
        return 2 * hkv * (d + 2 * d // 64)
    if fmt == "k8v4":
        return hkv * ((d + 2 * d // 64) + (d // 2 + 2 * d // 32))
    if fmt == "q4":
        return 2 * hkv * (d // 2 + 2 * d // 32)
    if fmt in ("k8vbf16", "kbf16v8"):
        return hkv * ((d + 2 * d // 64) + 2 * d)
    per_block = 50 if fmt == "iso3" else 66
    return 2 * hkv * (d // 128) * per_block


def _time_graph(torch, stream, fn, steps, reps, bracket=False):
    """Capture `steps` calls of fn(i) in a graph; return (ms per call over `reps`
    replays, mean ms of one call bracketed by event records or None)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(steps):
            fn(i)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(reps):
            g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    per = t0.elapsed_time(t1) / (steps * reps)
    one = None
    if bracket:
        def ev():
            try:
                return torch.cuda.Event(enable_timing=True, external=True)
            except TypeError:
                return torch.cuda.Event(enable_timing=True)
        evs = [(ev(), ev()) for _ in range(steps)]
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            for i in range(steps):
                evs[i][0].record(stream)
                fn(i)
                evs[i][1].record(stream)
        with torch.cuda.stream(stream):
            g2.replay()
            g2.replay()
        torch.cuda.synchronize()
        one = statistics.mean(a.elapsed_time(b) for a, b in evs)
    return per, one


def run_decode_config(args, name):
    import torch

    import quantized_paged_kv_append_gb300 as qkv
    from quantized_paged_kv_append_gb300 import build as qbuild
    from quantized_paged_kv_append_gb300 import synth

    cfg = DECODE_CONFIGS[name]
    fmt, hq, hkv, d, L_ = cfg["fmt"], cfg["HQ"], cfg["HKV"], cfg["D"], cfg["L"]
    qbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    bpt = kv_bytes_per_token(fmt, hkv, d)
    step_bytes = L_ * bpt
    copies = int(min(64, max(2, math.ceil(600e6 / step_bytes))))   # working set well above L2
    pages = (L_ + 15) // 16
    seed = args.seed
    k = synth.tensor_bf16(seed, "k", (L_, hkv, d), outlier_scale=20.0)
    v = synth.tensor_bf16(seed, "v", (L_, hkv, d))
    quat = synth.unit_quaternion(seed).tolist() if fmt.startswith("iso") else None
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    k_d, v_d = bf(k), bf(v)
    seq_all, pos_all = i32(np.zeros(L_, np.int32)), i32(np.arange(L_, dtype=np.int32))
    caches, tabs = [], []
    for c in range(copies):
        cache = qkv.PagedKVCache(fmt, pages, hkv, d, device=dev, quat=quat)
        t = i32(synth.page_table(seed * 100 + c, [pages])[0])
        qkv.append(cache, k_d, v_d, seq_all, pos_all, t)
        caches.append(cache)
        tabs.append(t)
    del k_d, v_d
    q_d = bf(synth.tensor_bf16(seed, "q", (copies, 1, hq, d)))
    kn_d = bf(synth.tensor_bf16(seed, "k_new", (copies, 1, hkv, d), outlier_scale=20.0))
    vn_d = bf(synth.tensor_bf16(seed, "v_new", (copies, 1, hkv, d)))
    lens = i32(np.array([L_], np.int32))
    out = torch.empty((1, hq, d), dtype=torch.bfloat16, device=dev)
    ws = qkv.decode_workspace(caches[0], 1, hq, L_, device=dev)
    stream = torch.cuda.Stream(device=dev)
    scale = 1.0 / math.sqrt(d)

    def step(i):
        c = i % copies
        qkv.decode(caches[c], q_d[c], tabs[c], lens, L_, scale=scale, out=out, workspace=ws, stream=stream,
                   k_new=kn_d[c, 0], v_new=vn_d[c, 0])

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(i)
    torch.cuda.synchronize()
    assert qkv.device_error() == 0
    proc, cpath = _clock_sampler()
    per_ms, one_ms = _time_graph(torch, stream, step, args.steps, max(3, args.reps), bracket=True)
    clocks = _clock_summary(proc, cpath, 0)
    peak, peak_kind = peaks()
    value = step_bytes / (per_ms / 1e3) / 1e9
    achieved = value   # the graph step time: main + merge launch, overlapped (see the headline line)
    kernel = f"decode_tc_kernel<{d},{min(hq // hkv, 8)},{fmt}> (+ decode_tc_combine)"
    res = {"metric": f"decode-attn packed-KV HBM GB/s, {name}", "value": round(value, 1), "unit": "GB/s",
           "n_gpus": 1, "steps": args.steps * max(3, args.reps), "warmup": max(3, args.warmup),
           "ms_per_step": round(per_ms, 5), "us_per_step": round(per_ms * 1e3, 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": fmt, "data": "synthetic (seeded splitmix64 + Box-Muller, bf16)",
           "config": {"workload": f"{fmt} KV decode, batch 1, {hq} q heads / {hkv} KV heads, head_dim {d}, "
                                  f"{L_} cached tokens, page 16, shuffled page table; step = quantize-on-write "
                                  f"of 1 token + decode", "layer_copies": copies,
                      "l2": f"inputs larger than L2: {copies} caches ({copies * step_bytes / 1e9:.2f} GB) cycled"},
           "pct_of_peak": round(100.0 * value / peak, 2),
           "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(achieved / peak, 4), "traffic": WORKLOAD_NCU_TRAFFIC.get(name),
                        "peak_kind": peak_kind, "kernel": kernel,
                        "bytes_per_launch": step_bytes,
                        "timing": "graph step time (main + merge launch per call, overlapped by programmatic "
                                  "dependent launch)"},
           "us_per_call_bracketed": round(one_ms * 1e3, 2),
           "clocks": clocks}
    print(json.dumps(res))


def run_mixed(args):
    """The serving step: 32 decode sequences (lengths uniform on [4096, 65536]),
    one extend of 2048 tokens over a 32768-token prefix, then the append of the
    2080 new tokens; int8, 16 q heads / 2 KV heads, head_dim 256. Each phase is
    timed on its own graph."""
    import torch

    import quantized_paged_kv_append_gb300 as qkv
    from quantized_paged_kv_append_gb300 import build as qbuild
    from quantized_paged_kv_append_gb300 import synth

    qbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hq, hkv, d, nb, T, L0 = 16, 2, 256, 32, 2048, 32768
    seed = args.seed
    lens = synth.seq_lengths(seed, nb, 4096, 65536)
    lmax = int(lens.max())
    pages = [int((x + 1 + 15) // 16) for x in lens] + [(L0 + T + 15) // 16]
    table, npages = synth.page_table(seed, pages)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    cache = qkv.PagedKVCache("int8", npages, hkv, d, device=dev)
    tab_d = i32(table)
    kbase = bf(synth.tensor_bf16(seed, "k", (max(lmax, L0), hkv, d), outlier_scale=20.0))
    vbase = bf(synth.tensor_bf16(seed, "v", (max(lmax, L0), hkv, d)))
    for b in range(nb + 1):
        n = int(lens[b]) if b < nb else L0
        qkv.append(cache, kbase[:n], vbase[:n], i32(np.full(n, b, np.int32)), i32(np.arange(n, dtype=np.int32)), tab_d)
    del kbase, vbase
    # decode phase (sequences 0..31; row 32 is the extend sequence)
    q_dec = bf(synth.tensor_bf16(seed, "q", (nb, hq, d)))
    lens_d = i32(lens)
    tab_dec = tab_d[:nb].contiguous()
    ws = qkv.decode_workspace(cache, nb, hq, lmax, device=dev)
    out_dec = torch.empty((nb, hq, d), dtype=torch.bfloat16, device=dev)
    # extend phase
    q_ext = bf(synth.tensor_bf16(seed, "q_ext", (T, hq, d)))
    k_ext = bf(synth.tensor_bf16(seed, "k_ext", (T, hkv, d), outlier_scale=20.0))
    v_ext = bf(synth.tensor_bf16(seed, "v_ext", (T, hkv, d)))
    cu = i32(np.array([0, T], np.int32))
    pre = i32(np.array([L0], np.int32))
    tab_ext = tab_d[nb:nb + 1].contiguous()
    out_ext = torch.empty((T, hq, d), dtype=torch.bfloat16, device=dev)
    ws_ext = qkv.extend_workspace(cache, 1, T, int(tab_ext.shape[1]), device=dev)
    # append phase: the 32 decode tokens (position L_b) and the 2048 extend tokens
    k_new = torch.cat([bf(synth.tensor_bf16(seed, "k_new", (nb, hkv, d), outlier_scale=20.0)), k_ext])
    v_new = torch.cat([bf(synth.tensor_bf16(seed, "v_new", (nb, hkv, d))), v_ext])
    seq_new = i32(np.concatenate([np.arange(nb), np.full(T, nb)]).astype(np.int32))
    pos_new = i32(np.concatenate([lens, L0 + np.arange(T)]).astype(np.int32))
    stream = torch.cuda.Stream(device=dev)
    scale = 1.0 / math.sqrt(d)
    phases = {
        "decode": lambda i: qkv.decode(cache, q_dec, tab_dec, lens_d, lmax, scale=scale, out=out_dec, workspace=ws,
                                       stream=stream),
        "extend": lambda i: qkv.extend(cache, q_ext, k_ext, v_ext, cu, pre, tab_ext, T, scale=scale, out=out_ext,
                                       stream=stream, workspace=ws_ext),
        "append": lambda i: qkv.append(cache, k_new, v_new, seq_new, pos_new, tab_d, stream=stream),
    }
    for fn in phases.values():
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i)
    torch.cuda.synchronize()
    assert qkv.device_error() == 0
    proc, cpath = _clock_sampler()
    res_ph = {}
    steps = max(10, min(args.steps, 50))
    for name, fn in phases.items():
        per_ms, _ = _time_graph(torch, stream, fn, steps, 3)
        res_ph[name] = per_ms * 1e3
    clocks = _clock_summary(proc, cpath, 0)
    peak, _ = peaks()
    tflops_peak = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"]) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else 1900.0
    dec_bytes = int(lens.sum()) * kv_bytes_per_token("int8", hkv, d)
    ext_flop = 4.0 * T * hq * d * (L0 + (T + 1) / 2)
    app_bytes = (nb + T) * hkv * (2 * d * 2 + 2 * (d + 2 * d // 64))   # bf16 K, V in; packed K, V out
    total_us = sum(res_ph.values())
    res = {"metric": "mixed serving step time (decode 32 seqs + extend 2048 over 32768 + append 2080), int8",
           "value": round(total_us, 1), "unit": "us", "n_gpus": 1, "steps": steps * 3, "warmup": 3,
           "ms_per_step": round(total_us / 1e3, 5), "higher_is_better": False, "scaling": "weak",
           "vs_baseline": None, "dtype": "int8", "data": "synthetic (seeded splitmix64 + Box-Muller, bf16)",
           "config": {"workload": "32 decode sequences, lengths uniform on [4096, 65536] (seeded), one extend of "
                                  "2048 tokens over a 32768-token prefix, then the append of the 2080 new tokens; "
                                  "int8, 16 q heads / 2 KV heads, head_dim 256, page 16",
                      "decode_tokens": int(lens.sum()), "l2": "decode reads 1.2 GB per step (inputs larger than L2)"},
           "phases_us": {k: round(v, 2) for k, v in res_ph.items()},
           "decode_gbs": round(dec_bytes / (res_ph["decode"] / 1e6) / 1e9, 1),
           "decode_pct_of_hbm_peak": round(100 * dec_bytes / (res_ph["decode"] / 1e6) / 1e9 / peak, 2),
           "extend_tflops": round(ext_flop / (res_ph["extend"] / 1e6) / 1e12, 1),
           "extend_pct_of_bf16_peak": round(100 * ext_flop / (res_ph["extend"] / 1e6) / 1e12 / tflops_peak, 2),
           "append_gbs": round(app_bytes / (res_ph["append"] / 1e6) / 1e9, 1),
           "clocks": clocks}
    print(json.dumps(res))


EXTEND_CONFIGS = {
    # format, q heads, KV heads, head_dim: the serving-step chunk (2048 new tokens over a 32768-token
    # prefix) at each format's decode shape
    "extend_k8v4": ("k8v4", 16, 2, 256),
    "extend_iso3": ("iso3", 16, 4, 128),
    "extend_iso4": ("iso4", 16, 4, 128),
    # ISO at head_dim 256 (two 128-value blocks per head), the int8 decode shape
    "extend_iso3_d256": ("iso3", 16, 2, 256),
    "extend_iso4_d256": ("iso4", 16, 2, 256),
    "extend_q4": ("q4", 16, 2, 256),
    "extend_k8vbf16": ("k8vbf16", 16, 2, 256),
    "extend_kbf16v8": ("kbf16v8", 16, 2, 256),
}


def run_extend_config(args, name):
    """Extend alone over a k8v4 / ISO prefix: prep (dequantize prefix and chunk) +
    tensor-core attention, timed as one call."""
    import torch

    import quantized_paged_kv_append_gb300 as qkv
    from quantized_paged_kv_append_gb300 import build as qbuild
    from quantized_paged_kv_append_gb300 import synth

    qbuild.build()
    fmt, hq, hkv, d = EXTEND_CONFIGS[name]
    T, L0 = 2048, 32768
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    seed = args.seed
    table, npages = synth.page_table(seed, [(L0 + T + 15) // 16])
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    quat = synth.unit_quaternion(seed).tolist() if fmt.startswith("iso") else None
    cache = qkv.PagedKVCache(fmt, npages, hkv, d, device=dev, quat=quat)
    tab = i32(table)
    qkv.append(cache, bf(synth.tensor_bf16(seed, "k", (L0, hkv, d), outlier_scale=20.0)),
               bf(synth.tensor_bf16(seed, "v", (L0, hkv, d))), i32(np.zeros(L0, np.int32)),
               i32(np.arange(L0, dtype=np.int32)), tab)
    q = bf(synth.tensor_bf16(seed, "q_ext", (T, hq, d)))
    kn = bf(synth.tensor_bf16(seed, "k_ext", (T, hkv, d), outlier_scale=20.0))
    vn = bf(synth.tensor_bf16(seed, "v_ext", (T, hkv, d)))
    cu, pre = i32(np.array([0, T], np.int32)), i32(np.array([L0], np.int32))
    out = torch.empty((T, hq, d), dtype=torch.bfloat16, device=dev)
    ws = qkv.extend_workspace(cache, 1, T, int(tab.shape[1]), device=dev)
    stream = torch.cuda.Stream(device=dev)
    scale = 1.0 / math.sqrt(d)

    def step(i):
        qkv.extend(cache, q, kn, vn, cu, pre, tab, T, scale=scale, out=out, stream=stream, workspace=ws)

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(i)
    torch.cuda.synchronize()
    assert qkv.device_error() == 0
    proc, cpath = _clock_sampler()
    steps = max(10, min(args.steps, 50))
    per_ms, _ = _time_graph(torch, stream, step, steps, 3)
    clocks = _clock_summary(proc, cpath, 0)
    tflops_peak = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"]) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else 1900.0
    flop = 4.0 * T * hq * d * (L0 + (T + 1) / 2)
    tflops = flop / (per_ms / 1e3) / 1e12
    res = {"metric": f"extend attention TFLOP/s, {name}", "value": round(tflops, 1), "unit": "TFLOP/s", "n_gpus": 1,
           "steps": steps * 3, "warmup": max(3, args.warmup), "ms_per_step": round(per_ms, 5),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16 (fp32 accumulate)",
           "data": "synthetic (seeded splitmix64 + Box-Muller, bf16)",
           "config": {"workload": f"{fmt} extend: 2048 new bf16 tokens over a 32768-token packed prefix, causal, "
                                  f"{hq} q heads / {hkv} KV heads, head_dim {d}, page 16",
                      "l2": "prefix and dequantized planes re-read per call (L2-resident working set)"},
           "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": tflops_peak, "unit": "TFLOP/s",
                        "frac": round(tflops / tflops_peak, 4), "traffic": None,
                        "kernel": "extend_prep_kernel + extend_kernel", "flop_per_launch": flop},
           "clocks": clocks}
    print(json.dumps(res))


def run_verify(args):
    """The verify window at the 128K int8 shape: 4 queries at positions L - 4 .. L - 1 of one
    sequence (the window's tokens already packed), one kv_verify_attn call per step."""
    import torch

    import quantized_paged_kv_append_gb300 as qkv
    from quantized_paged_kv_append_gb300 import build as qbuild
    from quantized_paged_kv_append_gb300 import synth

    qbuild.build()
    W = 4
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    seed = args.seed
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    pages = (L + 15) // 16
    k_d = bf(synth.tensor_bf16(seed, "k", (L, HKV, D), outlier_scale=20.0))
    v_d = bf(synth.tensor_bf16(seed, "v", (L, HKV, D)))
    caches, tabs = [], []
    for c in range(LAYERS):
        cache = qkv.PagedKVCache("int8", pages, HKV, D, device=dev)
        t = i32(synth.page_table(seed * 100 + c, [pages])[0])
        qkv.append(cache, k_d, v_d, i32(np.zeros(L, np.int32)), i32(np.arange(L, dtype=np.int32)), t)
        caches.append(cache)
        tabs.append(t)
    del k_d, v_d
    q_d = bf(synth.tensor_bf16(seed, "q_verify", (LAYERS, W, HQ, D)))
    cu, lens = i32(np.array([0, W], np.int32)), i32(np.array([L], np.int32))
    out = torch.empty((W, HQ, D), dtype=torch.bfloat16, device=dev)
    ws = qkv.verify_workspace(caches[0], HQ, W, pages, device=dev)
    stream = torch.cuda.Stream(device=dev)

    wsf = qkv.verify_fixed_workspace(caches[0], 1, W, HQ, pages, device=dev)

    def step_expanded(i):
        c = i % LAYERS
        qkv.verify(caches[c], q_d[c], cu, lens, tabs[c], L, scale=1.0 / math.sqrt(D), out=out, workspace=ws,
                   stream=stream)

    def step(i):
        # the window in one pass: its W x 8 queries per KV head as 16-column tile passes
        c = i % LAYERS
        qkv.verify_fixed(caches[c], q_d[c], lens, tabs[c], L, W, scale=1.0 / math.sqrt(D), out=out, workspace=wsf,
                         stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(i)
    torch.cuda.synchronize()
    assert qkv.device_error() == 0
    with torch.cuda.stream(stream):
        for i in range(3):
            step_expanded(i)
    torch.cuda.synchronize()
    assert qkv.device_error() == 0
    proc, cpath = _clock_sampler()
    per_ms, _ = _time_graph(torch, stream, step, args.steps, max(3, args.reps))
    exp_ms, _ = _time_graph(torch, stream, step_expanded, args.steps, max(3, args.reps))
    clocks = _clock_summary(proc, cpath, 0)
    res = {"metric": "verify window call time, int8 128K, W = 4", "value": round(per_ms * 1e3, 2), "unit": "us",
           "n_gpus": 1, "steps": args.steps * max(3, args.reps), "warmup": max(3, args.warmup),
           "ms_per_step": round(per_ms, 5), "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
           "dtype": "int8", "data": "synthetic (seeded splitmix64 + Box-Muller, bf16)",
           "config": {"workload": f"verify window of {W} queries over one {L}-token int8 sequence, {HQ} q heads / "
                                  f"{HKV} KV heads, head_dim {D}, page 16; kv_verify_attn_fixed: the window's "
                                  f"{W * HQ // HKV} queries per KV head as 16-column passes of the tensor-core "
                                  f"decode", "layer_copies": LAYERS,
                      "l2": f"inputs larger than L2: {LAYERS} caches cycled"},
           "packed_gbs_per_query": round(DECODE_BYTES * W / (per_ms / 1e3) / 1e9, 1),
           "expanded_us": round(exp_ms * 1e3, 2),   # kv_verify_attn: one decode row per query
           "clocks": clocks}
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--reps", type=int, default=5, help="graph replays of the K captured steps")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=8, help="layer caches cycled (8 keeps the working set >> L2)")
    ap.add_argument("--workload", default="int8_128k",
                    choices=["int8_128k", "mixed", "verify_int8_128k"] + sorted(DECODE_CONFIGS) + sorted(EXTEND_CONFIGS),
                    help="int8_128k (default) is the headline line; the others print their own line")
    args = ap.parse_args()
    global LAYERS
    LAYERS = max(1, args.layers)
    if args.workload != "int8_128k" and args.impl == "cuda":
        if args.workload == "mixed":
            run_mixed(args)
        elif args.workload in EXTEND_CONFIGS:
            run_extend_config(args, args.workload)
        elif args.workload == "verify_int8_128k":
            run_verify(args)
        else:
            run_decode_config(args, args.workload)
        return
    if args.impl == "reference":
        if args.steps > 10:
            args.steps = 10   # each oracle step is seconds of CPU work
        args.warmup = min(args.warmup, 3)
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
