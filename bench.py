#!/usr/bin/env python3
"""Throughput of the compressed sparse attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 0..4] [--extra 1,3,4|none]
                    [--impl csa|reference]

One step is one pass of the hot path over one batch of a workload: for every
layer, csa_compress_insert of the step's new tokens, csa_indexer_topk (c4a
layers) and the sparse attention call.  A token is one query row that
completes that pass for one layer.  On a c4a layer compress_insert runs on a
second stream beside the indexer and top-k, joined before the attention (the
multi-stream split of the decode path; --one-stream puts every call on one
stream).

The headline workload is c4a DSA decode: 64 sequences at contexts uniform in
[32768, 65536], D=512, H=64, indexer 64 heads x 128 dims, top-512, bf16.  The
other full-size workloads are measured the same way and reported under
"configs" (c128a dense decode at 131072; c4a decode at 2^20 with the fp8
attention cache and fp4 indexer cache; mixed chunked prefill + decode with a
c4a and a c128a layer; the c4a decode on the partial token-wise fp8 cache).

Timing: W eager warm-up steps, then K steps replayed from CUDA graphs (a
few consecutive steps per graph, as a serving loop captures consecutive
layers) on one stream, bracketed by CUDA events with a device
synchronise (and, under torchrun, a barrier) on both sides; the max over
ranks is reported.  When a step's working set is smaller than L2 the steps
rotate over R copies of every cache with R x (bytes a step touches) >
2.5 x L2, so no step finds its inputs in L2.  Each call of the step is then
event-timed on its own over the same rotation, for the per-call roofline; the
dominant call's (the longest) is the line's `roofline`.  `e2e` repeats the
step with its inputs copied from pinned host memory and its output read back
to the host every step.  `gpu_launches` is the library's launches captured
into the step graphs (its own host-side count) times the steps replayed.

Under torchrun each rank runs its own replica of the workload on its own GPU
(sequences are independent; no collective on the data path), so the scaling
is weak and value = tokens of all ranks / max time.

`cpu_baseline` and `--impl reference` time the CPU oracle (fp64 numpy) on
this machine's host cores: a pool of one single-threaded worker process per
core, each answering whole query rows of the same workload.
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "c4a/c128a sparse decode attention tokens/s; achieved HBM GB/s vs ~8 TB/s"
UNIT = "tokens/s"
L2_BYTES = 129 * 2 ** 20
HEADLINE = 2
EXTRA = (1, 3, 4, 5)


def _args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", type=int, default=HEADLINE)
    ap.add_argument("--extra", default=",".join(str(i) for i in EXTRA),
                    help="comma-separated workloads also measured and reported under 'configs', or 'none'")
    ap.add_argument("--extra-steps", type=int, default=200, help="timed steps of each extra workload (at most K)")
    ap.add_argument("--impl", choices=["csa", "reference"], default="csa")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--reference-seconds", type=float, default=150.0,
                    help="the reference arm stops after this many seconds of timed steps")
    ap.add_argument("--one-stream", action="store_true",
                    help="run every call of a c4a layer on one stream (default: compress_insert on a second "
                         "stream, beside the indexer + top-k)")
    ap.add_argument("--load-seconds", type=float, default=1.5,
                    help="untimed graph replays before the timed steps, so the clock sampler sees load")
    return ap.parse_args(argv)


def _extras(args):
    if args.extra in ("", "none"):
        return []
    return [int(x) for x in args.extra.split(",") if int(x) != args.workload]


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


def max_over_ranks(x: float, world: int, device="cuda") -> float:
    """The largest value of x over all ranks (every rank gets it)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_throughput(units_per_rank: int, steps: int, world: int, ms_max: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank."""
    return units_per_rank * steps * world / (ms_max / 1e3)


# ---------------------------------------------------------------- algorithmic bytes and flops

def _elem_bytes(dt: str) -> float:
    return {"f32": 4.0, "bf16": 2.0, "e4m3": 1.0, "e2m1": 0.5}[dt]


def _row_bytes(dt: str, dim: int, tail: int = 64) -> float:
    if dt == "e4m3r":  # e4m3 codes + fp32 scale, the rotary tail in bf16
        return (dim - tail) + 2 * tail + 4
    b = dim * _elem_bytes(dt)
    if dt == "e4m3":
        b += 4  # fp32 scale per row
    if dt == "e2m1":
        b += dim / 16  # e4m3 scale per 16 elements
    return b


def _by_sequence(ld):
    """Positions of the step's rows grouped by sequence (each row its own
    sequence when the rows carry no sequence ids)."""
    pos = [int(p) for p in ld.host["pos"]]
    seq = ld.host.get("seq_id") if isinstance(ld.host, dict) else None
    if seq is None:
        return [[p] for p in pos]
    groups = {}
    for b, p in zip(seq, pos):
        groups.setdefault(int(b), []).append(p)
    return list(groups.values())


def _union_len(intervals) -> int:
    """Integers covered by closed intervals [lo, hi]."""
    total, end = 0, None
    for lo, hi in sorted(intervals):
        if end is None or lo > end:
            total += hi - lo + 1
            end = hi
        elif hi > end:
            total += hi - end
            end = hi
    return total


def _attended_keys(ld) -> int:
    """Distinct key rows the attention must read: per sequence, its rows'
    selected (c4a) or visible (c128a) entries, at most every visible entry, and
    the union of its rows' windows.  One row per sequence (decode) gives each
    row's selection + window."""
    from harness import n_visible
    L = ld.L
    keys = 0
    for ps in _by_sequence(ld):
        n_max = max(n_visible(p, L.ratio, L.window) for p in ps)
        if L.has_indexer:
            keys += min(n_max, sum(min(L.topk, n_visible(p, L.ratio, L.window)) for p in ps))
        else:
            keys += n_max
        keys += _union_len([(max(0, p - L.swa + 1), p) for p in ps])
    return keys


def _attended_pairs(ld) -> int:
    """(row, key) pairs of the attention: the work of its contractions."""
    from harness import n_visible
    L = ld.L
    keys = 0
    for p in ld.host["pos"]:
        n = n_visible(int(p), L.ratio, L.window)
        sel = min(L.topk, n) if L.has_indexer else n
        keys += sel + min(L.swa, int(p) + 1)
    return keys


def attention_bytes(ld) -> float:
    """Algorithmic bytes of one sparse-attention launch: every distinct key row
    read once, queries read once, outputs written once."""
    L = ld.L
    q = ld.n_rows * L.heads * L.dim * _elem_bytes(L.in_dtype)
    out = ld.n_rows * L.heads * (L.dim * _elem_bytes(L.out_dtype) + (4 if L.out_dtype == "e4m3" else 0))
    return _attended_keys(ld) * _row_bytes(L.cache_dtype, L.dim) + q + out


def attention_flops(ld) -> float:
    """q.k and p.v for every head of every row over every key it attends."""
    L = ld.L
    return 4.0 * L.heads * L.dim * _attended_pairs(ld)


def _visible_sum(ld) -> int:
    from harness import n_visible
    L = ld.L
    return sum(n_visible(int(p), L.ratio, L.window) for p in ld.host["pos"])


def indexer_bytes(ld) -> float:
    """Every visible indexer key of each sequence read once (the rows of one
    sequence share theirs), the indexer queries and weights read once, the
    selection written once (score scratch not counted)."""
    from harness import n_visible
    L = ld.L
    if not L.has_indexer:
        return 0.0
    keys = sum(max(n_visible(p, L.ratio, L.window) for p in ps) for ps in _by_sequence(ld))
    q = ld.n_rows * L.idx_heads * (L.idx_dim * _elem_bytes(L.in_dtype) + 4)
    return keys * _row_bytes(L.idx_dtype, L.idx_dim) + q + ld.n_rows * L.topk * 4


def indexer_flops(ld) -> float:
    L = ld.L
    return 2.0 * L.idx_heads * L.idx_dim * _visible_sum(ld) if L.has_indexer else 0.0


def compress_bytes(ld) -> float:
    """Raw rows in, state + window rows out, and for each closing window its
    state rows read and its entry written."""
    L = ld.L
    n = ld.n_rows
    inb = n * 2 * L.dim * _elem_bytes(L.in_dtype)
    outb = n * (2 * L.dim * _elem_bytes(L.in_dtype) + _row_bytes(L.cache_dtype, L.dim))
    closing = sum(1 for p in ld.host["pos"] if p >= L.window - 1 and (p - L.window + 1) % L.ratio == 0)
    emit = closing * (L.window * 2 * L.dim * _elem_bytes(L.in_dtype) + _row_bytes(L.cache_dtype, L.dim))
    return inb + outb + emit


def call_roofline(name: str, nbytes: float, flops: float, ms: float, hbm_gbs: float, tflops: float,
                  traffic=None) -> dict:
    """Roofline of one call: bound by HBM or by the tensor pipe, whichever takes longer at peak."""
    t_hbm = nbytes / (hbm_gbs * 1e9)
    t_tc = flops / (tflops * 1e12)
    if t_tc > t_hbm:
        achieved = flops / (ms / 1e3) / 1e12
        return {"call": name, "bound": "tensor", "achieved": achieved, "peak": tflops, "unit": "TFLOP/s",
                "frac": achieved / tflops, "traffic": traffic, "algorithmic_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": ms}
    achieved = nbytes / (ms / 1e3) / 1e9
    return {"call": name, "bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
            "frac": achieved / hbm_gbs, "traffic": traffic, "algorithmic_bytes_per_launch": nbytes,
            "algorithmic_flops_per_launch": flops, "avg_launch_ms": ms}


# DRAM bytes (read + write) per launch of a call from an ncu capture, keyed by
# (workload, call); valid only for the kernel source it was taken on (sha256 of
# the call's kernel file).
TRAFFIC = {
    # ncu --set full --clock-control none, one launch of indexer_tc_kernel on the workload
    ("c4a_decode_b64_64k", "indexer_topk"): (199313920.0 + 5145344.0, "fe4c3295e7a072e78f961bd38cb71df3da34e45b3ecb7d051c5bbc4ba9797f3c"),
    # the same for one launch of attn_tc_kernel
    ("c128a_decode_b32_128k", "attention"): (40029696.0 + 3328.0, "4fdeee2cb2e6e8999e370c0ccbcd24f37fdcc26d1980a1d01873efd6f1f68d19"),
    # the same for one launch of the e2m1 indexer_tc_kernel
    ("c4a_decode_b4_1m_fp8", "indexer_topk"): (75728896.0 + 1843968.0, "fe4c3295e7a072e78f961bd38cb71df3da34e45b3ecb7d051c5bbc4ba9797f3c"),
}
_CALL_SOURCE = {"attention": "k_attn_tc.cu", "indexer_topk": "k_indexer_tc.cu", "compress_insert": "k_compress.cu"}


def _kernel_digest(name="k_attn_tc.cu"):
    """sha256 of a kernel source file as it stands."""
    import hashlib
    src = os.path.join(ROOT, "compressed_sparse_long_c128a_gb300", "csrc", name)
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def measured_traffic(workload_name: str, call: str):
    """Measured DRAM traffic per launch, or None when absent or taken on another source."""
    entry = TRAFFIC.get((workload_name, call))
    if entry is None:
        return None
    return float(entry[0]) if _kernel_digest(_CALL_SOURCE[call]) == entry[1] else None


# ---------------------------------------------------------------- clocks

class Clocks:
    """nvidia-smi samples every 200 ms while the GPU is under load."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


# ---------------------------------------------------------------- CPU oracle timing

def host_cpu() -> dict:
    """The host's CPU model and core count (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.TimeoutExpired):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
    return {"model": model or platform.processor() or "unknown", "machine": platform.machine(),
            "logical_cpus": os.cpu_count() or 1}


def _sample_rows(wl, n: int):
    """An evenly spaced sample of n query rows (sequence, row) of the workload."""
    rows = [(b, r) for b, s in enumerate(wl.seqs) for r in range(s.n_new)]
    stride = max(1, len(rows) // max(n, 1))
    return rows[::stride][:n] if n else rows


def _oracle_worker(job):
    """One worker of the pool: answer query rows with the oracle until the deadline.

    job = (workload index, [(sequence, row), ...], wall-clock deadline or None).
    Returns the number of rows answered (every layer of each row)."""
    wl_idx, rows, deadline = job
    import synth
    from oracle import SequenceOracle
    wl = synth.workload(wl_idx)
    cache = {}
    done = 0
    for b, r in rows:
        if deadline is not None and time.time() >= deadline:
            break
        for L in wl.layers:
            key = (L.tid, b)
            if key not in cache:
                cache.clear()
                cache[key] = SequenceOracle(wl, L, b)
            cache[key].attend(r)
        done += 1
    return done


class OraclePool:
    """Single-threaded oracle workers, one per host core, started with spawn."""

    def __init__(self, workers: int | None = None):
        import multiprocessing as mp
        self.workers = workers or (os.cpu_count() or 1)
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"  # inherited by the spawned workers: one thread each
        try:
            self.pool = mp.get_context("spawn").Pool(self.workers)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def run(self, wl_idx: int, rows, deadline=None) -> int:
        """Rows of `rows` answered; rows are dealt to workers by sequence, so each reuses its set-up."""
        by_seq = {}
        for b, r in rows:
            by_seq.setdefault(b, []).append((b, r))
        jobs = [[] for _ in range(self.workers)]
        for i, seq_rows in enumerate(sorted(by_seq.values(), key=len, reverse=True)):
            min(jobs, key=len).extend(seq_rows)
        jobs = [(wl_idx, j, deadline) for j in jobs if j]
        return sum(self.pool.map(_oracle_worker, jobs))

    def close(self):
        self.pool.terminate()
        self.pool.join()


def oracle_baseline(pool: OraclePool, wl_idx: int, seconds: float) -> dict:
    """Rows per second of the oracle on the pool, over a bounded sample of the workload."""
    import synth
    wl = synth.workload(wl_idx)
    rows = _sample_rows(wl, 64 * pool.workers)
    t0 = time.time()
    n = passes = 0
    while passes == 0 or time.time() - t0 < 0.9 * seconds:  # whole passes over the sample, about `seconds` long
        n += pool.run(wl_idx, rows, deadline=t0 + seconds)
        passes += 1
    dt = time.time() - t0
    return {"value": n / dt, "unit": UNIT, "cores": pool.workers, "kind": "oracle",
            "sample": f"{n} query rows of {wl.name} ({passes} passes over {len(rows)} rows spread evenly over "
                      f"the batch; every layer of each row), fp64 numpy, {pool.workers} single-threaded worker "
                      f"processes, {dt:.1f} s",
            "cpu": host_cpu()}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return
    import synth
    wl = synth.workload(args.workload)
    pool = OraclePool()
    try:
        rows = _sample_rows(wl, 64 * pool.workers)
        per_step = pool.workers  # one row per worker and step
        for i in range(args.warmup):
            pool.run(args.workload, rows[(i * per_step) % len(rows):][:per_step])
        t0 = time.time()
        steps = n = 0
        while steps < args.steps and time.time() - t0 < args.reference_seconds:
            k = (steps * per_step) % len(rows)
            n += pool.run(args.workload, (rows[k:] + rows[:k])[:per_step])
            steps += 1
        dt = time.time() - t0
    finally:
        pool.close()
    value = n / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": steps, "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / max(steps, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": _config(wl, None),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.workers, "kind": "oracle",
                             "sample": f"{n} query rows of {wl.name} in {steps} steps of {per_step} rows "
                                       f"(every layer of each row), fp64 numpy, {pool.workers} single-threaded "
                                       f"worker processes", "cpu": host_cpu()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def _config(wl, replicas):
    L = wl.layers[0]
    ctx = sorted({s.first_new for s in wl.seqs})
    cfg = {"workload": wl.name, "batch": len(wl.seqs), "rows_per_step": wl.n_rows,
           "context": ctx[0] if len(ctx) == 1 else [ctx[0], ctx[-1]],
           "layers": [x.name for x in wl.layers], "dim": L.dim, "heads": L.heads, "cache": L.cache_dtype,
           "indexer_cache": L.idx_dtype if L.has_indexer else None, "out": L.out_dtype,
           "topk": L.topk or "dense", "swa": L.swa}
    if replicas is not None:
        cfg["l2"] = (f"inputs larger than L2: {replicas} rotating cache replicas" if replicas > 1
                     else "inputs larger than L2: the step's working set exceeds 2.5 x L2")
    return cfg


# ---------------------------------------------------------------- CUDA arm

def _clone_layer(ld):
    import copy
    import compressed_sparse_long_c128a_gb300 as csa
    c = copy.copy(ld)

    def cl(pc):
        if pc is None:
            return None
        return dataclasses.replace(pc, data=pc.data.clone(), scales=None if pc.scales is None else pc.scales.clone())

    c.comp, c.swa, c.state, c.idx = cl(ld.comp), cl(ld.swa), cl(ld.state), cl(ld.idx)
    return c


def _call_fns(ld, csa, stream):
    """The step's calls of one layer, as (name, fn) in step order."""
    L, io = ld.L, ld.io
    fns = [("compress_insert", lambda: ld.compress_insert(io["kv"], io["gate"], io["seq_id"], io["pos"], stream))]
    if L.has_indexer:
        fns.append(("indexer_topk", lambda: csa.indexer_topk(
            io["q_idx"], io["w"], io["seq_id"], io["pos"], L.ratio, L.window, ld.idx, ld.tables["idx"], L.topk,
            max(ld.max_n, 1), io["topk"], ld.ws_idx, ld.err, stream)))
    attn = csa.sparse_attn_prefill if ld.prefill else csa.sparse_attn_decode
    topk = io["topk"] if L.has_indexer else None
    fns.append(("attention", lambda: attn(
        ld.c_layer, io["q"], io["seq_id"], io["pos"], ld.comp, ld.tables["comp"], topk,
        L.topk if L.has_indexer else 0, max(ld.max_n, 1), ld.swa, ld.tables["swa"], io["out"],
        csa.DTYPES[L.out_dtype], io["out_scales"], ld.ws_attn, ld.err, stream)))
    return fns


def measure_workload(idx: int, args, steps: int, world: int, local: int, pool=None, headline=False) -> dict:
    """Time one workload: K graph-replayed steps, each call alone, e2e, and the CPU baseline."""
    import torch

    import compressed_sparse_long_c128a_gb300 as csa
    import synth
    from harness import WorkloadDev

    hbm, tflops, peak_src = _peaks()
    wl = synth.workload(idx)
    wd = WorkloadDev(wl)
    base = wd.layers
    step_bytes = sum(attention_bytes(ld) + indexer_bytes(ld) + compress_bytes(ld) for ld in base)
    replicas = 1 if step_bytes > 2.5 * L2_BYTES else int(math.ceil(2.5 * L2_BYTES / step_bytes)) + 1
    reps = [base] + [[_clone_layer(ld) for ld in base] for _ in range(replicas - 1)]
    stream = torch.cuda.Stream()
    side = None if args.one_stream else torch.cuda.Stream()

    def step(rep, s=None):
        for ld in rep:
            ld.step(s, side_stream=side)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, replicas)):
            step(reps[i % replicas], stream)
    stream.synchronize()
    wd.check("warm-up")

    # consecutive steps are captured together (as a serving loop captures its
    # layers), cycling over the replicas: `spg` steps per graph, and one more
    # graph for the remainder so that exactly `steps` steps are timed
    spg = replicas * max(1, -(-8 // replicas)) if step_bytes < 2 ** 30 else replicas

    def capture(n_steps):
        g = torch.cuda.CUDAGraph()
        n0 = csa.launch_count()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_steps):
                step(reps[i % replicas], stream)
        return g, csa.launch_count() - n0  # the library's kernels in the graph

    full, full_launches = capture(spg)
    n_full, n_rest = divmod(steps, spg)
    rest, rest_launches = capture(n_rest) if n_rest else (None, 0)
    torch.cuda.synchronize()
    kernels_per_step = full_launches // spg

    clocks = Clocks(local)
    clocks.start()
    t_load = time.perf_counter()
    i = 0
    with torch.cuda.stream(stream):  # a graph replays on the current stream
        while time.perf_counter() - t_load < args.load_seconds:
            full.replay()
            i += 1
            if i % 8 == 0:
                stream.synchronize()
    stream.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(n_full):
            full.replay()
        if rest is not None:
            rest.replay()
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), world)
    rows_per_step = sum(ld.n_rows for ld in base)
    value = weak_throughput(rows_per_step, steps, world, ms_total)
    wd.check("timed steps")

    # every call of every layer on its own: n_call launches of it over the same
    # rotation, captured into one graph, replayed between two events (no host gaps)
    n_call = max(3, min(steps, 200 if replicas > 1 else 20))
    n_call = -(-n_call // replicas) * replicas
    calls = {}
    for li in range(len(base)):
        for ci, (name, _) in enumerate(_call_fns(base[li], csa, stream)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for k in range(n_call):
                    _call_fns(reps[k % replicas][li], csa, stream)[ci][1]()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                g.replay()  # warm
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / n_call
            del g
            ld = base[li]
            if name == "attention":
                nb, fl = attention_bytes(ld), attention_flops(ld)
            elif name == "indexer_topk":
                nb, fl = indexer_bytes(ld), indexer_flops(ld)
            else:
                nb, fl = compress_bytes(ld), 0.0
            key = f"{ld.L.name}.{name}" if len(base) > 1 else name
            calls[key] = call_roofline(key, nb, fl, ms, hbm, tflops, measured_traffic(wl.name, name))
    wd.check("per-call timing")
    dominant = max(calls.values(), key=lambda c: c["avg_launch_ms"])

    del full, rest
    e2e = None if args.no_e2e else _e2e(min(steps, 200), reps, stream, rows_per_step, world, step)
    res = {"value": value, "unit": UNIT, "steps": steps, "ms_per_step": ms_total / steps,
           "dtype": base[0].L.cache_dtype, "config": _config(wl, replicas),
           "achieved_gbs_step": step_bytes / (ms_total / steps / 1e3) / 1e9,
           "algorithmic_bytes_per_step": step_bytes,
           "roofline": dict(dominant, peak_source=f"{peak_src} (copy bandwidth / cuBLAS bf16, burst)"),
           "calls": calls, "clocks": clk,
           "gpu_launches": n_full * full_launches + rest_launches,
           "kernels_per_step": kernels_per_step, "steps_per_graph": spg, "e2e": e2e}
    if side is not None and any(ld.L.has_indexer for ld in base):
        res["config"]["streams"] = "compress_insert on a second stream, beside indexer_topk"
    if pool is not None:
        res["cpu_baseline"] = oracle_baseline(pool, idx, args.cpu_seconds)
    del reps, base, wd
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_csa(args):
    import torch

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from compressed_sparse_long_c128a_gb300 import build as csa_build

    csa_build.build()
    pool = OraclePool() if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    try:
        head = measure_workload(args.workload, args, args.steps, world, local, pool, headline=True)
        extra = {}
        for idx in _extras(args):
            r = measure_workload(idx, args, max(3, min(args.steps, args.extra_steps)), world, local, pool)
            extra[r["config"]["workload"]] = r
    finally:
        if pool is not None:
            pool.close()
    line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
            "config": head["config"], "roofline": head["roofline"], "clocks": head["clocks"],
            "gpu_launches": head["gpu_launches"], "e2e": head["e2e"],
            "achieved_gbs_step": head["achieved_gbs_step"], "calls": head["calls"],
            "kernels_per_step": head["kernels_per_step"]}
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if extra:
        line["configs"] = extra
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def _e2e(k_steps, reps, stream, rows_per_step, world, step):
    """Same steps with inputs copied from pinned host memory and the output read back every step.

    Each replica's step is captured once more as one CUDA graph that also holds
    the host-to-device copies of the step's inputs and the device-to-host copy
    of its output, as a serving loop would launch it; the host waits for every
    step's result before launching the next.  If the copies cannot be captured,
    the step is issued eagerly between them instead.
    """
    import torch
    base = reps[0]
    host_in, host_out = [], []
    for ld in base:
        hin = {k: ld.io[k].cpu().pin_memory() for k in ("seq_id", "pos", "kv", "gate", "q", "q_idx", "w")
               if k in ld.io}
        host_in.append(hin)
        hout = [ld.io["out"].cpu().pin_memory()]
        if ld.io["out_scales"] is not None:
            hout.append(ld.io["out_scales"].cpu().pin_memory())
        host_out.append(hout)
    bi = sum(t.numel() * t.element_size() for h in host_in for t in h.values())
    bo = sum(t.numel() * t.element_size() for h in host_out for t in h)

    def copy_in():
        for ld, hin in zip(base, host_in):  # replicas share the step's io buffers
            for key, t in hin.items():
                ld.io[key].copy_(t, non_blocking=True)

    def copy_out():
        for ld, hout in zip(base, host_out):
            hout[0].copy_(ld.io["out"], non_blocking=True)
            if len(hout) > 1:
                hout[1].copy_(ld.io["out_scales"], non_blocking=True)

    full = []
    try:
        for rep in reps:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                copy_in()
                step(rep, stream)
                copy_out()
            full.append(g)
        torch.cuda.synchronize()
    except RuntimeError:
        full = []
        torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    with torch.cuda.stream(stream):
        for k in range(k_steps):
            if full:
                full[k % len(full)].replay()
            else:
                copy_in()
                step(reps[k % len(reps)], stream)
                copy_out()
            stream.synchronize()  # the host reads the step's result
    t1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), world)
    return {"value": weak_throughput(rows_per_step, k_steps, world, ms), "unit": UNIT, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "steps": k_steps, "copies_in_graph": bool(full)}


def main():
    args = _args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_csa(args)


if __name__ == "__main__":
    main()
