#!/usr/bin/env python3
"""Throughput of the compressed sparse attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 0..4] [--impl csa|reference]

One step is one pass of the hot path over one batch of the workload: for
every layer, csa_compress_insert of the step's new tokens, csa_indexer_topk
(c4a layers) and the sparse attention call.  A token is one query row that
completes that pass for one layer.  The default workload is c128a dense
decode: 32 sequences at context 131072, D=512, H=64, bf16.

Timing: W eager warm-up steps, then K steps replayed from CUDA graphs (one
graph per step) on one stream, bracketed by CUDA events with a device
synchronise (and, under torchrun, a barrier) on both sides; the max over
ranks is reported.  The step's working set is smaller than L2, so the steps
rotate over R copies of every cache with R x (bytes a step touches) > 2.5 x
L2; no step finds its inputs in L2.  The dominant kernel (sparse attention)
is timed in a second event-timed pass of K launches over the same replicas.
`e2e` repeats the step through the public API with its inputs copied from
pinned host memory and its output read back to the host every step.

Under torchrun each rank runs its own replica of the workload on its own GPU
(sequences are independent; no collective on the data path), so the scaling
is weak and value = tokens of all ranks / max time.

--side-stream runs each c4a layer's indexer and top-k on a second stream,
forked from the step's stream before compress_insert and joined before the
attention (both streams are captured into the same graph).

--impl reference times the CPU oracle on this machine's host cores on the
same workload, one bounded sample of rows per step.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "c4a/c128a sparse decode attention tokens/s; achieved HBM GB/s vs ~8 TB/s"
UNIT = "tokens/s"
L2_BYTES = 129 * 2 ** 20


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", type=int, default=1)
    ap.add_argument("--impl", choices=["csa", "reference"], default="csa")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--side-stream", action="store_true",
                    help="run each c4a layer's indexer + top-k on a second stream, beside compress_insert")
    ap.add_argument("--load-seconds", type=float, default=1.5,
                    help="untimed graph replays before the timed steps, so the clock sampler sees load")
    return ap.parse_args()


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


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


# ---------------------------------------------------------------- byte accounting

def _elem_bytes(dt: str) -> float:
    return {"f32": 4.0, "bf16": 2.0, "e4m3": 1.0, "e2m1": 0.5}[dt]


def _row_bytes(dt: str, dim: int) -> float:
    b = dim * _elem_bytes(dt)
    if dt == "e4m3":
        b += 4  # fp32 scale per row
    if dt == "e2m1":
        b += dim / 16  # e4m3 scale per 16 elements
    return b


def attention_bytes(ld) -> float:
    """Algorithmic bytes of one sparse-attention launch: every key row read once,
    queries read once, outputs written once."""
    from harness import n_visible
    L = ld.L
    keys = 0
    for p in ld.host["pos"]:
        n = n_visible(int(p), L.ratio, L.window)
        sel = min(L.topk, n) if L.has_indexer else n
        keys += sel + min(L.swa, int(p) + 1)
    q = ld.n_rows * L.heads * L.dim * _elem_bytes(L.in_dtype)
    out = ld.n_rows * L.heads * (L.dim * _elem_bytes(L.out_dtype) + (4 if L.out_dtype == "e4m3" else 0))
    return keys * _row_bytes(L.cache_dtype, L.dim) + q + out


def indexer_bytes(ld) -> float:
    from harness import n_visible
    L = ld.L
    if not L.has_indexer:
        return 0.0
    n = sum(n_visible(int(p), L.ratio, L.window) for p in ld.host["pos"])
    q = ld.n_rows * L.idx_heads * (L.idx_dim * _elem_bytes(L.in_dtype) + 4)
    return n * _row_bytes(L.idx_dtype, L.idx_dim) + q + ld.n_rows * L.topk * 4


def compress_bytes(ld) -> float:
    """Raw rows in, state + window rows out, and for each closing window its
    state rows read and its entry written."""
    L = ld.L
    from harness import n_visible  # noqa: F401
    n = ld.n_rows
    inb = n * 2 * L.dim * _elem_bytes(L.in_dtype)
    outb = n * (2 * L.dim * _elem_bytes(L.in_dtype) + _row_bytes(L.cache_dtype, L.dim))
    closing = sum(1 for p in ld.host["pos"] if p >= L.window - 1 and (p - L.window + 1) % L.ratio == 0)
    emit = closing * (L.window * 2 * L.dim * _elem_bytes(L.in_dtype) + _row_bytes(L.cache_dtype, L.dim))
    return inb + outb + emit


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

def oracle_rows_per_second(wl, seconds: float, max_rows: int | None = None):
    """Time the oracle on whole query rows of the workload (all layers per row)."""
    from oracle import SequenceOracle
    rows = [(b, r) for b, s in enumerate(wl.seqs) for r in range(s.n_new)]
    stride = max(1, len(rows) // 64)
    rows = rows[::stride]
    done = 0
    t0 = time.perf_counter()
    cache = {}
    while time.perf_counter() - t0 < seconds and (max_rows is None or done < max_rows):
        b, r = rows[done % len(rows)]
        for L in wl.layers:
            key = (L.tid, b)
            if key not in cache:
                cache.clear()
                cache[key] = SequenceOracle(wl, L, b)
            cache[key].attend(r)
        done += 1
    dt = time.perf_counter() - t0
    return done, dt


def _cores() -> int:
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return os.cpu_count() or 1


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return
    import synth
    wl = synth.workload(args.workload)
    for _ in range(args.warmup):
        oracle_rows_per_second(wl, 0.0, max_rows=1)
    t0 = time.perf_counter()
    rows = 0
    for _ in range(args.steps):
        n, _ = oracle_rows_per_second(wl, 1e9, max_rows=1)
        rows += n
    dt = time.perf_counter() - t0
    value = rows / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(wl, None),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                             "sample": f"one query row (all layers) of {wl.name} per step, fp64 numpy"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def _config(wl, replicas):
    L = wl.layers[0]
    ctx = sorted({s.first_new for s in wl.seqs})
    cfg = {"workload": wl.name, "batch": len(wl.seqs), "rows_per_step": wl.n_rows,
           "context": ctx[0] if len(ctx) == 1 else [ctx[0], ctx[-1]],
           "layers": [x.name for x in wl.layers], "dim": L.dim, "heads": L.heads, "cache": L.cache_dtype,
           "topk": L.topk or "dense", "swa": L.swa}
    if replicas is not None:
        cfg["l2"] = f"inputs larger than L2: {replicas} rotating cache replicas"
    return cfg


# ---------------------------------------------------------------- CUDA arm

def _clone_layer(ld):
    import copy
    import compressed_sparse_long_c128a_gb300 as csa
    c = copy.copy(ld)

    def cl(pc):
        if pc is None:
            return None
        return csa.PagedCache(pc.data.clone(), None if pc.scales is None else pc.scales.clone(), pc.dtype,
                              pc.rows_per_block, pc.dim)

    c.comp, c.swa, c.state, c.idx = cl(ld.comp), cl(ld.swa), cl(ld.state), cl(ld.idx)
    return c


def _launches_per_step(ld) -> int:
    """Kernel launches of one layer step, following the library's dispatch rules."""
    import compressed_sparse_long_c128a_gb300 as csa
    L = ld.L
    n = 2  # compress_insert: ingest + emit
    if L.has_indexer:
        n += 1  # scores (tensor-core or generic)
        chunks = -(-max(ld.max_n, 1) // 16384)  # top-k chunks of 16384 scores
        two_stage = 2 <= chunks <= 64 and 4 * (chunks * L.topk + chunks * L.topk // 32 + 1 + chunks * L.topk) <= 200 * 1024
        n += 2 if two_stage else 1  # chunk select (+ merge)
    tc = L.dim == 512 and L.heads == 64 and L.cache_dtype in ("bf16", "e4m3") and L.rope_dim <= 128
    if tc:
        n += 1  # one launch; split rows merge inside it
    else:
        kq = L.topk if L.has_indexer else ld.max_n
        n += 2 if csa.sparse_attn_workspace_size(ld.c_layer, ld.n_rows, kq) > 0 else 1  # (+ split merge)
    return n


def run_csa(args):
    import torch

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import compressed_sparse_long_c128a_gb300 as csa
    from compressed_sparse_long_c128a_gb300 import build as csa_build
    import synth
    from harness import WorkloadDev

    csa_build.build()
    wl = synth.workload(args.workload)
    wd = WorkloadDev(wl)
    base = wd.layers

    step_bytes = sum(attention_bytes(ld) + indexer_bytes(ld) + compress_bytes(ld) for ld in base)
    replicas = 1 if step_bytes > 2.5 * L2_BYTES else int(math.ceil(2.5 * L2_BYTES / step_bytes)) + 1
    reps = [base] + [[_clone_layer(ld) for ld in base] for _ in range(replicas - 1)]
    stream = torch.cuda.Stream()
    side = torch.cuda.Stream() if args.side_stream else None

    def step(rep, s=None):
        for ld in rep:
            ld.step(s, side_stream=side)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, replicas)):
            step(reps[i % replicas], stream)
    stream.synchronize()
    wd.check("warm-up")

    graphs = []
    for rep in reps:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(rep, stream)
        graphs.append(g)
    torch.cuda.synchronize()

    clocks = Clocks(local)
    clocks.start()
    # keep the GPU loaded for a while so the clock sampler sees it under load
    t_load = time.perf_counter()
    i = 0
    with torch.cuda.stream(stream):  # a graph replays on the current stream
        while time.perf_counter() - t_load < args.load_seconds:
            graphs[i % replicas].replay()
            i += 1
            if i % 256 == 0:
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
        for k in range(args.steps):
            graphs[k % replicas].replay()
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), world)
    rows_per_step = sum(ld.n_rows for ld in base)
    value = weak_throughput(rows_per_step, args.steps, world, ms_total)
    wd.check("timed steps")

    # dominant kernel: sparse attention of the first layer, event-timed per launch
    att_ms = []
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            ld = reps[k % replicas][0]
            io = ld.io
            L = ld.L
            topk = io.get("topk") if L.has_indexer else None
            attn = csa.sparse_attn_prefill if ld.prefill else csa.sparse_attn_decode
            ev[k][0].record(stream)
            attn(ld.c_layer, io["q"], io["seq_id"], io["pos"], ld.comp, ld.tables["comp"], topk,
                 L.topk if L.has_indexer else 0, max(ld.max_n, 1), ld.swa, ld.tables["swa"], io["out"],
                 csa.DTYPES[L.out_dtype], io["out_scales"], ld.ws_attn, ld.err, stream)
            ev[k][1].record(stream)
    torch.cuda.synchronize()
    att_ms = [a.elapsed_time(b) for a, b in ev]
    att_avg_ms = sum(att_ms) / len(att_ms)
    att_bytes = attention_bytes(base[0])
    peak, peak_src = _peaks()
    achieved = att_bytes / (att_avg_ms / 1e3) / 1e9

    e2e = None
    if not args.no_e2e:
        e2e = _e2e(args, reps, graphs, stream, rows_per_step, world, step)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": base[0].L.cache_dtype, "data": "synthetic",
            "config": _config(wl, replicas),
            "achieved_gbs_step": step_bytes / (ms_total / args.steps / 1e3) / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": _attn_traffic(wl.name), "kernel": "sparse attention",
                         "algorithmic_bytes_per_launch": att_bytes, "avg_launch_ms": att_avg_ms,
                         "peak_source": f"{peak_src} hbm_gbs (copy bandwidth, burst)"},
            "clocks": clk,
            "gpu_launches": sum(_launches_per_step(ld) for ld in base) * args.steps,
            "e2e": e2e}
    if side is not None:
        line["config"]["indexer_stream"] = "side"
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, dt = oracle_rows_per_second(wl, args.cpu_seconds)
        line["cpu_baseline"] = {"value": n / dt, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                                "sample": f"{n} query rows of {wl.name} (all layers each), fp64 numpy, "
                                          f"{dt:.1f} s"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


# DRAM bytes (read + write) of one attention launch from an ncu capture, keyed by
# workload, valid only for the kernel source it was taken on (sha256 of
# k_attn_tc.cu); see profiles/attn_tc_c128a_decode_b32.md.
ATTN_TRAFFIC = {
    "c128a_decode_b32_128k": (40027392 + 768, "c2649c649246d32f996d462908a44e4a6c7dab5bb4b687a4794092a98d9c1985"),
}


def _attn_traffic(workload_name):
    """Measured DRAM traffic per attention launch, or None when absent or taken on other source."""
    import hashlib
    entry = ATTN_TRAFFIC.get(workload_name)
    if entry is None:
        return None
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "compressed_sparse_long_c128a_gb300", "csrc",
                       "k_attn_tc.cu")
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()
    return float(entry[0]) if digest == entry[1] else None


def _e2e(args, reps, graphs, stream, rows_per_step, world, step):
    """Same steps with inputs copied from pinned host memory and the output read back every step.

    Each replica's step is captured once more as one CUDA graph that also holds
    the host-to-device copies of the step's inputs and the device-to-host copy
    of its output, as a serving loop would launch it; the host waits for every
    step's result before launching the next.  If the copies cannot be captured,
    they are issued around the replay of the kernel-only graph instead.
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
    k_steps = min(args.steps, 200)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    with torch.cuda.stream(stream):
        for k in range(k_steps):
            if full:
                full[k % len(full)].replay()
            else:
                copy_in()
                graphs[k % len(graphs)].replay()
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
