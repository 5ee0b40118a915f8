"""Host-side helpers of bench.py (CPU only)."""

import bench


def test_traffic_only_for_the_captured_source(monkeypatch):
    key = ("c4a_decode_b64_64k", "indexer_topk")
    monkeypatch.setitem(bench.TRAFFIC, key, (123456.0, bench._kernel_digest("k_indexer_tc.cu")))
    assert bench.measured_traffic(*key) == 123456.0
    monkeypatch.setitem(bench.TRAFFIC, key, (123456.0, "0" * 64))
    assert bench.measured_traffic(*key) is None
    assert bench.measured_traffic("no_such_workload", "attention") is None


def test_call_roofline_picks_the_longer_bound():
    # 1 GB in 0.5 ms against 4000 GB/s: HBM-bound (0.25 ms at peak) at 2000 GB/s = half of peak
    r = bench.call_roofline("x", 1e9, 1e9, 0.5, 4000.0, 1000.0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 2000.0) < 1e-6 and abs(r["frac"] - 0.5) < 1e-9
    # 10 TFLOP over 1 MB: tensor-bound; 10 TFLOP in 20 ms is 500 TFLOP/s of 1000
    r = bench.call_roofline("y", 1e6, 1e13, 20.0, 4000.0, 1000.0)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 500.0) < 1e-6 and abs(r["frac"] - 0.5) < 1e-9


def test_oracle_baseline_reports_the_workers_it_ran():
    """The CPU baseline runs the oracle in single-threaded worker processes and
    reports how many it used and what the host CPU is."""
    pool = bench.OraclePool(workers=2)
    try:
        res = bench.oracle_baseline(pool, 0, seconds=3.0)
    finally:
        pool.close()
    assert res["cores"] == 2 and res["kind"] == "oracle" and res["value"] > 0
    assert res["cpu"]["logical_cpus"] >= 1 and res["cpu"]["model"]


def test_weak_throughput_counts_all_ranks():
    # 32 rows a step, 10 steps, 2 ranks, 5 ms of wall time
    assert bench.weak_throughput(32, 10, 2, 5.0) == 32 * 10 * 2 / 5e-3


def test_attention_bytes_match_the_closed_form():
    """c128a dense decode, B = 32 at p = 131072: 1024 entries + 128 window rows of
    1 KiB per row, plus 64 KiB of query and 64 KiB of output per row."""
    import types

    import numpy as np

    import synth
    wl = synth.workload(1)
    L = wl.layers[0]
    pos = np.array([s.first_new for s in wl.seqs], dtype=np.int64)
    assert np.all(pos == 131072)
    ld = types.SimpleNamespace(L=L, n_rows=len(pos), host={"pos": pos})
    assert bench.attention_bytes(ld) == 32 * ((1024 + 128) * 1024 + 2 * 64 * 512 * 2)
    assert bench.indexer_bytes(ld) == 0.0


def test_indexer_bytes_count_every_visible_key():
    import types

    import numpy as np

    import synth
    wl = synth.workload(2)
    L = wl.layers[0]
    pos = np.array([s.first_new for s in wl.seqs], dtype=np.int64)
    ld = types.SimpleNamespace(L=L, n_rows=len(pos), host={"pos": pos})
    n = sum((int(p) - L.window) // L.ratio + 1 for p in pos)
    q = len(pos) * L.idx_heads * (L.idx_dim * 2 + 4)
    assert bench.indexer_bytes(ld) == n * L.idx_dim * 2 + q + len(pos) * L.topk * 4


def test_cache_replicas_keep_every_field():
    # a partial-fp8 cache's bf16 tail must survive the replica copy
    import types

    import torch

    import compressed_sparse_long_c128a_gb300 as csa

    pc = csa.PagedCache.empty(2, 4, 64, csa.E4M3R, "cpu", 16)
    ld = types.SimpleNamespace(comp=pc, swa=pc, state=None, idx=None)
    c = bench._clone_layer(ld)
    assert c.comp.tail_bf16 == 16 and c.comp.dim == 64 and c.comp.dtype == csa.E4M3R
    assert c.comp.data.data_ptr() != pc.data.data_ptr() and torch.equal(c.comp.data, pc.data)
    assert c.state is None


def test_prefill_rows_of_one_sequence_share_their_keys():
    # four rows of one sequence at consecutive positions read the keys of the
    # longest once; two rows of other sequences read their own
    import types

    import numpy as np

    import synth
    L = synth.workload(4).layers[0]
    pos = np.array([4000, 4001, 4002, 4003, 9000, 9000], dtype=np.int64)
    seq = np.array([0, 0, 0, 0, 1, 2], dtype=np.int32)
    ld = types.SimpleNamespace(L=L, n_rows=6, host={"pos": pos, "seq_id": seq})
    nv = lambda p: (p - L.window) // L.ratio + 1
    keys = nv(4003) + 2 * nv(9000)
    q = 6 * L.idx_heads * (L.idx_dim * 2 + 4)
    assert bench.indexer_bytes(ld) == keys * L.idx_dim * 2 + q + 6 * L.topk * 4
    # attention: selections capped by the visible entries, windows as a union
    att = min(nv(4003), 4 * L.topk) + (4003 - (4000 - L.swa + 1) + 1) + 2 * (L.topk + L.swa)
    q_out = 6 * L.heads * L.dim * 2 * 2
    assert bench.attention_bytes(ld) == att * L.dim * 2 + q_out
    assert bench.attention_flops(ld) == 4.0 * L.heads * L.dim * (4 * (L.topk + L.swa) + 2 * (L.topk + L.swa))
