"""Host-side helpers of bench.py (CPU only)."""

import bench


def test_attention_traffic_only_for_the_captured_source(monkeypatch):
    name = "c128a_decode_b32_128k"
    assert name in bench.ATTN_TRAFFIC
    nbytes, digest = bench.ATTN_TRAFFIC[name]
    # the committed entry describes the kernel source as it stands
    assert bench._attn_traffic(name) == float(nbytes)
    monkeypatch.setitem(bench.ATTN_TRAFFIC, name, (nbytes, "0" * 64))
    assert bench._attn_traffic(name) is None
    assert bench._attn_traffic("no_such_workload") is None


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


def _layer_stand_in(wl, L):
    """What _launches_per_step reads of a device layer, without a device."""
    import types

    import compressed_sparse_long_c128a_gb300 as csa
    from harness.device import n_visible

    pos = [p for s in wl.seqs for p in range(s.first_new, s.end)]
    return types.SimpleNamespace(L=L, n_rows=len(pos), max_n=max(n_visible(p, L.ratio, L.window) for p in pos),
                                 c_layer=csa.make_layer(L.ratio, L.window, L.dim, L.rope_dim, L.heads, L.swa,
                                                        L.theta, L.eps))


def test_launch_count_matches_the_launch_lists():
    """Kernel launches per step, from the dispatch rules, against what ncu listed per
    step: c128a decode 3 (ingest, emit, attention), c4a decode 5 (+ indexer, one top-k
    chunk launch), c4a at 2^20 with the fp4 indexer 6 (+ the top-k merge)."""
    import synth

    for idx, want in ((1, 3), (2, 5), (3, 6)):
        wl = synth.workload(idx)
        got = sum(bench._launches_per_step(_layer_stand_in(wl, L)) for L in wl.layers)
        assert got == want, f"workload {idx}: {got} launches per step, the launch list shows {want}"
