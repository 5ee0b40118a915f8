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
