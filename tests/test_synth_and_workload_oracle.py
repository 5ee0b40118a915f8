"""The seeded generator and the oracle's per-sequence driver (CPU only)."""

import numpy as np
import pytest
import torch

import synth
from oracle import SequenceOracle
from oracle import csa_oracle as O


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(synth.round_bf16(x), ref)


def test_draws_are_deterministic_and_distinct_per_sequence():
    wl = synth.workload(0)
    L = wl.layers[0]
    a = synth.seq_raw(wl, L, 0)
    b = synth.seq_raw(wl, L, 0)
    assert a[0] == b[0] and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert not np.array_equal(a[1], a[2])
    wl2 = synth.workload(2)
    assert not np.array_equal(synth.seq_queries(wl2, wl2.layers[0], 0)[0],
                              synth.seq_queries(wl2, wl2.layers[0], 1)[0])


def test_workload_shapes():
    w0, w1, w2, w3, w4 = (synth.workload(i) for i in range(5))
    assert [s.first_new for s in w0.seqs] == [1009] and w0.seqs[0].n_new == 16
    assert len(w1.seqs) == 32 and all(s.first_new == 131072 for s in w1.seqs)
    assert len(w2.seqs) == 64 and all(32768 <= s.first_new <= 65536 for s in w2.seqs)
    assert len(w3.seqs) == 4 and all(s.first_new == 1 << 20 for s in w3.seqs)
    pre = w4.seqs[:8]
    assert all(s.n_new == 2048 and s.first_new % 4 != 0 for s in pre)
    assert [s.first_new + (-s.first_new % 128 or 128) for s in pre] == \
        [4096, 16384, 65536, 131072, 262144, 262144, 524288, 1048576]
    assert len(w4.seqs) == 32 and all(s.first_new == 65536 and s.n_new == 1 for s in w4.seqs[8:])
    assert w4.n_rows == 8 * 2048 + 24


@pytest.mark.parametrize("idx", [0, 2, 4])
def test_block_tables_are_permutations(idx):
    wl = synth.workload(idx)
    for L in wl.layers:
        for kind in synth.CACHE_KINDS:
            t, n = synth.block_table(wl, L, kind)
            used = t[t >= 0]
            assert sorted(used.tolist()) == list(range(n))
            for b, s in enumerate(wl.seqs):
                last = (s.end - 1) // synth.BLOCK_POSITIONS
                assert t[b, last] >= 0
                first = 0 if kind in ("comp", "idx") else s.raw_from(L) // synth.BLOCK_POSITIONS
                assert np.all(t[b, first:last + 1] >= 0)


def test_random_subset_distinct():
    wl = synth.workload(2)
    s = synth.random_subset(wl, wl.layers[0], 3, 0, 10000, 512)
    assert len(set(s.tolist())) == 512 and s.min() >= 0 and s.max() < 10000
    assert len(synth.random_subset(wl, wl.layers[0], 3, 0, 100, 512)) == 100


# ------------------------------------------------------------------ per-sequence oracle


def test_tiny_rows():
    wl = synth.workload(0)
    so = SequenceOracle(wl, wl.layers[0], 0)
    assert so.emitted() == list(range(0, 255))  # entries closing at tokens 7 .. 1023
    for r in (0, 7, 15):
        res = so.attend(r)
        p = 1009 + r
        assert res["p"] == p
        n = O.n_visible(p, 4, 8)
        assert len(res["entries"]) == 64 and res["entries"].max() < n
        assert res["out"].shape == (8, 128) and np.all(np.isfinite(res["out"]))


def test_future_raw_rows_do_not_reach_a_query():
    wl = synth.workload(0)
    so = SequenceOracle(wl, wl.layers[0], 0)
    r = 5
    p = 1009 + r
    base = so.attend(r)["out"]
    so.kv = so.kv.copy()
    so.gate = so.gate.copy()
    so.kv[p + 1 - so.raw_lo:] += 10.0
    so.gate[p + 1 - so.raw_lo:] -= 3.0
    np.testing.assert_array_equal(so.attend(r)["out"], base)
    # the query's own row is in its window
    so.kv[p - so.raw_lo] += 1.0
    assert not np.allclose(so.attend(r)["out"], base)


def test_history_versus_ingested_entries():
    wl = synth.workload(2)
    L = wl.layers[0]
    so = SequenceOracle(wl, L, 0)
    s = wl.seqs[0]
    em = so.emitted()
    assert em and all(s.ingest_from <= so.last_token(i) < s.end for i in em)
    old = [i for i in range(min(em) - 3, min(em))]
    assert all(so.last_token(i) < s.ingest_from for i in old)
    np.testing.assert_array_equal(so.stored_entries(old), so.history[old].astype(np.float64))
    got = so.stored_entries(em[:2])
    assert not np.allclose(got, so.history[em[:2]])
    np.testing.assert_allclose(np.sqrt(np.mean(got ** 2, axis=1)), 1.0, rtol=0.05)  # RMS-normalised


def test_dense_layer_attends_every_visible_entry():
    wl = synth.workload(1)
    so = SequenceOracle(wl, wl.layers[0], 0)
    res = so.attend(0)
    assert list(res["entries"]) == list(range(1024))
