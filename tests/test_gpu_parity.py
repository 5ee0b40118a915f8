"""Parity of the CUDA path (through the C ABI) with the oracle, on all five
synthetic workloads at their full sizes.

Inputs come from `synth` on both sides; the oracle never sees a value the
GPU produced.  Per workload:
  * caches: every entry and window row written by the set-up ingest and the
    step, and the state rows, against the oracle's values;
  * indexer cache bytes (e2m1) against the oracle's codec on the same draws;
  * top-k: index sets against the oracle's, ties within 1e-5 of the k-th
    score allowed to differ;
  * attention with a generator-drawn selection (one per row) against the
    oracle on the same selection;
  * end to end (the GPU's own selection): rows whose selection equals the
    oracle's are compared element by element;
  * one attention kernel reading a bf16 cache (a prefill call) and a partial
    token-wise fp8 cache (a decode call) of the same entries.

Tolerances: fp32 workload 1e-4 max-abs; bf16 2e-2 max-abs and 1e-2 rel-L2
against the unrounded fp64 oracle; e4m3 caches within one e4m3 step of the
oracle's code for every element and at most 0.1% of elements on another code;
e4m3 output 6e-2 max-abs / 3e-2 rel-L2, each element within one e4m3 step plus
1% of its head's amax, scales within 1%.
"""


import numpy as np
import pytest
import torch

import synth
from oracle import SequenceOracle
from oracle import csa_oracle as O
from parity_util import _assert_values, _check_topk_row, _e4m3_step

pytestmark = pytest.mark.gpu

_DEVS = {}


def _dev(idx):
    if idx not in _DEVS:
        from compressed_sparse_long_c128a_gb300 import build as csa_build
        from harness import WorkloadDev

        csa_build.build()
        _DEVS.clear()  # one workload resident at a time
        torch.cuda.empty_cache()
        wd = WorkloadDev(synth.workload(idx))
        wd.step()
        torch.cuda.synchronize()
        wd.check("first step")
        _DEVS[idx] = wd
    return _DEVS[idx]


def _rows_to_check(wl):
    """(sequence, row) pairs: every row of the decode workloads; a sample of prefill rows."""
    out = []
    for b, s in enumerate(wl.seqs):
        if s.n_new == 1:
            if len(wl.seqs) <= 64 or b % 8 == 0:
                out.append((b, 0))
        elif s.n_new <= 16:
            out += [(b, r) for r in range(s.n_new)]
        else:
            rs = {0, 1, 2, 3, 5, 127, 128, 129, 1023, 2046, 2047}
            rs |= {r for r in range(0, 24) if (s.first_new + r) % 4 == 0}  # a new entry becomes visible
            out += [(b, r) for r in sorted(rs) if r < s.n_new]
    return out


WORKLOADS = [0, 1, 2, 3, 4, 5]


@pytest.mark.parametrize("idx", WORKLOADS)
def test_caches(idx):
    wd = _dev(idx)
    wl = wd.wl
    for ld in wd.layers:
        L = ld.L
        seqs = sorted({b for b, _ in _rows_to_check(wl)})
        for b in seqs:
            s = wl.seqs[b]
            so = SequenceOracle(wl, L, b)
            # raw state rows: the ingested tokens' kv | gate, bit for bit
            pos = np.arange(s.ingest_from, s.end)
            got_state = ld.read_cache("state", b, pos)
            want_state = np.concatenate([so.kv[pos - so.raw_lo], so.gate[pos - so.raw_lo]], axis=1)
            np.testing.assert_array_equal(got_state, want_state.astype(np.float64))
            # window rows
            sw_pos = pos if len(pos) <= 300 else np.concatenate([pos[:150], pos[-150:]])
            got = ld.read_cache("swa", b, sw_pos)
            want = so.stored_swa(sw_pos)
            sc = ld.read_cache_bytes("swa", b, sw_pos)[1] if L.cache_dtype in ("e4m3", "e4m3r") else None
            _assert_values(got, want, L.cache_dtype, f"swa rows seq {b}", sc, L.rope_dim)
            # entries emitted by ingest
            em = so.emitted()
            if len(em) > 200:
                em = em[:100] + em[-100:]
            if em:
                got = ld.read_cache("comp", b, em)
                want = so.stored_entries(em)
                sc = ld.read_cache_bytes("comp", b, em)[1] if L.cache_dtype in ("e4m3", "e4m3r") else None
                _assert_values(got, want, L.cache_dtype, f"emitted entries seq {b}", sc, L.rope_dim)
            # a few history entries: stored exactly as the oracle's codec stores the draw
            if s.ingest_from > 0:
                hid = [0, 1, max(0, min(em) - 1) if em else 2]
                got = ld.read_cache("comp", b, hid)
                want = so.stored_entries(hid)
                np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("idx", [2, 3])
def test_index_cache_bytes(idx):
    wd = _dev(idx)
    wl = wd.wl
    ld = wd.layers[0]
    L = ld.L
    for b in (0, len(wl.seqs) - 1):
        keys = synth.seq_index_keys(wl, L, b)
        ids = np.unique(np.concatenate([np.arange(64), np.linspace(0, len(keys) - 1, 200).astype(np.int64)]))
        if L.idx_dtype == "e2m1":
            packed, sc = ld.read_cache_bytes("idx", b, ids)
            want_p, want_s = O.quantize_nvfp4(keys[ids])
            np.testing.assert_array_equal(O.dequantize_nvfp4(packed, sc), O.dequantize_nvfp4(want_p, want_s))
            np.testing.assert_array_equal(sc, want_s)
        else:
            np.testing.assert_array_equal(ld.read_cache("idx", b, ids), keys[ids].astype(np.float64))


def _topk_sets(wd, ld):
    return ld.io["topk"].cpu().numpy()


@pytest.mark.parametrize("idx", [0, 2, 3, 4, 5])
def test_topk(idx):
    wd = _dev(idx)
    wl = wd.wl
    ld = wd.layers[0]
    L = ld.L
    assert L.has_indexer
    topk = _topk_sets(wd, ld)
    exact = 0
    rows = _rows_to_check(wl)
    for b, r in rows:
        so = SequenceOracle(wl, L, b)
        exact += _check_topk_row(topk[ld.row_index(b, r)], so.scores(r), L.topk, f"seq {b} row {r}")
    assert exact >= len(rows) - max(1, len(rows) // 20)


def _compare_out(ld, got_all, codes, scales, row, res, what, e2e=False):
    L = ld.L
    got = got_all[row]
    if L.out_dtype == "e4m3":
        want = res["out"]
        diff = np.abs(got - want)
        rel = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert diff.max() <= 6e-2 and rel <= 3e-2, f"{what}: max-abs {diff.max():.3g} rel {rel:.3g}"
        # one e4m3 step of rounding, plus the error of the bf16 operands the tensor
        # cores take (q and P rounded to bf16): P's rounding moves an element by at
        # most 2^-9 x (a weighted mean of |K|, ~0.8), q's the weights by ~0.1%;
        # with head amax ~0.25 for these inputs, 1% of the head's amax bounds both
        sc = scales[row][:, None]
        step = np.maximum(_e4m3_step(want, sc), _e4m3_step(got, sc))
        amax = np.abs(want).max(axis=1, keepdims=True)
        assert np.all(diff <= step * 1.0001 + 1e-2 * amax), f"{what}: beyond one e4m3 step + 1% of amax"
        np.testing.assert_allclose(scales[row], res["out_scale"], rtol=1e-2)
    else:
        _assert_values(got, res["out"], L.out_dtype, what)


@pytest.mark.parametrize("idx", WORKLOADS)
def test_attention_on_drawn_selection(idx):
    wd = _dev(idx)
    wl = wd.wl
    for ld in wd.layers:
        L = ld.L
        if not L.has_indexer:
            continue  # dense layers: covered by the end-to-end test
        # rows outside the checked sample get an empty selection (window only)
        sel = np.full((ld.n_rows, L.topk), -1, dtype=np.int32)
        drawn = {}
        for b, r in _rows_to_check(wl):
            n = O.n_visible(wl.seqs[b].first_new + r, L.ratio, L.window)
            d = synth.random_subset(wl, L, b, r, n, L.topk)
            sel[ld.row_index(b, r), :len(d)] = d
            drawn[(b, r)] = d
        ld.step(topk_override=torch.from_numpy(sel).cuda())
        torch.cuda.synchronize()
        ld.check("attention on drawn selection")
        got_all, codes, scales = ld.output()
        for b, r in _rows_to_check(wl):
            so = SequenceOracle(wl, L, b)
            res = so.attend(r, entry_ids=drawn[(b, r)])
            _compare_out(ld, got_all, codes, scales, ld.row_index(b, r), res, f"{L.name} seq {b} row {r}")
        ld.step()  # restore the layer's own selection for the other tests
        torch.cuda.synchronize()


@pytest.mark.parametrize("idx", WORKLOADS)
def test_end_to_end(idx):
    wd = _dev(idx)
    wl = wd.wl
    for ld in wd.layers:
        L = ld.L
        got_all, codes, scales = ld.output()
        topk = _topk_sets(wd, ld) if L.has_indexer else None
        compared = 0
        rows = _rows_to_check(wl)
        for b, r in rows:
            so = SequenceOracle(wl, L, b)
            row = ld.row_index(b, r)
            ids = None
            if L.has_indexer:
                ref = so.topk(r)
                g = topk[row][topk[row] >= 0]
                if set(g.tolist()) != set(ref.tolist()):
                    continue  # a tie inside the band: checked by test_topk, nothing unique to compare
                ids = ref
            res = so.attend(r, entry_ids=ids)
            _compare_out(ld, got_all, codes, scales, row, res, f"{L.name} seq {b} row {r}", e2e=True)
            compared += 1
        assert compared >= len(rows) - max(1, len(rows) // 20)



def _snapshot(wd):
    snap = []
    for ld in wd.layers:
        t = {"out": ld.io["out"].clone(), "comp": ld.comp.data.clone(), "swa": ld.swa.data.clone(),
             "state": ld.state.data.clone()}
        if ld.io["out_scales"] is not None:
            t["out_scales"] = ld.io["out_scales"].clone()
        if ld.comp.scales is not None:
            t["comp_scales"] = ld.comp.scales.clone()
        if "topk" in ld.io:
            t["topk"] = ld.io["topk"].clone()
        snap.append(t)
    return snap


def _describe_diff(name, key, a, b):
    """Where two snapshots of one tensor differ (rows and heads for outputs)."""
    if key != "out" or a.dim() != 3:
        return f"{name}: {key} differs in {int((a != b).sum())} elements"
    d = (a.float() - b.float()).abs().nan_to_num(nan=1e9).amax(dim=2) > 0
    pairs = d.nonzero().cpu().numpy()
    zero_a = int((a.float().abs().amax(dim=2) == 0).sum())
    zero_b = int((b.float().abs().amax(dim=2) == 0).sum())
    return (f"{name}: out differs at {len(pairs)} (row, head) pairs, first {pairs[:8].tolist()}; "
            f"all-zero heads: {zero_a} before, {zero_b} after")


def _assert_same(wd, a_snap, b_snap, what):
    for ld, a, b in zip(wd.layers, a_snap, b_snap):
        assert a.keys() == b.keys()
        for key in a:
            assert torch.equal(a[key], b[key]), f"{what}: " + _describe_diff(ld.L.name, key, a[key], b[key])


def _run_step(wd, stream, side=None):
    """One step on `stream` (outputs and selections poisoned first), checked for
    device errors.  The snapshot's copies run on the current (default) stream,
    which a torch pool stream does not wait for, so they are complete before
    this returns: the next step's poisoning must not overtake them."""
    with torch.cuda.stream(stream):
        for ld in wd.layers:
            ld.io["out"].zero_()
            if "topk" in ld.io:
                ld.io["topk"].fill_(-2)
        wd.step(stream, side_stream=side)
    torch.cuda.synchronize()
    wd.check("two-stream step" if side is not None else "one-stream step")
    snap = _snapshot(wd)
    torch.cuda.synchronize()
    return snap


def _check_against_oracle(wd, what):
    """Every checked row of every layer against the oracle (the end-to-end comparison)."""
    wl = wd.wl
    for ld in wd.layers:
        L = ld.L
        got_all, codes, scales = ld.output()
        topk = _topk_sets(wd, ld) if L.has_indexer else None
        for b, r in _rows_to_check(wl):
            so = SequenceOracle(wl, L, b)
            row = ld.row_index(b, r)
            ids = None
            if L.has_indexer:
                ids = topk[row][topk[row] >= 0]
                _check_topk_row(topk[row], so.scores(r), L.topk, f"{what}: {L.name} seq {b} row {r}")
            res = so.attend(r, entry_ids=ids)
            _compare_out(ld, got_all, codes, scales, row, res, f"{what}: {L.name} seq {b} row {r}")


@pytest.mark.parametrize("idx", [4, 0, 2])  # 4 first: still resident from test_end_to_end
def test_two_stream_step_matches_one_stream(idx):
    """A c4a layer's indexer and top-k on a second stream, beside compress_insert
    on the first and joined before the attention: each run is checked against
    the oracle (stage-isolated on its own selection, which must be a valid
    top-k), then the two runs must have written the same bytes -- the launches
    are the same, only the order of independent ones changes (the indexer reads
    nothing compress_insert writes)."""
    wd = _dev(idx)
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    one = _run_step(wd, main)
    _check_against_oracle(wd, "one stream")
    two = _run_step(wd, main, side)
    _check_against_oracle(wd, "two streams")
    _assert_same(wd, one, two, "one vs two streams")


@pytest.mark.parametrize("idx", [4, 2, 3])
def test_step_is_deterministic(idx):
    """Re-running a step on one stream rewrites the same bytes into outputs,
    selections and caches (a step is idempotent: it re-ingests the same tokens)."""
    wd = _dev(idx)
    s = torch.cuda.Stream()
    first = _run_step(wd, s)
    for rep in range(3):
        _assert_same(wd, first, _run_step(wd, s), f"repeat {rep + 1}")
    # and on the default stream, as the other tests run it
    _assert_same(wd, first, _run_step(wd, torch.cuda.current_stream()), "default stream")


def test_device_bounds_are_reported_not_faulted():
    """An unmapped block and an out-of-range selection set the error word; the kernels skip them."""
    import compressed_sparse_long_c128a_gb300 as csa

    wd = _dev(0)
    ld = wd.layers[0]
    L = ld.L
    assert csa.read_status(ld.err) == 0
    bad = ld.tables["comp"].clone()
    bad[0, 1] = -1
    io = ld.io
    ws = torch.empty(max(1, csa.sparse_attn_workspace_size(ld.c_layer, ld.n_rows, ld.max_n)), dtype=torch.uint8,
                     device="cuda")
    csa.sparse_attn_decode(ld.c_layer, io["q"], io["seq_id"], io["pos"], ld.comp, bad, None, 0, ld.max_n,
                           ld.swa, ld.tables["swa"], io["out"], csa.F32, None, ws, ld.err)
    assert csa.read_status(ld.err) == csa.ERR_DEVICE_BOUNDS
    sel = torch.full((ld.n_rows, L.topk), -1, dtype=torch.int32, device="cuda")
    sel[:, 0] = 10 ** 6  # far beyond the visible entries
    csa.sparse_attn_decode(ld.c_layer, io["q"], io["seq_id"], io["pos"], ld.comp, ld.tables["comp"], sel,
                           L.topk, ld.max_n, ld.swa, ld.tables["swa"], io["out"], csa.F32, None, ld.ws_attn,
                           ld.err)
    assert csa.read_status(ld.err) == csa.ERR_DEVICE_BOUNDS
    assert csa.read_status(ld.err) == 0  # cleared by the previous read
    ld.step()
    torch.cuda.synchronize()
    ld.check("restored step")


def test_one_attention_kernel_reads_bf16_and_partial_fp8_caches():
    """The same attention kernel serves a prefill call on a bf16 cache and a
    decode call on a "partial token-wise fp8" cache (e4m3 non-rotary dims with
    a row scale, bf16 rotary dims) holding the same entries; each output is
    compared with the oracle attending over the values that cache stores."""
    import compressed_sparse_long_c128a_gb300 as csa

    from compressed_sparse_long_c128a_gb300 import build as csa_build

    csa_build.build()
    rng = np.random.default_rng(31)
    D, r, H, n_ent, k = 512, 64, 64, 2048, 512
    layer = csa.make_layer(4, 8, D, r, H)
    entries = rng.standard_normal((n_ent, D)).astype(np.float32)
    window = rng.standard_normal((256, D)).astype(np.float32)  # window rows of positions 0..255 of block 0
    pos = np.array([8150, 8160, 8190, 8197], dtype=np.int32)    # queries see entries < n_visible(p)
    n_rows = len(pos)
    q = torch.from_numpy(synth.round_bf16(rng.standard_normal((n_rows, H, D)))).to(torch.bfloat16).cuda()
    sel = np.stack([rng.choice(O.n_visible(int(p), 4, 8), size=k, replace=False) for p in pos]).astype(np.int32)
    comp_bt = torch.arange(32, dtype=torch.int32).reshape(1, 32).cuda()
    # the window rows of every position live in the SWA cache's block = position // 256
    swa_bt = torch.zeros((1, 33), dtype=torch.int32).cuda()
    seq = torch.zeros(n_rows, dtype=torch.int32).cuda()
    err = torch.zeros(1, dtype=torch.int32).cuda()
    results = {}
    for dtype, tail, call in (("bf16", 0, csa.sparse_attn_prefill), ("e4m3r", r, csa.sparse_attn_decode)):
        dt = csa.DTYPES[dtype]
        comp = csa.PagedCache.empty(32, 64, D, dt, "cuda", tail)
        swa = csa.PagedCache.empty(1, 256, D, dt, "cuda", tail)
        csa.cache_store(torch.from_numpy(entries).cuda(), torch.zeros(n_ent, dtype=torch.int32).cuda(),
                        torch.arange(n_ent, dtype=torch.int32).cuda(), comp, comp_bt, err)
        swa_rows = torch.arange(256, dtype=torch.int32).cuda()
        csa.cache_store(torch.from_numpy(window).cuda(), torch.zeros(256, dtype=torch.int32).cuda(), swa_rows, swa,
                        swa_bt, err)
        out = torch.zeros((n_rows, H, D), dtype=torch.bfloat16).cuda()
        ws = torch.empty(max(1, csa.sparse_attn_workspace_size(layer, n_rows, k)), dtype=torch.uint8).cuda()
        call(layer, q, seq, torch.from_numpy(pos).cuda(), comp, comp_bt, torch.from_numpy(sel).cuda(), k, n_ent, swa,
             swa_bt, out, csa.BF16, None, ws, err)
        torch.cuda.synchronize()
        assert csa.read_status(err) == 0, dtype
        results[dtype] = out.to(torch.float64).cpu().numpy()
    qh = q.to(torch.float64).cpu().numpy()
    for dtype, tail in (("bf16", 0), ("e4m3r", r)):
        if dtype == "bf16":
            stored_ent = synth.round_bf16(entries).astype(np.float64)
            stored_win = synth.round_bf16(window).astype(np.float64)
        else:
            stored_ent = O.dequantize_rows_e4m3_rope_bf16(*O.quantize_rows_e4m3_rope_bf16(entries, r))
            stored_win = O.dequantize_rows_e4m3_rope_bf16(*O.quantize_rows_e4m3_rope_bf16(window, r))
        for i, p in enumerate(pos):
            # window rows [p-127, p] are positions of block p // 256 -- all mapped to block 0 by swa_bt
            wpos = np.asarray(O.swa_positions(int(p), 128))
            keys = np.concatenate([stored_ent[sel[i]], stored_win[wpos % 256]])
            want = O.attention(qh[i], int(p), keys, D ** -0.5, r, 10000.0)
            _assert_values(results[dtype][i], want, "bf16", f"{dtype} cache, row {i}")

