"""Every query row of two prefill chunks of the mixed workload, on both layers.

The mixed prefill/decode workload carries 2048-token prefill chunks at contexts
from 4k to 1M.  The parity tests compare a sample of their rows; here every one
of the 2048 rows of the 4k-context chunk (sequence 0) and of the 1M-context
chunk (sequence 7) is compared, for the c4a layer and the c128a layer, over
eight of the 64 heads (the heads are independent given the shared keys, so a
fault confined to some heads would still show unless it spares all eight;
0, 9, ..., 63 reach every 8-head group of the attention kernel's tiles).

  * c128a (dense over the visible entries): end to end against the oracle,
    every row, both chunks.
  * c4a, 4k chunk: end to end.  Every row's selection is checked against the
    oracle's scores (exact up to ties within 1e-5 of the k-th score), and the
    attention over the GPU's selection against the oracle: where the selection
    equals the oracle's (all rows but ties) that is the end-to-end value.
  * c4a, 1M chunk: stage-isolated.  The oracle's scores over 262k entries cost
    about a second per row, so every row's selection is checked for its form
    (k distinct visible entries) and its attention against the oracle on that
    selection; the selection itself against the scores on rows spread over the
    chunk (the parity tests check more rows of it).

Tolerance: bf16 output, 2e-2 max-abs and 1e-2 rel-L2 per row against the
unrounded fp64 oracle (the rule of the parity tests).
"""

import numpy as np
import pytest
import torch

import synth
from oracle import SequenceOracle
from oracle import csa_oracle as O
from parity_util import _assert_values, _check_topk_row

pytestmark = pytest.mark.gpu

WORKLOAD = 4
HEADS = np.arange(0, 64, 9)
CHUNKS = {"4k": 0, "1M": 7}


@pytest.fixture(scope="module")
def wd():
    from compressed_sparse_long_c128a_gb300 import build as csa_build
    from harness import WorkloadDev

    csa_build.build()
    torch.cuda.empty_cache()
    w = WorkloadDev(synth.workload(WORKLOAD))
    w.step()
    torch.cuda.synchronize()
    w.check("step")
    yield w
    del w
    torch.cuda.empty_cache()


class _Stored:
    """The oracle's stored rows for one sequence, each computed once: the
    entries formed by the ingest, and the window rows of the chunk."""

    def __init__(self, so: SequenceOracle):
        self.so, L, s = so, so.layer, so.seq
        new = so.emitted()
        self.i0 = new[0] if new else 1 << 62
        assert new == list(range(self.i0, self.i0 + len(new))), "emitted entries are consecutive"
        self.new = so.stored_entries(new) if new else np.zeros((0, L.dim))
        self.swa_lo = max(0, s.first_new - L.swa + 1)
        self.swa = so.stored_swa(range(self.swa_lo, s.end))

    def entries(self, ids) -> np.ndarray:
        ids = np.asarray(ids, np.int64)
        out = np.empty((len(ids), self.so.layer.dim))
        h = ids < self.i0
        out[h] = self.so._as_stored(self.so.history[ids[h]], self.so.layer.cache_dtype)
        out[~h] = self.new[ids[~h] - self.i0]
        return out

    def attend(self, r: int, ids) -> np.ndarray:
        """Output of row r over entries `ids` plus its window, for HEADS only."""
        so, L = self.so, self.so.layer
        p = so.seq.first_new + r
        keys = [self.entries(ids)] if len(ids) else []
        w_lo = max(0, p - L.swa + 1)
        keys.append(self.swa[w_lo - self.swa_lo: p + 1 - self.swa_lo])
        q = so.queries[0][r][HEADS]
        return O.attention(q, p, np.concatenate(keys), so.scale, L.rope_dim, L.theta)


def _gpu(ld, b):
    lo, n = ld.row_index(b, 0), ld.wl.seqs[b].n_new
    heads = torch.as_tensor(HEADS, device=ld.io["out"].device)
    out = ld.io["out"][lo:lo + n].index_select(1, heads).to(torch.float64).cpu().numpy()
    topk = ld.io["topk"][lo:lo + n].cpu().numpy() if "topk" in ld.io else None
    return out, topk


def _layer(wd, name):
    return next(ld for ld in wd.layers if ld.L.name == name)


def _sanity(st, r, ids):
    """The memoised rows give what SequenceOracle.attend computes from scratch."""
    ref = st.so.attend(r, entry_ids=ids)["out"][HEADS]
    np.testing.assert_allclose(st.attend(r, ids), ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("chunk", list(CHUNKS))
def test_c128a_every_row_end_to_end(wd, chunk):
    ld = _layer(wd, "c128a")
    b = CHUNKS[chunk]
    so = SequenceOracle(wd.wl, ld.L, b)
    st = _Stored(so)
    out, _ = _gpu(ld, b)
    n_last = so.n_visible(so.seq.end - 1)
    table = st.entries(np.arange(n_last))
    _sanity(st, so.seq.n_new - 1, np.arange(n_last))
    for r in range(so.seq.n_new):
        p = so.seq.first_new + r
        n = so.n_visible(p)
        w_lo = max(0, p - ld.L.swa + 1)
        keys = np.concatenate([table[:n], st.swa[w_lo - st.swa_lo: p + 1 - st.swa_lo]])
        want = O.attention(so.queries[0][r][HEADS], p, keys, so.scale, ld.L.rope_dim, ld.L.theta)
        _assert_values(out[r], want, "bf16", f"c128a {chunk} chunk row {r} (p={p})")


def test_c4a_4k_chunk_every_row_end_to_end(wd):
    ld = _layer(wd, "c4a")
    b = CHUNKS["4k"]
    so = SequenceOracle(wd.wl, ld.L, b)
    st = _Stored(so)
    out, topk = _gpu(ld, b)
    _, q_idx, w = so.queries
    exact = 0
    for r in range(so.seq.n_new):
        p = so.seq.first_new + r
        n = so.n_visible(p)
        what = f"c4a 4k chunk row {r} (p={p})"
        exact += _check_topk_row(topk[r], O.indexer_scores(q_idx[r], w[r], so.index_keys[:n]), ld.L.topk, what)
        sel = topk[r][topk[r] >= 0]
        if r in (0, so.seq.n_new - 1):
            _sanity(st, r, sel)
        _assert_values(out[r], st.attend(r, sel), "bf16", what)
    assert exact >= so.seq.n_new - max(1, so.seq.n_new // 20), f"{exact} exact selections"


def test_c4a_1m_chunk_every_row_stage_isolated(wd):
    ld = _layer(wd, "c4a")
    b = CHUNKS["1M"]
    so = SequenceOracle(wd.wl, ld.L, b)
    st = _Stored(so)
    out, topk = _gpu(ld, b)
    k = ld.L.topk
    for r in range(so.seq.n_new):
        p = so.seq.first_new + r
        n = so.n_visible(p)
        what = f"c4a 1M chunk row {r} (p={p})"
        sel = topk[r][topk[r] >= 0]
        assert len(sel) == min(k, n) and len(np.unique(sel)) == len(sel), f"{what}: size / duplicates"
        assert sel.min() >= 0 and sel.max() < n, f"{what}: index range"
        if r in (0, so.seq.n_new - 1):
            _sanity(st, r, sel)
        _assert_values(out[r], st.attend(r, sel), "bf16", what)
    for r in (0, 683, 1366, so.seq.n_new - 1):
        _check_topk_row(topk[r], so.scores(r), k, f"c4a 1M chunk row {r} selection")
