"""The oracle's steps applied to one sequence of a synthetic workload.

TEST INFRASTRUCTURE (see csa_oracle).  Inputs come only from `synth`; every
expected value is computed here from those inputs by the fp64 steps of
csa_oracle.  What the caches are expected to hold:

  * entries whose window ends before the sequence's `ingest_from` hold their
    directly drawn history vector, as the cache stores it;
  * entries whose window ends in [ingest_from, end) are emitted by ingest:
    gated window sum -> RMSNorm -> RoPE at the anchor;
  * sliding-window rows for positions [ingest_from, end) are RMSNorm -> RoPE of
    the raw kv row at its own position.

A cache stored as e4m3 (or e4m3r: e4m3 non-rotary dims, bf16 rotary dims)
holds the codec's dequantised value of the fp32 form of the above; bf16 and fp32 caches are compared against the unrounded fp64
value, so the oracle never models the kernels' rounding.
"""

from __future__ import annotations

import math
from functools import cached_property

import numpy as np

import synth

from . import csa_oracle as O


class SequenceOracle:
    def __init__(self, wl: synth.Workload, layer: synth.LayerSpec, b: int):
        self.wl, self.layer, self.b = wl, layer, b
        self.seq = wl.seqs[b]
        prm = synth.layer_params(wl, layer)
        self.bias, self.gamma_c, self.gamma_swa = prm["bias"], prm["gamma_c"], prm["gamma_swa"]
        self.raw_lo, self.kv, self.gate = synth.seq_raw(wl, layer, b)
        self.scale = 1.0 / math.sqrt(layer.dim)

    # ------------------------------------------------------------ geometry

    def last_token(self, i: int) -> int:
        return O.window_span(i, self.layer.ratio, self.layer.window)[1]

    def emitted(self, lo: int | None = None, hi: int | None = None) -> list:
        """Entries whose window closes at a token ingested in [lo, hi) (default: set-up + step)."""
        L = self.layer
        lo = self.seq.ingest_from if lo is None else lo
        hi = self.seq.end if hi is None else hi
        out = []
        for t in range(lo, hi):
            i = O.closing_entry(t, L.ratio, L.window)
            if i is not None:
                out.append(i)
        return out

    def n_visible(self, p: int) -> int:
        return O.n_visible(p, self.layer.ratio, self.layer.window)

    # ------------------------------------------------------------ cache contents

    @cached_property
    def history(self) -> np.ndarray:
        return synth.seq_history(self.wl, self.layer, self.b)

    def computed_entry(self, i: int) -> np.ndarray:
        L = self.layer
        return O.compressed_entry(self.kv, self.gate, self.raw_lo, i, L.ratio, L.window, self.bias,
                                  self.gamma_c, L.eps, L.rope_dim, L.theta)

    def _as_stored(self, rows: np.ndarray, dtype: str) -> np.ndarray:
        if dtype == "e4m3":
            codes, scale = O.quantize_rows_e4m3(np.asarray(rows, np.float32))
            return O.dequantize_rows_e4m3(codes, scale)
        if dtype == "e4m3r":
            codes, scale, rope = O.quantize_rows_e4m3_rope_bf16(np.asarray(rows, np.float32), self.layer.rope_dim)
            return O.dequantize_rows_e4m3_rope_bf16(codes, scale, rope)
        return np.asarray(rows, np.float64)

    def stored_entries(self, ids) -> np.ndarray:
        """What the compressed cache holds for entries `ids` after the step, fp64 [n, D]."""
        ids = np.asarray(ids, dtype=np.int64)
        out = np.empty((len(ids), self.layer.dim), dtype=np.float64)
        from_hist = np.array([self.last_token(int(i)) < self.seq.ingest_from for i in ids], dtype=bool)
        if from_hist.any():
            out[from_hist] = self._as_stored(self.history[ids[from_hist]], self.layer.cache_dtype)
        rest = np.nonzero(~from_hist)[0]
        if len(rest):
            vals = np.stack([self.computed_entry(int(ids[k])) for k in rest])
            out[rest] = self._as_stored(vals, self.layer.cache_dtype)
        return out

    def swa_value(self, t: int) -> np.ndarray:
        L = self.layer
        return O.swa_row(self.kv[t - self.raw_lo], t, self.gamma_swa, L.eps, L.rope_dim, L.theta)

    def stored_swa(self, positions) -> np.ndarray:
        vals = np.stack([self.swa_value(int(t)) for t in positions])
        return self._as_stored(vals, self.layer.cache_dtype)

    @cached_property
    def index_keys(self) -> np.ndarray:
        """Indexer keys as the indexer cache holds them, fp64 [n, d_I]."""
        k = synth.seq_index_keys(self.wl, self.layer, self.b)
        if self.layer.idx_dtype == "e2m1":
            packed, sc = O.quantize_nvfp4(k)
            return O.dequantize_nvfp4(packed, sc)
        return np.asarray(k, np.float64)

    @cached_property
    def queries(self):
        return synth.seq_queries(self.wl, self.layer, self.b)

    # ------------------------------------------------------------ per query row

    def scores(self, r: int) -> np.ndarray:
        p = self.seq.first_new + r
        n = self.n_visible(p)
        _, q_idx, w = self.queries
        return O.indexer_scores(q_idx[r], w[r], self.index_keys[:n])

    def topk(self, r: int) -> np.ndarray:
        return O.topk_select(self.scores(r), self.layer.topk)

    def attend(self, r: int, entry_ids=None) -> dict:
        """Output of query row r over `entry_ids` (default: the layer's own selection)."""
        L = self.layer
        p = self.seq.first_new + r
        if entry_ids is None:
            entry_ids = self.topk(r) if L.has_indexer else np.arange(self.n_visible(p))
        entry_ids = np.asarray(entry_ids, dtype=np.int64)
        keys = [self.stored_entries(entry_ids)] if len(entry_ids) else []
        keys.append(self.stored_swa(O.swa_positions(p, L.swa)))
        q = self.queries[0][r]
        out = O.attention(q, p, np.concatenate(keys), self.scale, L.rope_dim, L.theta)
        res = {"p": p, "entries": entry_ids, "out": out}
        if L.out_dtype == "e4m3":
            codes, sc = O.quantize_rows_e4m3(out.astype(np.float32))
            res["out_codes"], res["out_scale"] = codes, sc
        return res
