"""Device-side set-up of a synthetic workload, driven through libcsa.

For every layer of a workload this allocates the paged caches that the
generator's block tables describe, then:
  1. stores each sequence's directly drawn history entries, and its indexer
     keys, through csa_cache_store (quantising to the cache dtype);
  2. copies the raw (kv | gate) rows that precede the set-up ingest into the
     compressor state cache (a caller restoring its rolling residual);
  3. ingests positions [ingest_from, first_new) through csa_compress_insert;
  4. stages the step's inputs: the new tokens (which are also the query rows),
     queries, indexer queries and weights.
`WorkloadDev.step()` is then one pass of the hot path: per layer,
compress_insert of the new tokens, indexer_topk (c4a layers) and sparse
attention.  Re-running it is idempotent.

This is test / benchmark plumbing: it calls only the library's C ABI for the
method's arithmetic, and never imports the oracle.
"""

from __future__ import annotations

import numpy as np
import torch

import compressed_sparse_long_c128a_gb300 as csa
import synth

_TORCH_IN = {"f32": torch.float32, "bf16": torch.bfloat16}


def n_visible(p: int, ratio: int, window: int) -> int:
    """Entries a query at p may read (their last raw token is before p)."""
    return 0 if p < window else (p - window) // ratio + 1


def _dev(x, dtype=None, device="cuda"):
    x = np.ascontiguousarray(x)
    t = torch.from_numpy(x if x.flags.writeable else x.copy())
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device, non_blocking=False)


class LayerDev:
    """Caches, block tables, parameters and step buffers of one layer."""

    def __init__(self, wl: synth.Workload, L: synth.LayerSpec, device="cuda"):
        self.wl, self.L, self.device = wl, L, device
        self.c_layer = csa.make_layer(L.ratio, L.window, L.dim, L.rope_dim, L.heads, L.swa, L.theta, L.eps)
        self.tables, self.n_blocks = {}, {}
        for kind in synth.CACHE_KINDS:
            if kind == "idx" and not L.has_indexer:
                continue
            t, n = synth.block_table(wl, L, kind)
            self.tables[kind] = _dev(t, device=device)
            self.n_blocks[kind] = n
        cd = csa.DTYPES[L.cache_dtype]
        tail = L.rope_dim if L.cache_dtype == "e4m3r" else 0  # rotary dims kept in bf16
        self.comp = csa.PagedCache.empty(self.n_blocks["comp"], L.entries_per_block, L.dim, cd, device, tail)
        self.swa = csa.PagedCache.empty(self.n_blocks["swa"], synth.BLOCK_POSITIONS, L.dim, cd, device, tail)
        self.state = csa.PagedCache.empty(self.n_blocks["state"], synth.BLOCK_POSITIONS, 2 * L.dim,
                                          csa.DTYPES[L.in_dtype], device)
        self.idx = None
        if L.has_indexer:
            self.idx = csa.PagedCache.empty(self.n_blocks["idx"], L.entries_per_block, L.idx_dim,
                                            csa.DTYPES[L.idx_dtype], device)
        prm = synth.layer_params(wl, L)
        self.bias = _dev(prm["bias"], device=device)
        self.gamma_c = _dev(prm["gamma_c"], device=device)
        self.gamma_swa = _dev(prm["gamma_swa"], device=device)
        self.gamma_q = _dev(prm["gamma_q"], device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    # ------------------------------------------------------------------ set-up

    def load_history(self):
        wl, L = self.wl, self.L
        for b, s in enumerate(wl.seqs):
            hist = synth.seq_history(wl, L, b)
            if len(hist):
                self._store(hist, b, self.comp, self.tables["comp"])
            if L.has_indexer:
                self._store(synth.seq_index_keys(wl, L, b), b, self.idx, self.tables["idx"])
            lo, kv, gate = synth.seq_raw(wl, L, b)
            n_pre = s.ingest_from - lo
            if n_pre > 0:
                blk, row = synth.physical_row(synth.block_table(wl, L, "state")[0], b,
                                              np.arange(lo, s.ingest_from), synth.BLOCK_POSITIONS)
                rows = np.concatenate([kv[:n_pre], gate[:n_pre]], axis=1)
                dst = _dev(rows, _TORCH_IN[L.in_dtype], self.device)
                self.state.data[_dev(blk.astype(np.int64), device=self.device),
                                _dev(row.astype(np.int64), device=self.device)] = dst
        self.check("history load")

    def _store(self, rows: np.ndarray, b: int, cache, table, chunk: int = 1 << 16):
        for c0 in range(0, len(rows), chunk):
            part = rows[c0:c0 + chunk]
            n = len(part)
            seq = torch.full((n,), b, dtype=torch.int32, device=self.device)
            idx = torch.arange(c0, c0 + n, dtype=torch.int32, device=self.device)
            csa.cache_store(_dev(part, torch.float32, self.device), seq, idx, cache, table, self.err)

    def ingest(self, seq_ids: np.ndarray, positions: np.ndarray, kv: np.ndarray, gate: np.ndarray):
        """compress_insert of raw tokens given on the host."""
        dt = _TORCH_IN[self.L.in_dtype]
        self.compress_insert(_dev(kv, dt, self.device), _dev(gate, dt, self.device),
                             _dev(seq_ids.astype(np.int32), device=self.device),
                             _dev(positions.astype(np.int32), device=self.device))

    def compress_insert(self, kv, gate, seq_id, pos, stream=None):
        csa.compress_insert(self.c_layer, kv, gate, seq_id, pos, self.bias, self.gamma_c, self.gamma_swa,
                            self.state, self.tables["state"], self.swa, self.tables["swa"], self.comp,
                            self.tables["comp"], self.err, stream)

    def compress_insert_qnorm(self, kv, gate, seq_id, pos, q, q_out, stream=None):
        """compress_insert with the query RMSNorm (gamma_q) of the same tokens in its launch."""
        csa.compress_insert_qnorm(self.c_layer, kv, gate, seq_id, pos, self.bias, self.gamma_c, self.gamma_swa,
                                  self.state, self.tables["state"], self.swa, self.tables["swa"], self.comp,
                                  self.tables["comp"], q, self.gamma_q, q_out, self.err, stream)

    def setup_ingest(self):
        """Ingest [ingest_from, first_new) of every sequence in one call."""
        seqs, poss, kvs, gates = [], [], [], []
        for b, s in enumerate(self.wl.seqs):
            lo, kv, gate = synth.seq_raw(self.wl, self.L, b)
            a, e = s.ingest_from - lo, s.first_new - lo
            if e > a:
                seqs.append(np.full(e - a, b))
                poss.append(np.arange(s.ingest_from, s.first_new))
                kvs.append(kv[a:e])
                gates.append(gate[a:e])
        if seqs:
            self.ingest(np.concatenate(seqs), np.concatenate(poss), np.concatenate(kvs), np.concatenate(gates))
        self.check("set-up ingest")

    # ------------------------------------------------------------------ step inputs

    def stage_step(self):
        """Host copies of the step's inputs (tokens = query rows), in sequence order."""
        wl, L = self.wl, self.L
        seqs, poss, kvs, gates, qs, qis, ws = [], [], [], [], [], [], []
        for b, s in enumerate(wl.seqs):
            lo, kv, gate = synth.seq_raw(wl, L, b)
            a = s.first_new - lo
            seqs.append(np.full(s.n_new, b))
            poss.append(np.arange(s.first_new, s.end))
            kvs.append(kv[a:a + s.n_new])
            gates.append(gate[a:a + s.n_new])
            q, qi, w = synth.seq_queries(wl, L, b)
            qs.append(q)
            if L.has_indexer:
                qis.append(qi)
                ws.append(w)
        host = {"seq_id": np.concatenate(seqs).astype(np.int32), "pos": np.concatenate(poss).astype(np.int32),
                "kv": np.concatenate(kvs), "gate": np.concatenate(gates), "q": np.concatenate(qs)}
        if L.has_indexer:
            host["q_idx"] = np.concatenate(qis)
            host["w"] = np.concatenate(ws)
        self.host = host
        self.n_rows = len(host["pos"])
        self.max_n = max(n_visible(int(p), L.ratio, L.window) for p in host["pos"])
        self.prefill = any(s.n_new > 1 for s in wl.seqs)
        # device buffers
        dt = _TORCH_IN[L.in_dtype]
        d = self.device
        self.io = {"seq_id": _dev(host["seq_id"], device=d), "pos": _dev(host["pos"], device=d),
                   "kv": _dev(host["kv"], dt, d), "gate": _dev(host["gate"], dt, d), "q": _dev(host["q"], dt, d)}
        if L.has_indexer:
            self.io["q_idx"] = _dev(host["q_idx"], dt, d)
            self.io["w"] = _dev(host["w"], torch.float32, d)
            self.io["topk"] = torch.full((self.n_rows, L.topk), -1, dtype=torch.int32, device=d)
            n = csa.indexer_topk_workspace_size(self.n_rows, max(self.max_n, 1), L.topk)
            self.ws_idx = torch.empty(max(n, 1), dtype=torch.uint8, device=d)
        if L.out_dtype == "e4m3":
            self.io["out"] = torch.zeros((self.n_rows, L.heads, L.dim), dtype=torch.uint8, device=d)
            self.io["out_scales"] = torch.zeros((self.n_rows, L.heads), dtype=torch.float32, device=d)
        else:
            self.io["out"] = torch.zeros((self.n_rows, L.heads, L.dim), dtype=_TORCH_IN[L.out_dtype], device=d)
            self.io["out_scales"] = None
        kq = L.topk if L.has_indexer else self.max_n
        n = csa.sparse_attn_workspace_size(self.c_layer, self.n_rows, kq)
        self.ws_attn = torch.empty(max(n, 1), dtype=torch.uint8, device=d)

    def input_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for k, t in self.io.items()
                   if k in ("seq_id", "pos", "kv", "gate", "q", "q_idx", "w"))

    def output_bytes(self) -> int:
        o = self.io["out"]
        n = o.numel() * o.element_size()
        if self.io["out_scales"] is not None:
            n += self.io["out_scales"].numel() * 4
        return n

    # ------------------------------------------------------------------ the hot path

    def step(self, stream=None, topk_override=None, side_stream=None):
        """compress_insert -> (indexer_topk) -> sparse attention.

        With `side_stream`, a c4a layer's compress_insert runs on it in
        parallel with the indexer pipeline on `stream`, and is joined before
        the attention (the indexer reads only the indexer cache and the step's
        indexer queries, nothing compress_insert writes).  The indexer stays
        on `stream`, right behind the previous attention, so that it takes
        every SM as soon as that ends; compress_insert, which waits for the
        previous attention as a whole, fills the SMs the indexer's shorter
        ranges leave."""
        L, io = self.L, self.io
        main = torch.cuda.current_stream() if stream is None else stream
        use_side = side_stream is not None and L.has_indexer and topk_override is None
        if use_side:
            fork = torch.cuda.Event()
            fork.record(main)
            side_stream.wait_event(fork)
            self.compress_insert(io["kv"], io["gate"], io["seq_id"], io["pos"], side_stream)
        else:
            self.compress_insert(io["kv"], io["gate"], io["seq_id"], io["pos"], main)
        topk, k = None, 0
        if L.has_indexer:
            k = L.topk
            if topk_override is not None:
                topk = topk_override
            else:
                csa.indexer_topk(io["q_idx"], io["w"], io["seq_id"], io["pos"], L.ratio, L.window, self.idx,
                                 self.tables["idx"], k, max(self.max_n, 1), io["topk"], self.ws_idx, self.err, main)
                topk = io["topk"]
        if use_side:
            join = torch.cuda.Event()
            join.record(side_stream)
            main.wait_event(join)
        attn = csa.sparse_attn_prefill if self.prefill else csa.sparse_attn_decode
        attn(self.c_layer, io["q"], io["seq_id"], io["pos"], self.comp, self.tables["comp"], topk, k,
             max(self.max_n, 1), self.swa, self.tables["swa"], io["out"], csa.DTYPES[L.out_dtype],
             io["out_scales"], self.ws_attn, self.err, main)

    def check(self, what: str):
        st = csa.read_status(self.err, reset=True)
        if st != 0:
            raise csa.CsaError(st, f"device status after {what}")

    # ------------------------------------------------------------------ read-back (tests)

    def _rows(self, cache, table_kind, b, logical):
        logical = np.asarray(logical, dtype=np.int64)
        blk, row = synth.physical_row(synth.block_table(self.wl, self.L, table_kind)[0], b, logical,
                                      cache.rows_per_block)
        bi = torch.from_numpy(blk.astype(np.int64)).to(self.device)
        ri = torch.from_numpy(row.astype(np.int64)).to(self.device)
        return bi, ri

    def read_cache(self, kind: str, b: int, logical) -> np.ndarray:
        """Values of logical rows of sequence b, dequantised to float64 (E2M1 excluded)."""
        cache = {"comp": self.comp, "swa": self.swa, "state": self.state, "idx": self.idx}[kind]
        bi, ri = self._rows(cache, kind, b, logical)
        d = cache.data[bi, ri]
        if cache.dtype == csa.E4M3:
            v = d.view(torch.float8_e4m3fn).to(torch.float64) * cache.scales[bi, ri].to(torch.float64)[:, None]
        elif cache.dtype == csa.E4M3R:
            dq = cache.dim - cache.tail_bf16
            head = d[:, :dq].view(torch.float8_e4m3fn).to(torch.float64) * cache.scales[bi, ri].to(torch.float64)[:, None]
            tail = d[:, dq:].contiguous().view(torch.bfloat16).to(torch.float64)
            v = torch.cat([head, tail], dim=1)
        elif cache.dtype == csa.E2M1:
            raise ValueError("use read_cache_bytes for e2m1")
        else:
            v = d.to(torch.float64)
        return v.cpu().numpy()

    def read_cache_bytes(self, kind: str, b: int, logical):
        cache = {"comp": self.comp, "swa": self.swa, "idx": self.idx}[kind]
        bi, ri = self._rows(cache, kind, b, logical)
        sc = cache.scales[bi, ri].cpu().numpy() if cache.scales is not None else None
        return cache.data[bi, ri].cpu().numpy(), sc

    def output(self):
        """(out float64 [rows, H, D] dequantised, codes or None, scales or None)."""
        o = self.io["out"]
        if self.L.out_dtype == "e4m3":
            sc = self.io["out_scales"]
            v = o.view(torch.float8_e4m3fn).to(torch.float64) * sc.to(torch.float64)[..., None]
            return v.cpu().numpy(), o.cpu().numpy(), sc.cpu().numpy()
        return o.to(torch.float64).cpu().numpy(), None, None

    def row_index(self, b: int, r: int) -> int:
        """Row number of query r of sequence b in the step's row order."""
        return sum(s.n_new for s in self.wl.seqs[:b]) + r


class WorkloadDev:
    """All layers of a workload, set up and ready to step."""

    def __init__(self, wl: synth.Workload, device="cuda"):
        self.wl = wl
        self.layers = [LayerDev(wl, L, device) for L in wl.layers]
        for ld in self.layers:
            ld.load_history()
            ld.setup_ingest()
            ld.stage_step()
        torch.cuda.synchronize()

    def step(self, stream=None, side_stream=None):
        for ld in self.layers:
            ld.step(stream, side_stream=side_stream)

    def check(self, what="step"):
        for ld in self.layers:
            ld.check(what)
