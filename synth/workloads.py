"""Workload shapes and their seeded draws.

Five workloads, each named by what it is:

  tiny_c4a_f32            one c4a layer in fp32: D=128, H=8, indexer 4 heads x 32,
                          top-64; one sequence whose raw tokens 0..1024 all go
                          through ingest; the step ingests positions 1009..1024
                          and answers one query at each of them.
  c128a_decode_b32_128k   c128a dense decode in bf16: 32 sequences at context
                          131072, D=512 (64 rotary dims), H=64.
  c4a_decode_b64_64k      c4a sparse decode in bf16: 64 sequences, contexts
                          uniform in [32768, 65536], D=512, H=64, indexer 64 x 128,
                          top-512.
  c4a_decode_b4_1m_fp8    c4a sparse decode at context 2^20, 4 sequences; e4m3
                          attention cache (fp32 scale per row), e2m1 indexer cache
                          (e4m3 scale per 16 elements), e4m3 output (fp32 scale per
                          token and head).
  mixed_prefill_decode    8 prefill chunks of 2048 tokens over contexts
                          4k..1M with unaligned starts, plus 24 decode rows at
                          context 65536, for a c4a and a c128a layer, bf16.
  c4a_decode_b64_64k_pfp8 the c4a sparse decode above with the "partial
                          token-wise fp8" attention cache: per row, e4m3 codes
                          with one fp32 scale for the non-rotary dims and the 64
                          rotary dims in bf16 (cache dtype "e4m3r").

How a sequence's history is given.  A step sees a sequence whose first
`first_new` positions are already cached.  Drawing every raw token of a
1M-token history is out of reach for a CPU oracle, so the history is split:

  * every compressed entry whose window starts before `first_new` gets a
    direct N(0,1) draw per element (the distribution of an RMS-normalised,
    rotated vector with unit gain).  The harness stores all of them into the
    paged cache; entries that the library's own ingest later emits overwrite
    theirs.  Entries whose window ends before `ingest_from` keep the draw.
  * raw (kv, gate) rows are drawn for positions [raw_from, first_new + n_new)
    with raw_from = max(0, ingest_from - window of the layer's compressor).
    Rows before `ingest_from` only fill the compressor's state rows; rows from
    `ingest_from` to `first_new` are ingested through the library during
    set-up; the `n_new` rows from `first_new` on are the timed step's tokens.
  * ingest_from = max(0, first_new - 128): set-up ingest writes every
    sliding-window row that a query of the step can see.

The tiny workload has ingest_from = 0 and draws no history entries.

Nothing here computes any part of the method: draws, rounding to the storage
type, shapes and block-table bookkeeping only.
"""

from __future__ import annotations

from dataclasses import dataclass
from functools import lru_cache

import numpy as np

BLOCK_POSITIONS = 256  # one logical cache block covers 256 native positions
SWA = 128  # raw sliding-window length
CACHE_KINDS = ("comp", "idx", "swa", "state")

# seeding keys: (workload seed, tensor id, layer id, sequence, ...)
_T_BIAS, _T_GAMMA_C, _T_GAMMA_SWA, _T_KV, _T_GATE, _T_HIST, _T_KIDX = 1, 2, 3, 4, 5, 6, 7
_T_Q, _T_QIDX, _T_W, _T_LENGTHS, _T_TABLE, _T_SUBSET, _T_OFFSETS = 8, 9, 10, 11, 12, 13, 14
_T_IK_KV, _T_IK_GATE, _T_IK_BIAS, _T_IK_GAMMA, _T_IK_TABLE = 15, 16, 17, 18, 19
_T_GAMMA_Q = 20


def _rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def round_bf16(x) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns fp32 holding bf16 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def _stored(x: np.ndarray, dtype: str) -> np.ndarray:
    """A draw as the caller hands it over: bf16 inputs are bf16 values, all others
    fp32 (quantised caches receive fp32 rows and quantise them on insert)."""
    if dtype == "bf16":
        return round_bf16(x)
    return np.ascontiguousarray(x, dtype=np.float32)


@dataclass(frozen=True)
class LayerSpec:
    name: str
    ratio: int  # compression stride (4 or 128)
    window: int  # raw tokens per compressed entry (8 or 128)
    dim: int  # latent dim D
    heads: int  # query heads H
    in_dtype: str = "bf16"  # raw kv / gate and query
    cache_dtype: str = "bf16"  # compressed and sliding-window caches
    out_dtype: str = "bf16"
    topk: int = 0  # 0: attend to every visible entry (no indexer)
    idx_heads: int = 0
    idx_dim: int = 0
    idx_dtype: str = "bf16"
    rope_dim: int = 64
    theta: float = 10000.0
    eps: float = 1e-6
    swa: int = SWA
    tid: int = 0  # seeding id of the layer

    @property
    def entries_per_block(self) -> int:
        return BLOCK_POSITIONS // self.ratio

    @property
    def has_indexer(self) -> bool:
        return self.topk > 0


@dataclass(frozen=True)
class SeqSpec:
    first_new: int  # position of the step's first token
    n_new: int  # tokens the step ingests; each is also a query row
    ingest_from: int  # set-up ingests [ingest_from, first_new) through the library

    @property
    def end(self) -> int:
        return self.first_new + self.n_new

    def raw_from(self, layer: LayerSpec) -> int:
        return max(0, self.ingest_from - layer.window)


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    layers: tuple
    seqs: tuple
    title: str = ""

    @property
    def n_rows(self) -> int:
        return sum(s.n_new for s in self.seqs)


def _tiny() -> Workload:
    c4 = LayerSpec("c4a", 4, 8, dim=128, heads=8, in_dtype="f32", cache_dtype="f32",
                   out_dtype="f32", topk=64, idx_heads=4, idx_dim=32, idx_dtype="f32")
    return Workload("tiny_c4a_f32", 0, (c4,), (SeqSpec(1009, 16, 0),),
                    "c4a fp32, D=128, H=8, one sequence, queries at 1009..1024")


def _c128a_decode() -> Workload:
    c128 = LayerSpec("c128a", 128, 128, dim=512, heads=64)
    p = 131072
    return Workload("c128a_decode_b32_128k", 1, (c128,),
                    tuple(SeqSpec(p, 1, p - SWA) for _ in range(32)),
                    "c128a dense decode, bf16, B=32, context 131072, D=512, H=64")


def _c4a_decode() -> Workload:
    c4 = LayerSpec("c4a", 4, 8, dim=512, heads=64, topk=512, idx_heads=64, idx_dim=128)
    lens = _rng(2, _T_LENGTHS).integers(32768, 65536, size=64, endpoint=True)
    return Workload("c4a_decode_b64_64k", 2, (c4,),
                    tuple(SeqSpec(int(n), 1, int(n) - SWA) for n in lens),
                    "c4a sparse decode, bf16, B=64, context U[32768,65536], top-512")


def _c4a_decode_1m_fp8() -> Workload:
    c4 = LayerSpec("c4a", 4, 8, dim=512, heads=64, cache_dtype="e4m3", out_dtype="e4m3",
                   topk=512, idx_heads=64, idx_dim=128, idx_dtype="e2m1")
    p = 1 << 20
    return Workload("c4a_decode_b4_1m_fp8", 3, (c4,),
                    tuple(SeqSpec(p, 1, p - SWA) for _ in range(4)),
                    "c4a sparse decode at 2^20, B=4, e4m3 cache, e2m1 indexer, e4m3 out")


def _mixed_prefill_decode() -> Workload:
    c4 = LayerSpec("c4a", 4, 8, dim=512, heads=64, topk=512, idx_heads=64, idx_dim=128, tid=0)
    c128 = LayerSpec("c128a", 128, 128, dim=512, heads=64, tid=1)
    contexts = [4096, 16384, 65536, 131072, 262144, 262144, 524288, 1048576]
    cand = _rng(4, _T_OFFSETS).integers(1, 127, size=256, endpoint=True)
    offsets = [int(c) for c in cand if c % 4 != 0][: len(contexts)]
    seqs = [SeqSpec(c - r, 2048, c - r - SWA) for c, r in zip(contexts, offsets)]
    seqs += [SeqSpec(65536, 1, 65536 - SWA) for _ in range(24)]
    return Workload("mixed_prefill_decode", 4, (c4, c128), tuple(seqs),
                    "8 prefill chunks of 2048 (contexts 4k..1M) + 24 decode rows at 64k")


def _c4a_decode_partial_fp8() -> Workload:
    c4 = LayerSpec("c4a", 4, 8, dim=512, heads=64, cache_dtype="e4m3r", topk=512, idx_heads=64, idx_dim=128)
    lens = _rng(5, _T_LENGTHS).integers(32768, 65536, size=64, endpoint=True)
    return Workload("c4a_decode_b64_64k_pfp8", 5, (c4,),
                    tuple(SeqSpec(int(n), 1, int(n) - SWA) for n in lens),
                    "c4a sparse decode, partial token-wise fp8 cache (e4m3 + bf16 rotary dims), B=64")


_BUILDERS = {0: _tiny, 1: _c128a_decode, 2: _c4a_decode, 3: _c4a_decode_1m_fp8, 4: _mixed_prefill_decode,
             5: _c4a_decode_partial_fp8}
WORKLOADS = {0: "tiny_c4a_f32", 1: "c128a_decode_b32_128k", 2: "c4a_decode_b64_64k",
             3: "c4a_decode_b4_1m_fp8", 4: "mixed_prefill_decode", 5: "c4a_decode_b64_64k_pfp8"}


@lru_cache(maxsize=None)
def workload(key) -> Workload:
    """Workload by index (0..4) or by name."""
    if isinstance(key, str):
        key = {v: k for k, v in WORKLOADS.items()}[key]
    return _BUILDERS[int(key)]()


# ---------------------------------------------------------------- draws


@lru_cache(maxsize=16)
def layer_params(wl: Workload, layer: LayerSpec) -> dict:
    """Per-layer learned parameters: offset bias [window, D] ~N(0, 0.1^2), gains ~1+N(0, 0.02^2)."""
    D = layer.dim
    bias = _rng(wl.seed, _T_BIAS, layer.tid).normal(0.0, 0.1, size=(layer.window, D)).astype(np.float32)
    gamma_c = (1.0 + _rng(wl.seed, _T_GAMMA_C, layer.tid).normal(0.0, 0.02, size=D)).astype(np.float32)
    gamma_swa = (1.0 + _rng(wl.seed, _T_GAMMA_SWA, layer.tid).normal(0.0, 0.02, size=D)).astype(np.float32)
    gamma_q = (1.0 + _rng(wl.seed, _T_GAMMA_Q, layer.tid).normal(0.0, 0.02, size=D)).astype(np.float32)
    return {"bias": bias, "gamma_c": gamma_c, "gamma_swa": gamma_swa, "gamma_q": gamma_q}


def seq_raw(wl: Workload, layer: LayerSpec, b: int):
    """Raw rows of sequence b: (first position, kv [n, D], gate [n, D]), each ~N(0,1)."""
    s = wl.seqs[b]
    lo, hi = s.raw_from(layer), s.end
    shape = (hi - lo, layer.dim)
    kv = _stored(_rng(wl.seed, _T_KV, layer.tid, b).standard_normal(shape, dtype=np.float32), layer.in_dtype)
    gate = _stored(_rng(wl.seed, _T_GATE, layer.tid, b).standard_normal(shape, dtype=np.float32), layer.in_dtype)
    return lo, kv, gate


def seq_history(wl: Workload, layer: LayerSpec, b: int) -> np.ndarray:
    """Directly drawn compressed entries [n, D] ~N(0,1) for every entry whose window starts before first_new."""
    s = wl.seqs[b]
    n = 0 if s.ingest_from == 0 else -(-s.first_new // layer.ratio)
    x = _rng(wl.seed, _T_HIST, layer.tid, b).standard_normal((n, layer.dim), dtype=np.float32)
    return _stored(x, layer.cache_dtype)


def seq_index_keys(wl: Workload, layer: LayerSpec, b: int):
    """Indexer keys [n, d_I] ~N(0,1), one per entry whose window starts before the step's end."""
    if not layer.has_indexer:
        return None
    s = wl.seqs[b]
    n = -(-s.end // layer.ratio)
    x = _rng(wl.seed, _T_KIDX, layer.tid, b).standard_normal((n, layer.idx_dim), dtype=np.float32)
    return _stored(x, layer.idx_dtype)


def seq_queries(wl: Workload, layer: LayerSpec, b: int):
    """Per query row of sequence b: q [n, H, D] ~N(0,1); indexer q_idx [n, H_I, d_I] ~N(0,1), w [n, H_I] ~U(0,1)."""
    s = wl.seqs[b]
    q = _stored(_rng(wl.seed, _T_Q, layer.tid, b).standard_normal((s.n_new, layer.heads, layer.dim),
                                                                    dtype=np.float32), layer.in_dtype)
    if not layer.has_indexer:
        return q, None, None
    q_idx = _stored(_rng(wl.seed, _T_QIDX, layer.tid, b).standard_normal(
        (s.n_new, layer.idx_heads, layer.idx_dim), dtype=np.float32), layer.in_dtype)
    w = _rng(wl.seed, _T_W, layer.tid, b).random((s.n_new, layer.idx_heads), dtype=np.float32)
    return q, q_idx, w


def random_subset(wl: Workload, layer: LayerSpec, b: int, row: int, n: int, m: int) -> np.ndarray:
    """m distinct indices drawn uniformly from range(n), in random order (int32)."""
    m = min(m, n)
    return _rng(wl.seed, _T_SUBSET, layer.tid, b, row).choice(n, size=m, replace=False).astype(np.int32)


# ---------------------------------------------------------------- paging


def _logical_blocks(wl: Workload, layer: LayerSpec, kind: str, b: int):
    s = wl.seqs[b]
    hi = -(-s.end // BLOCK_POSITIONS)
    lo = 0 if kind in ("comp", "idx") else s.raw_from(layer) // BLOCK_POSITIONS
    return lo, hi


@lru_cache(maxsize=64)
def block_table(wl: Workload, layer: LayerSpec, kind: str):
    """Logical -> physical block map for one cache kind of one layer.

    Returns (table [n_seq, max_blocks] int32 with -1 where nothing is mapped,
    number of physical blocks).  Physical ids are one seeded permutation of
    range(n_physical), handed out in (sequence, logical block) order.  The
    compressed and indexer caches map every block of the context; the
    sliding-window and state caches map only the blocks from raw_from on.
    """
    spans = [_logical_blocks(wl, layer, kind, b) for b in range(len(wl.seqs))]
    max_blocks = max(hi for _, hi in spans)
    total = sum(hi - lo for lo, hi in spans)
    perm = _rng(wl.seed, _T_TABLE, layer.tid, CACHE_KINDS.index(kind)).permutation(total).astype(np.int32)
    table = np.full((len(wl.seqs), max_blocks), -1, dtype=np.int32)
    k = 0
    for b, (lo, hi) in enumerate(spans):
        table[b, lo:hi] = perm[k:k + hi - lo]
        k += hi - lo
    table.setflags(write=False)
    return table, total


def physical_row(table: np.ndarray, b: int, logical_row, rows_per_block: int):
    """(physical block, row within block) of logical row(s) of sequence b."""
    logical_row = np.asarray(logical_row)
    blk = table[b, logical_row // rows_per_block]
    if np.any(blk < 0):
        raise IndexError("logical row maps to an unmapped block")
    return blk, logical_row % rows_per_block


# ---------------------------------------------------------------- indexer-key compressor


def index_key_case(seed: int, lengths, dim: int = 128, window: int = 8, in_dtype: str = "bf16") -> dict:
    """Inputs of the indexer-key compressor for sequences of the given lengths.

    Sequence b holds raw tokens at positions 0 .. lengths[b]-1: kv and gate
    [lengths[b], dim] ~N(0,1) in `in_dtype`.  Learned parameters: offset bias
    [window, dim] ~N(0, 0.1^2), gain [dim] ~1+N(0, 0.02^2).  Block tables map
    the ceil(length/256) logical blocks of each sequence through one seeded
    permutation per cache kind ("state": the compressor state, "idx": the
    indexer cache), as the workloads' tables do.
    """
    kv = [_stored(_rng(seed, _T_IK_KV, b).standard_normal((n, dim), dtype=np.float32), in_dtype)
          for b, n in enumerate(lengths)]
    gate = [_stored(_rng(seed, _T_IK_GATE, b).standard_normal((n, dim), dtype=np.float32), in_dtype)
            for b, n in enumerate(lengths)]
    bias = _rng(seed, _T_IK_BIAS).normal(0.0, 0.1, size=(window, dim)).astype(np.float32)
    gamma = (1.0 + _rng(seed, _T_IK_GAMMA).normal(0.0, 0.02, size=dim)).astype(np.float32)
    blocks = [-(-n // BLOCK_POSITIONS) for n in lengths]
    tables = {}
    for kind in ("state", "idx"):
        perm = _rng(seed, _T_IK_TABLE, CACHE_KINDS.index(kind)).permutation(sum(blocks)).astype(np.int32)
        t = np.full((len(lengths), max(blocks)), -1, dtype=np.int32)
        k = 0
        for b, nb in enumerate(blocks):
            t[b, :nb] = perm[k:k + nb]
            k += nb
        tables[kind] = t
    return {"kv": kv, "gate": gate, "bias": bias, "gamma": gamma, "tables": tables, "n_blocks": sum(blocks)}
