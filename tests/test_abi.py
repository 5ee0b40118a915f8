"""The C-ABI library builds, loads and exports every symbol its header declares;
host-side validation answers without touching a GPU (CPU only)."""

import ctypes
import os
import re
import subprocess

import pytest

import compressed_sparse_long_c128a_gb300 as csa
from compressed_sparse_long_c128a_gb300 import build as csa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")


@pytest.fixture(scope="module")
def lib():
    csa_build.build()
    return csa.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = _declared()
    for n in ("csa_compress_insert", "csa_indexer_topk", "csa_sparse_attn_decode", "csa_sparse_attn_prefill",
              "csa_cache_store", "csa_read_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", csa_build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (csa_\w+)", out))
    assert set(_declared()) == exported  # nothing undeclared leaks out either
    assert set(csa.EXPORTED) == exported


def test_version_and_status_strings(lib):
    assert csa.version() == 100
    assert csa.status_string(csa.OK) == "ok"
    assert "workspace" in csa.status_string(csa.ERR_WORKSPACE)
    assert csa.status_string(12345) == "unknown status"


def test_library_refuses_to_load_when_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(csa, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(csa, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        csa.lib()


def _paged(dtype=csa.BF16, rows=64, dim=512):
    return csa.Paged(0x1000, 0x2000, dtype, 10, rows, dim)


def _bt():
    return csa.BlockTableC(0x3000, 2, 4)


def test_host_validation_rejects_bad_arguments(lib):
    L = csa.make_layer(4, 8, 512, 64, 64)
    P, B = _paged(), _bt()
    st, sw = _paged(csa.BF16, 256, 1024), _paged(csa.BF16, 256, 512)
    # null kv
    r = lib.csa_compress_insert(ctypes.byref(L), None, 0x10, csa.BF16, 4, 0x10, 0x10, 0x10, 0x10, 0x10,
                                ctypes.byref(st), ctypes.byref(B), ctypes.byref(sw), ctypes.byref(B),
                                ctypes.byref(P), ctypes.byref(B), 0x10, None)
    assert r == csa.ERR_INVALID_ARG
    # state dtype must equal the input dtype
    st32 = _paged(csa.F32, 256, 1024)
    r = lib.csa_compress_insert(ctypes.byref(L), 0x10, 0x10, csa.BF16, 4, 0x10, 0x10, 0x10, 0x10, 0x10,
                                ctypes.byref(st32), ctypes.byref(B), ctypes.byref(sw), ctypes.byref(B),
                                ctypes.byref(P), ctypes.byref(B), 0x10, None)
    assert r == csa.ERR_UNSUPPORTED
    # compressed cache must have 256/ratio rows per block
    bad = _paged(csa.BF16, 32, 512)
    r = lib.csa_compress_insert(ctypes.byref(L), 0x10, 0x10, csa.BF16, 4, 0x10, 0x10, 0x10, 0x10, 0x10,
                                ctypes.byref(st), ctypes.byref(B), ctypes.byref(sw), ctypes.byref(B),
                                ctypes.byref(bad), ctypes.byref(B), 0x10, None)
    assert r == csa.ERR_INVALID_ARG
    # zero tokens is a no-op
    r = lib.csa_compress_insert(ctypes.byref(L), None, None, csa.BF16, 0, None, None, None, None, None,
                                ctypes.byref(st), ctypes.byref(B), ctypes.byref(sw), ctypes.byref(B),
                                ctypes.byref(P), ctypes.byref(B), None, None)
    assert r == csa.OK
    # bad layer: ratio that does not divide 256
    L2 = csa.make_layer(3, 8, 512, 64, 64)
    r = lib.csa_compress_insert(ctypes.byref(L2), 0x10, 0x10, csa.BF16, 4, 0x10, 0x10, 0x10, 0x10, 0x10,
                                ctypes.byref(st), ctypes.byref(B), ctypes.byref(sw), ctypes.byref(B),
                                ctypes.byref(P), ctypes.byref(B), 0x10, None)
    assert r == csa.ERR_INVALID_ARG



def test_indexer_key_compressor_validation(lib):
    """compress_insert without a window cache (the indexer-key compressor) and
    into an e2m1 cache: the host checks that stop a call before any launch."""
    L = csa.make_layer(4, 8, 128, 64, 64)
    st, B = _paged(csa.BF16, 256, 256), _bt()
    sw = _paged(csa.BF16, 256, 128)
    idx = _paged(csa.E2M1, 64, 128)

    def call(layer, swa, swa_bt, gamma_swa, comp):
        return lib.csa_compress_insert(ctypes.byref(layer), 0x10, 0x10, csa.BF16, 4, 0x10, 0x10, 0x10, 0x10,
                                       gamma_swa, ctypes.byref(st), ctypes.byref(B), swa, swa_bt,
                                       ctypes.byref(comp), ctypes.byref(B), 0x10, None)

    # a window cache needs its gains and its block table
    assert call(L, ctypes.byref(sw), ctypes.byref(B), None, idx) == csa.ERR_INVALID_ARG
    assert call(L, ctypes.byref(sw), None, 0x10, idx) == csa.ERR_INVALID_ARG
    # e2m1 entries need the scale array and D % 16 == 0
    no_scales = csa.Paged(0x1000, None, csa.E2M1, 10, 64, 128)
    assert call(L, None, None, None, no_scales) == csa.ERR_INVALID_ARG
    L24 = csa.make_layer(4, 8, 24, 8, 8)
    st24 = _paged(csa.BF16, 256, 48)
    r = lib.csa_compress_insert(ctypes.byref(L24), 0x10, 0x10, csa.BF16, 4, 0x10, 0x10, 0x10, 0x10, None,
                                ctypes.byref(st24), ctypes.byref(B), None, None,
                                ctypes.byref(_paged(csa.E2M1, 64, 24)), ctypes.byref(B), 0x10, None)
    assert r == csa.ERR_INVALID_ARG
    # the window cache stays limited to the dtypes attention reads
    assert call(L, ctypes.byref(_paged(csa.E2M1, 256, 128)), ctypes.byref(B), 0x10, idx) == csa.ERR_UNSUPPORTED
    # no tokens: a no-op with or without a window cache
    r = lib.csa_compress_insert(ctypes.byref(L), None, None, csa.BF16, 0, None, None, None, None, None,
                                ctypes.byref(st), ctypes.byref(B), None, None, ctypes.byref(idx),
                                ctypes.byref(B), None, None)
    assert r == csa.OK

def test_query_norm_validation(lib):
    """csa_compress_insert_qnorm: the checks of the query rows that stop a call
    before any launch (null or out-of-range fields, dtypes, D and alignment)."""
    L = csa.make_layer(4, 8, 512, 64, 64)
    P, B = _paged(), _bt()
    st, sw = _paged(csa.BF16, 256, 1024), _paged(csa.BF16, 256, 512)

    def call(qn, layer=L, state=st, swa=sw, comp=P, n_tok=4):
        return lib.csa_compress_insert_qnorm(ctypes.byref(layer), 0x10, 0x10, csa.BF16, n_tok, 0x10, 0x10,
                                             0x10, 0x10, 0x10, ctypes.byref(state), ctypes.byref(B),
                                             ctypes.byref(swa), ctypes.byref(B), ctypes.byref(comp),
                                             ctypes.byref(B), qn, 0x10, None)

    def qn(q=0x1000, q_dtype=csa.BF16, heads=64, gamma=0x2000, q_out=0x3000, out_dtype=csa.BF16):
        return ctypes.byref(csa.QueryNormC(q, q_dtype, heads, gamma, q_out, out_dtype))

    assert call(None) == csa.ERR_INVALID_ARG                      # qn is required
    assert call(None, n_tok=0) == csa.ERR_INVALID_ARG             # even for no tokens
    assert call(qn(q=None)) == csa.ERR_INVALID_ARG
    assert call(qn(gamma=None)) == csa.ERR_INVALID_ARG
    assert call(qn(q_out=None)) == csa.ERR_INVALID_ARG
    assert call(qn(heads=0)) == csa.ERR_INVALID_ARG
    assert call(qn(heads=1025)) == csa.ERR_INVALID_ARG
    assert call(qn(q_dtype=csa.E4M3)) == csa.ERR_UNSUPPORTED
    assert call(qn(out_dtype=csa.E2M1)) == csa.ERR_UNSUPPORTED
    for field in ("q", "gamma", "q_out"):                          # 16-byte alignment
        assert call(qn(**{field: 0x1008})) == csa.ERR_UNSUPPORTED
    # D above 512, and D not a multiple of 8
    L1k = csa.make_layer(4, 8, 1024, 64, 64)
    r = call(qn(), layer=L1k, state=_paged(csa.BF16, 256, 2048), swa=_paged(csa.BF16, 256, 1024),
             comp=_paged(csa.BF16, 64, 1024))
    assert r == csa.ERR_UNSUPPORTED
    L20 = csa.make_layer(4, 8, 20, 8, 8)
    r = call(qn(), layer=L20, state=_paged(csa.BF16, 256, 40), swa=_paged(csa.BF16, 256, 20),
             comp=_paged(csa.BF16, 64, 20))
    assert r == csa.ERR_UNSUPPORTED
    # no tokens: a no-op once qn is given, whatever it holds
    assert call(qn(heads=0), n_tok=0) == csa.OK


def test_cache_store_validation(lib):
    """csa_cache_store: checks of the count, the pointers, the cache's dtype,
    dims and scales, and the block table, answered before any launch."""
    B = _bt()

    def call(cache, n=4, rows=0x10, bt=B):
        return lib.csa_cache_store(rows, n, 0x10, 0x10, ctypes.byref(cache) if cache else None,
                                   ctypes.byref(bt) if bt else None, 0x10, None)

    assert call(_paged(), n=-1) == csa.ERR_INVALID_ARG
    assert lib.csa_cache_store(None, 0, None, None, None, None, None, None) == csa.OK   # no rows: a no-op
    assert call(_paged(), rows=None) == csa.ERR_INVALID_ARG
    assert call(None) == csa.ERR_INVALID_ARG
    assert call(_paged(), bt=None) == csa.ERR_INVALID_ARG
    assert call(_paged(), bt=csa.BlockTableC(0x3000, 0, 4)) == csa.ERR_INVALID_ARG     # no sequences
    assert call(csa.Paged(0x1000, 0x2000, 7, 10, 64, 512)) == csa.ERR_INVALID_ARG       # no such dtype
    assert call(csa.Paged(0x1000, 0x2000, csa.BF16, 0, 64, 512)) == csa.ERR_INVALID_ARG  # no blocks
    assert call(csa.Paged(0x1000, 0x2000, csa.BF16, 10, 64, 511)) == csa.ERR_INVALID_ARG  # odd dim
    # quantised rows need their scales; e2m1 groups of 16
    assert call(csa.Paged(0x1000, None, csa.E4M3, 10, 64, 512)) == csa.ERR_INVALID_ARG
    assert call(csa.Paged(0x1000, None, csa.E2M1, 10, 64, 128)) == csa.ERR_INVALID_ARG
    assert call(_paged(csa.E2M1, 64, 120)) == csa.ERR_INVALID_ARG
    # the partial fp8 tail: required, a multiple of 16, no larger than the row;
    # every other dtype has none
    for tail in (0, 8, 520):
        assert call(csa.Paged(0x1000, 0x2000, csa.E4M3R, 10, 64, 512, tail)) == csa.ERR_INVALID_ARG
    assert call(csa.Paged(0x1000, 0x2000, csa.BF16, 10, 64, 512, 64)) == csa.ERR_INVALID_ARG


def test_sparse_attention_validation(lib):
    """csa_sparse_attn_prefill (the decode entry shares its checks): layer,
    counts, dtypes of query, output and caches, cache geometry and the shapes
    the kernels take, all answered before any launch."""
    L = csa.make_layer(4, 8, 512, 64, 64)
    B = _bt()
    C, S = _paged(csa.BF16, 64, 512), _paged(csa.BF16, 256, 512)

    def call(layer=L, n_rows=4, q_dtype=csa.BF16, comp=C, swa=S, topk=0x10, k=512, max_n=1000,
             out_dtype=csa.BF16, out_scales=None, q=0x10):
        return lib.csa_sparse_attn_prefill(ctypes.byref(layer), q, q_dtype, n_rows, 0x10, 0x10,
                                           ctypes.byref(comp), ctypes.byref(B), topk, k, max_n,
                                           ctypes.byref(swa), ctypes.byref(B), 0x10, out_dtype, out_scales,
                                           0x10, 1 << 40, 0x10, None)

    assert call(n_rows=0) == csa.OK
    assert call(n_rows=-1) == csa.ERR_INVALID_ARG
    assert call(max_n=-1) == csa.ERR_INVALID_ARG
    assert call(k=0) == csa.ERR_INVALID_ARG                      # a selection needs k >= 1
    assert call(q=None) == csa.ERR_INVALID_ARG
    assert call(layer=csa.make_layer(4, 0, 512, 64, 64)) == csa.ERR_INVALID_ARG
    assert call(q_dtype=csa.E4M3) == csa.ERR_UNSUPPORTED
    assert call(out_dtype=csa.E2M1) == csa.ERR_UNSUPPORTED
    assert call(out_dtype=csa.E4M3) == csa.ERR_INVALID_ARG      # e4m3 output without its scales
    assert call(comp=_paged(csa.E2M1, 64, 512)) == csa.ERR_UNSUPPORTED   # attention reads no e2m1
    assert call(comp=_paged(csa.BF16, 32, 512)) == csa.ERR_INVALID_ARG   # 256 / ratio rows a block
    assert call(swa=_paged(csa.BF16, 64, 512)) == csa.ERR_INVALID_ARG    # 256 window rows a block
    # the kernels take D a multiple of 32 up to 512 and heads a multiple of 8
    L48 = csa.make_layer(4, 8, 48, 16, 64)
    assert call(layer=L48, comp=_paged(csa.BF16, 64, 48), swa=_paged(csa.BF16, 256, 48)) == csa.ERR_UNSUPPORTED
    L1k = csa.make_layer(4, 8, 1024, 64, 64)
    assert call(layer=L1k, comp=_paged(csa.BF16, 64, 1024), swa=_paged(csa.BF16, 256, 1024)) == csa.ERR_UNSUPPORTED
    assert call(layer=csa.make_layer(4, 8, 512, 64, 12)) == csa.ERR_UNSUPPORTED


def test_indexer_validation_and_noalloc_refusal(lib):
    """csa_indexer_topk and csa_indexer_topk_noalloc share their argument
    checks; the allocation-free entry refuses a request larger than its fixed
    scratch before it looks the scratch up."""
    B = _bt()
    idx = _paged(csa.BF16, 64, 128)

    def call(fn, n_rows=4, q_dtype=csa.BF16, heads=64, dim=128, ratio=4, cache=idx, k=512, max_n=1000,
             q=0x10):
        args = [q, q_dtype, 0x10, n_rows, heads, dim, 0x10, 0x10, ratio, 8, ctypes.byref(cache),
                ctypes.byref(B), k, max_n, 0x10]
        if fn == "ws":
            return lib.csa_indexer_topk(*args, 0x10, 1 << 40, 0x10, None)
        return lib.csa_indexer_topk_noalloc(*args, 0x10, None)

    for fn in ("ws", "noalloc"):
        assert call(fn, n_rows=0) == csa.OK
        assert call(fn, n_rows=-1) == csa.ERR_INVALID_ARG
        assert call(fn, k=0) == csa.ERR_INVALID_ARG
        assert call(fn, max_n=-1) == csa.ERR_INVALID_ARG
        assert call(fn, ratio=3) == csa.ERR_INVALID_ARG          # the stride divides 256
        assert call(fn, q=None) == csa.ERR_INVALID_ARG
        assert call(fn, q_dtype=csa.E2M1) == csa.ERR_UNSUPPORTED
        assert call(fn, cache=_paged(csa.E4M3, 64, 128)) == csa.ERR_UNSUPPORTED   # keys: f32, bf16, e2m1
        assert call(fn, cache=_paged(csa.BF16, 32, 128)) == csa.ERR_INVALID_ARG
        assert call(fn, dim=512, cache=_paged(csa.BF16, 64, 512)) == csa.ERR_UNSUPPORTED  # dim <= 256
        assert call(fn, heads=512) == csa.ERR_UNSUPPORTED     # heads x dim <= 32768
    # 64 rows of 2^20 scores are 256 MiB, far beyond the fixed 16 MiB scratch
    assert call("noalloc", n_rows=64, max_n=1 << 20) == csa.ERR_WORKSPACE


def test_workspace_checks(lib):
    L = csa.make_layer(4, 8, 512, 64, 64)
    need = csa.indexer_topk_workspace_size(4, 262143, 512)
    assert need >= 4 * 262143 * 4
    idx = _paged(csa.E2M1, 64, 128)
    r = lib.csa_indexer_topk(0x10, csa.BF16, 0x10, 4, 64, 128, 0x10, 0x10, 4, 8, ctypes.byref(idx),
                             ctypes.byref(_bt()), 512, 262143, 0x10, 0x10, need - 1, 0x10, None)
    assert r == csa.ERR_WORKSPACE
    # attention with many splits needs a workspace; a small row count needs one
    ws = csa.sparse_attn_workspace_size(L, 4, 512)
    assert ws > 0
    P, S = _paged(csa.E4M3, 64, 512), _paged(csa.E4M3, 256, 512)
    r = lib.csa_sparse_attn_decode(ctypes.byref(L), 0x10, csa.BF16, 4, 0x10, 0x10, ctypes.byref(P),
                                   ctypes.byref(_bt()), 0x10, 512, 262143, ctypes.byref(S), ctypes.byref(_bt()),
                                   0x10, csa.E4M3, 0x10, None, 0, 0x10, None)
    assert r == csa.ERR_WORKSPACE
    # e4m3 output needs a scale buffer
    r = lib.csa_sparse_attn_decode(ctypes.byref(L), 0x10, csa.BF16, 4, 0x10, 0x10, ctypes.byref(P),
                                   ctypes.byref(_bt()), 0x10, 512, 262143, ctypes.byref(S), ctypes.byref(_bt()),
                                   0x10, csa.E4M3, None, 0x10, ws, 0x10, None)
    assert r == csa.ERR_INVALID_ARG


def test_topk_scratch_sizes(lib):
    """Rows of one 16384-entry chunk need only the score scratch; longer rows also
    need each chunk's top-k candidates (key and index) and a count.  Batches of
    fewer than 256 rows may instead be dealt over up to 256 CTAs that each keep
    two candidate lists of up to 2k (key, index) pairs, a count and a threshold
    each, plus each row's first CTA, list count and first list's slot."""
    def aligned(x):
        return (x + 255) // 256 * 256

    deal = 2 * aligned(2 * 256 * 1024 * 4) + 2 * aligned(2 * 256 * 4) + 3 * aligned(256 * 4)
    assert csa.indexer_topk_workspace_size(64, 16383, 512) == aligned(64 * 16383 * 4) + deal
    assert csa.indexer_topk_workspace_size(64, 16384, 512) == aligned(64 * 16384 * 4) + deal
    n = 262143
    chunks = (n + 16383) // 16384
    assert csa.indexer_topk_workspace_size(4, n, 512) == (aligned(4 * n * 4) + aligned(4 * chunks * (512 * 8 + 4))
                                                          + deal)
    assert csa.indexer_topk_workspace_size(256, 1000, 512) == aligned(256 * 1000 * 4)
    assert csa.indexer_topk_workspace_size(0, n, 512) == 0
