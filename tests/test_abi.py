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
