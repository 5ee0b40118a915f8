"""The allocation-free indexer entry point, csa_indexer_topk_noalloc (GPU).

That entry point serves callers that cannot allocate device memory -- a
plugin inside a host runtime that owns every device byte and gives its
extensions no allocator, or a serving loop that may not allocate on its hot
path.  Instead of a caller-provided workspace it uses a fixed 16 MiB scratch
array inside the library.

These tests call it through the C ABI and check that two calls in a row
select exactly the entries the workspace entry point (csa_indexer_topk)
selects on the same inputs, and that a request needing more than the fixed
scratch is refused before anything runs.  The file is named so that pytest
collects it last; it builds its own inputs, so it passes alone in a fresh
process as well as after the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _indexer_setup(idx):
    """Indexer cache and step inputs of a workload's c4a layer (no attention state)."""
    from compressed_sparse_long_c128a_gb300 import build as csa_build
    from harness import LayerDev

    csa_build.build()
    wl = synth.workload(idx)
    ld = LayerDev(wl, wl.layers[0])
    for b in range(len(wl.seqs)):
        ld._store(synth.seq_index_keys(wl, ld.L, b), b, ld.idx, ld.tables["idx"])
    ld.stage_step()
    torch.cuda.synchronize()
    ld.check("indexer set-up")
    return ld


@pytest.mark.parametrize("idx", [0, 2, 3])
def test_noalloc_selects_what_the_workspace_entry_point_selects(idx):
    import compressed_sparse_long_c128a_gb300 as csa

    ld = _indexer_setup(idx)
    L, io = ld.L, ld.io
    max_n = max(ld.max_n, 1)
    ref = torch.full((ld.n_rows, L.topk), -3, dtype=torch.int32, device="cuda")
    csa.indexer_topk(io["q_idx"], io["w"], io["seq_id"], io["pos"], L.ratio, L.window, ld.idx, ld.tables["idx"],
                     L.topk, max_n, ref, ld.ws_idx, ld.err)
    torch.cuda.synchronize()
    assert csa.read_status(ld.err) == 0
    want = ref.cpu().numpy()
    for call in range(2):  # the second call finds the first call's leftovers in the shared scratch
        out = torch.full_like(ref, -7)
        csa.indexer_topk_noalloc(io["q_idx"], io["w"], io["seq_id"], io["pos"], L.ratio, L.window, ld.idx,
                                 ld.tables["idx"], L.topk, max_n, out, ld.err)
        torch.cuda.synchronize()
        assert csa.read_status(ld.err) == 0, f"call {call}"
        got = out.cpu().numpy()
        for r in range(ld.n_rows):
            assert set(got[r].tolist()) == set(want[r].tolist()), f"call {call}, row {r}"
        np.testing.assert_array_equal(np.sort(got, axis=1), np.sort(want, axis=1))


def test_noalloc_matches_the_workspace_entry_point_when_max_n_is_zero():
    """max_n = 0 declares that no row sees an entry: both entry points then
    report every row that does see one as a device bounds error and select
    nothing (all -1), the same way."""
    import compressed_sparse_long_c128a_gb300 as csa

    ld = _indexer_setup(0)
    L, io = ld.L, ld.io
    outs, status = [], []
    for noalloc in (False, True):
        out = torch.full((ld.n_rows, L.topk), 5, dtype=torch.int32, device="cuda")
        if noalloc:
            csa.indexer_topk_noalloc(io["q_idx"], io["w"], io["seq_id"], io["pos"], L.ratio, L.window, ld.idx,
                                     ld.tables["idx"], L.topk, 0, out, ld.err)
        else:
            csa.indexer_topk(io["q_idx"], io["w"], io["seq_id"], io["pos"], L.ratio, L.window, ld.idx,
                             ld.tables["idx"], L.topk, 0, out, None, ld.err)
        torch.cuda.synchronize()
        status.append(csa.read_status(ld.err))
        outs.append(out.cpu().numpy())
    assert status == [csa.ERR_DEVICE_BOUNDS, csa.ERR_DEVICE_BOUNDS]
    np.testing.assert_array_equal(outs[0], outs[1])
    assert np.all(outs[1] == -1)


def test_noalloc_refuses_requests_beyond_its_scratch():
    import compressed_sparse_long_c128a_gb300 as csa

    lib = csa.lib()
    # 16408 rows over 262143 entries need far more than the fixed scratch
    assert csa.indexer_topk_workspace_size(16408, 262143, 512) > 16 << 20
    cache = csa.Paged(0x1000, 0x2000, csa.E2M1, 10, 64, 128)
    bt = csa.BlockTableC(0x3000, 2, 4)
    st = lib.csa_indexer_topk_noalloc(0x10, csa.BF16, 0x10, 16408, 64, 128, 0x10, 0x10, 4, 8, ctypes.byref(cache),
                                      ctypes.byref(bt), 512, 262143, 0x10, 0x10, None)
    assert st == csa.ERR_WORKSPACE
