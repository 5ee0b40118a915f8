"""Indexer-key compressor on the GPU: csa_compress_insert with no window cache,
writing the c4a indexer cache (e2m1 with e4m3 group scales, or bf16), against
the oracle's entries (`complete_entries` over the same seeded streams).

Three sequences of 1000, 777 and 64 raw tokens (positions 0..n-1) go in two
calls, all but the last 37 tokens of each and then the rest, so some windows
span the calls.  Checked: every complete window's entry (e2m1: the band
comparison of `fp4_band`; bf16: 2e-2 max-abs and 1e-2 rel-L2 against the fp64
entry), and that the rows of entries whose window is not complete stay zero.

The file name sorts after the parity tests, so that under -x a failure here
stops none of them, and before the allocation-free entry point's test, which
is collected last.
"""

import numpy as np
import pytest
import torch

import fp4_band
import synth
from oracle import csa_oracle as O

pytestmark = pytest.mark.gpu

RATIO, WINDOW, DIM, ROPE, THETA, EPS = 4, 8, 128, 64, 10000.0, 1e-6
LENGTHS = (1000, 777, 64)
SPLIT = 37
SEED = 11
ROWS = synth.BLOCK_POSITIONS // RATIO  # entries per logical block


def _compress(dtype_name):
    import compressed_sparse_long_c128a_gb300 as csa
    from compressed_sparse_long_c128a_gb300 import build as csa_build

    csa_build.build()
    case = synth.index_key_case(SEED, LENGTHS, DIM, WINDOW, "bf16")
    layer = csa.make_layer(RATIO, WINDOW, DIM, ROPE, 1, 128, THETA, EPS)
    nb = case["n_blocks"]
    state = csa.PagedCache.empty(nb, synth.BLOCK_POSITIONS, 2 * DIM, csa.BF16)
    idx = csa.PagedCache.empty(nb, ROWS, DIM, csa.DTYPES[dtype_name])
    tables = {k: torch.from_numpy(t).cuda() for k, t in case["tables"].items()}
    bias = torch.from_numpy(case["bias"]).cuda()
    gamma = torch.from_numpy(case["gamma"]).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def dev(parts, dtype):
        return torch.from_numpy(np.concatenate(parts)).to(dtype).cuda()

    for part in (0, 1):
        kv, gate, seq, pos = [], [], [], []
        for b, n in enumerate(LENGTHS):
            cut = max(0, n - SPLIT)
            lo, hi = (0, cut) if part == 0 else (cut, n)
            kv.append(case["kv"][b][lo:hi])
            gate.append(case["gate"][b][lo:hi])
            seq.append(np.full(hi - lo, b, np.int32))
            pos.append(np.arange(lo, hi, dtype=np.int32))
        csa.compress_insert(layer, dev(kv, torch.bfloat16), dev(gate, torch.bfloat16), dev(seq, torch.int32),
                            dev(pos, torch.int32), bias, gamma, None, state, tables["state"], None, None, idx,
                            tables["idx"], err)
    torch.cuda.synchronize()
    assert csa.read_status(err) == 0
    return case, idx


def _entries(case, b):
    return O.complete_entries(case["kv"][b].astype(np.float64), case["gate"][b].astype(np.float64), RATIO, WINDOW,
                              case["bias"], case["gamma"], EPS, ROPE, THETA)


def _read(t, case, b, ids):
    """Rows of logical entries `ids` of sequence b from a [blocks, ROWS, ...] tensor."""
    blk = case["tables"]["idx"][b, ids // ROWS]
    return t[torch.from_numpy(blk).long().cuda(), torch.from_numpy(ids % ROWS).long().cuda()].cpu()


def _untouched(idx, case, b, m):
    n_rows = ROWS * int(np.sum(case["tables"]["idx"][b] >= 0))
    rest = np.arange(m, n_rows)
    assert not bool((_read(idx.data, case, b, rest) != 0).any()), f"seq {b}: entries past the last window"
    if idx.scales is not None:
        assert not bool((_read(idx.scales, case, b, rest) != 0).any()), f"seq {b}: scales past the last window"


def test_e2m1_indexer_keys():
    case, idx = _compress("e2m1")
    for b in range(len(LENGTHS)):
        x = _entries(case, b)
        ids = np.arange(len(x))
        amb_s, amb_c = fp4_band.check_nvfp4(_read(idx.data, case, b, ids).numpy(),
                                            _read(idx.scales, case, b, ids).numpy(), x)
        assert amb_s < 0.01 and amb_c < 0.01, f"seq {b}: band used by {amb_s:.3%} of scales, {amb_c:.3%} of codes"
        _untouched(idx, case, b, len(x))


def test_bf16_indexer_keys():
    case, idx = _compress("bf16")
    for b in range(len(LENGTHS)):
        x = _entries(case, b)
        got = _read(idx.data, case, b, np.arange(len(x))).to(torch.float64).numpy()
        assert np.max(np.abs(got - x)) <= 2e-2, f"seq {b}: max-abs"
        assert np.linalg.norm(got - x) / np.linalg.norm(x) <= 1e-2, f"seq {b}: rel-L2"
        _untouched(idx, case, b, len(x))
