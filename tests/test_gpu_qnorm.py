"""The query RMSNorm fused into the compressor launch (csa_compress_insert_qnorm).

"vLLM解密：DeepSeek-V4本地部署為何如此困難" §3.2, third fusion: the query norm
and the raw window key's norm + RoPE + insert share one kernel, warps given
statically to query heads or to the key.  Checked here:
  * q_out against the oracle's per-head RMSNorm (bf16 out: each element within
    2^-8 of its magnitude, i.e. one bf16 rounding of an fp32 result; f32 out:
    1e-5 relative);
  * the caches it writes are bit-identical to those of csa_compress_insert on
    the same tokens (the decode-sized fused kernel and the prefill ingest
    kernel both carry the extra warps);
  * in place (q_out is q) gives the same result.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import csa_oracle as O

pytestmark = pytest.mark.gpu


def _layer(idx, li):
    from compressed_sparse_long_c128a_gb300 import build as csa_build
    from harness import LayerDev

    csa_build.build()
    torch.cuda.empty_cache()
    wl = synth.workload(idx)
    ld = LayerDev(wl, wl.layers[li])
    ld.load_history()
    ld.setup_ingest()
    ld.stage_step()
    torch.cuda.synchronize()
    return ld


def _caches(ld):
    out = {}
    for name in ("comp", "swa", "state"):
        c = getattr(ld, name)
        out[name] = c.data.clone()
        if c.scales is not None:
            out[name + ".scales"] = c.scales.clone()
    return out


def _check_qout(ld, q_out, rows):
    L = ld.L
    prm = synth.layer_params(ld.wl, L)
    q = np.asarray(ld.host["q"], np.float64)[rows]
    want = O.query_norm(q, prm["gamma_q"], L.eps)
    got = q_out[torch.as_tensor(rows, device=q_out.device)].float().cpu().numpy().astype(np.float64)
    if q_out.dtype == torch.bfloat16:
        bound = np.abs(want) * 2.0 ** -8 + 1e-6
    else:
        bound = np.abs(want) * 1e-5 + 1e-6
    bad = np.abs(got - want) > bound
    assert not bad.any(), (f"{bad.sum()} of {bad.size} q_out elements off; worst "
                           f"{np.max(np.abs(got - want) - bound):.3g} over the bound")


@pytest.mark.parametrize("idx,li", [(0, 0), (2, 0), (4, 1), (4, 0)])
def test_qnorm_matches_oracle_and_leaves_caches_as_compress_insert(idx, li):
    ld = _layer(idx, li)
    io = ld.io
    q = io["q"]
    q_out = torch.full_like(q, float("nan"))
    ld.compress_insert_qnorm(io["kv"], io["gate"], io["seq_id"], io["pos"], q, q_out)
    torch.cuda.synchronize()
    ld.check("compress_insert_qnorm")
    fused = _caches(ld)
    ld.compress_insert(io["kv"], io["gate"], io["seq_id"], io["pos"])
    torch.cuda.synchronize()
    ld.check("compress_insert")
    plain = _caches(ld)
    for k in plain:
        assert torch.equal(fused[k], plain[k]), f"{k} differs between the fused and the plain insert"
    n = q.shape[0]
    rows = np.arange(n) if n <= 256 else np.unique(np.r_[0, 1, n - 1, np.random.default_rng(7).integers(0, n, 253)])
    _check_qout(ld, q_out, rows)


def test_qnorm_f32_output_and_in_place():
    ld = _layer(2, 0)
    io = ld.io
    q = io["q"]
    out32 = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    ld.compress_insert_qnorm(io["kv"], io["gate"], io["seq_id"], io["pos"], q, out32)
    q_in = q.clone()
    ld.compress_insert_qnorm(io["kv"], io["gate"], io["seq_id"], io["pos"], q_in, q_in)  # in place
    out16 = torch.empty_like(q)
    ld.compress_insert_qnorm(io["kv"], io["gate"], io["seq_id"], io["pos"], q, out16)
    torch.cuda.synchronize()
    ld.check("compress_insert_qnorm")
    rows = np.arange(q.shape[0])
    _check_qout(ld, out32, rows)
    _check_qout(ld, q_in, rows)
    assert torch.equal(q_in, out16)
