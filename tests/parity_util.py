"""Value and selection checks shared by the GPU parity tests.

The tolerance rules (stated with the tests that use them): fp32 1e-4 max-abs;
bf16 2e-2 max-abs and 1e-2 rel-L2 against the unrounded fp64 oracle; e4m3
within one e4m3 step of the oracle's code for every element and at most 0.1% of
elements on another code; a selection exact up to ties within 1e-5 of the k-th
score.
"""

import numpy as np

from oracle import csa_oracle as O


def _e4m3_step(v, scale):
    """Spacing of the e4m3 grid at |v| (scaled units), times scale."""
    a = np.abs(v) / np.where(scale > 0, scale, 1.0)
    _, ex = np.frexp(a)
    e = np.maximum(ex - 1, -6)
    return np.ldexp(1.0, e - 3) * scale


def _assert_values(got, want, dtype, what, scale=None, tail=0):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    if dtype == "e4m3r":  # e4m3 over the non-rotary dims, bf16 over the `tail` rotary dims
        dq = got.shape[-1] - tail
        _assert_values(got[..., :dq], want[..., :dq], "e4m3", f"{what} (e4m3 dims)", scale)
        _assert_values(got[..., dq:], want[..., dq:], "bf16", f"{what} (bf16 rotary dims)")
        return
    assert got.shape == want.shape, what
    assert np.all(np.isfinite(got)), what
    diff = np.abs(got - want)
    if dtype == "f32":
        assert diff.max() <= 1e-4, f"{what}: max-abs {diff.max():.3g}"
    elif dtype == "bf16":
        rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
        assert diff.max() <= 2e-2 and rel <= 1e-2, f"{what}: max-abs {diff.max():.3g} rel-L2 {rel:.3g}"
    elif dtype == "e4m3":
        sc = np.broadcast_to(np.asarray(scale, np.float64).reshape(-1, *([1] * (got.ndim - 1))), got.shape)
        step = np.maximum(_e4m3_step(want, sc), _e4m3_step(got, sc))
        assert np.all(diff <= step * 1.0001 + 1e-12), f"{what}: beyond one e4m3 step"
        # a different code moves the value by a full step; the per-row fp32 scale
        # (amax/448 of slightly different fp32 rows) only moves it by scale ulps
        frac = np.mean(diff > 0.25 * step)
        assert frac <= 1e-3, f"{what}: {frac:.2%} of elements on a different code"
    else:
        raise ValueError(dtype)


def _check_topk_row(gpu_row, scores, k, what):
    n = len(scores)
    kk = min(k, n)
    sel = gpu_row[gpu_row >= 0]
    assert np.sum(gpu_row < 0) == k - kk, f"{what}: padding"
    assert len(sel) == kk and len(np.unique(sel)) == kk, f"{what}: size / duplicates"
    assert sel.min() >= 0 and sel.max() < n, f"{what}: index range"
    ref = O.topk_select(scores, k)
    if kk == n:
        assert set(sel.tolist()) == set(range(n)), what
        return True
    sk = scores[ref[-1]]
    tau = 1e-5 * abs(sk)
    chosen = np.zeros(n, bool)
    chosen[sel] = True
    assert np.all(scores[chosen] >= sk - tau), f"{what}: a pick below the k-th score"
    assert np.all(scores[~chosen] <= sk + tau), f"{what}: an omitted entry above the k-th score"
    return set(sel.tolist()) == set(ref.tolist())
