"""Plants plausible mistakes in the oracle, one at a time, on the CPU, and
checks that the pins of tests/test_oracle_pins.py catch every one.

Each mutation replaces one oracle function or table for the duration of one
run of all the pins (through pytest's monkeypatch, so nothing leaks out), and
at least one pin must fail.  The list covers the slips a restatement of the
method is prone to: RoPE sign, pairing, frequency exponent, rotated dims and
angle precision; softmax axis and bias indexing of the compressor; anchor and
order of norm and RoPE; RMSNorm epsilon and gain; the attention's inverse
RoPE, scale and split merge; tie order and visibility of the selection; relu
and weights of the indexer; the e4m3, e2m1 and bf16 codecs; the partial fp8
row scale; the query norm's extent; geometry constants.
"""

import numpy as np
import pytest

import test_oracle_pins as P
from oracle import csa_oracle as O

_rope, _entry, _rms, _attn, _topk = O.rope, O.compressed_entry, O.rms_norm, O.attention, O.topk_select
_gws, _merge, _quant, _e4m3_value = O.gated_window_sum, O.merge_partials, O.quantize_nvfp4, O.e4m3_value


def _rope_half(x, pos, rope_dim, theta, inverse=False):
    """Rotate-half pairing (d, d + r/2) instead of adjacent pairs."""
    x = np.array(x, dtype=np.float64, copy=True)
    if rope_dim == 0:
        return x
    D, h = x.shape[-1], rope_dim // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * O.rope_inv_freq(rope_dim, theta)
    ang = -ang if inverse else ang
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., D - rope_dim:D - h].copy(), x[..., D - h:].copy()
    x[..., D - rope_dim:D - h] = a * c - b * s
    x[..., D - h:] = a * s + b * c
    return x


def _rope_first_dims(x, pos, rope_dim, theta, inverse=False):
    x = np.array(x, dtype=np.float64, copy=True)
    y = _rope(x[..., ::-1], pos, rope_dim, theta, inverse)[..., ::-1]
    return np.ascontiguousarray(y)


def _rope_fp32_angle(x, pos, rope_dim, theta, inverse=False):
    x = np.array(x, dtype=np.float64, copy=True)
    if rope_dim == 0:
        return x
    D = x.shape[-1]
    ang = (np.asarray(pos, dtype=np.float32)[..., None] * O.rope_inv_freq(rope_dim, theta).astype(np.float32))
    ang = -ang.astype(np.float64) if inverse else ang.astype(np.float64)
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., D - rope_dim::2].copy(), x[..., D - rope_dim + 1::2].copy()
    x[..., D - rope_dim::2] = a * c - b * s
    x[..., D - rope_dim + 1::2] = a * s + b * c
    return x


def _gws_channel_axis(kv_win, gate_win, bias):
    logits = np.asarray(gate_win, np.float64) + np.asarray(bias, np.float64)
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    return ((e / e.sum(axis=1, keepdims=True)) * np.asarray(kv_win, np.float64)).sum(axis=0)


def _entry_bias_by_position(kv, gate, first_pos, i, ratio, window, bias, *rest):
    return _entry(kv, gate, first_pos, i, ratio, window, np.roll(bias, (ratio * i) % window, axis=0), *rest)


def _entry_anchor_last(kv, gate, first_pos, i, ratio, window, bias, gamma_c, eps, rope_dim, theta):
    e = _entry(kv, gate, first_pos, i, ratio, window, bias, gamma_c, eps, rope_dim, theta)
    lo, hi = O.window_span(i, ratio, window)
    return _rope(_rope(e, lo, rope_dim, theta, inverse=True), hi, rope_dim, theta)


def _entry_rope_before_norm(kv, gate, first_pos, i, ratio, window, bias, gamma_c, eps, rope_dim, theta):
    lo, hi = O.window_span(i, ratio, window)
    c = _gws(kv[lo - first_pos:hi - first_pos + 1], gate[lo - first_pos:hi - first_pos + 1], bias)
    return _rms(_rope(c, lo, rope_dim, theta), gamma_c, eps)


def _rms_eps_outside(x, gamma, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * np.asarray(gamma, np.float64)


def _attn_no_inverse(q, p, keys, scale, rope_dim, theta):
    return _rope(_attn(q, p, keys, scale, rope_dim, theta), p, rope_dim, theta)


def _attn_scale_squared(q, p, keys, scale, rope_dim, theta):
    return _attn(q, p, keys, scale * scale, rope_dim, theta)


def _merge_no_rescale(parts, p, rope_dim, theta):
    l = sum(pt[1] for pt in parts)
    acc = sum(pt[2] for pt in parts)
    return _rope(acc / l[:, None], p, rope_dim, theta, inverse=True)


def _topk_ties_high(scores, k):
    s = np.asarray(scores, np.float64)
    order = np.lexsort((-np.arange(len(s)), -s))
    return order[: min(k, len(s))].astype(np.int64)


def _quant_nibbles_swapped(x):
    packed, sc = _quant(x)
    return ((packed >> 4) | (packed << 4)).astype(np.uint8), sc


def _e4m3_value_subnormal(code):
    v = _e4m3_value(code)
    return v / 2.0 if ((code >> 3) & 0xF) == 0 else v


def _round_e2m1_step(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    step = np.where(a < 4.0, 0.5, 2.0)
    r = np.minimum(np.rint(a / step) * step, O.E2M1_MAX)
    return np.where(x < 0, -r, r)


def _round_e4m3_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)
    step = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
    r = np.minimum(np.floor(a / step) * step, O.E4M3_MAX)
    return np.where(x < 0, -r, r)


def _query_norm_joint(q, gamma_q, eps):
    """One RMS over all heads of a row instead of one per head."""
    q = np.asarray(q, np.float64)
    ms = np.mean(q * q, axis=(-2, -1), keepdims=True)
    return q / np.sqrt(ms + eps) * np.asarray(gamma_q, np.float64)


def _partial_fp8_scale_all_dims(x, rope_dim):
    """The row scale taken over every dim, rotary ones included."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    am = np.abs(x).max(axis=-1)
    inv = np.where(am > 0, 448.0 / np.where(am > 0, am, 1.0), 0.0).astype(np.float32)
    codes = O.e4m3_encode(x[..., : d - rope_dim] * inv[..., None])
    return codes, (am / 448.0).astype(np.float32), O.round_bf16(x[..., d - rope_dim:])


def _round_bf16_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)
    step = np.ldexp(1.0, np.maximum(ex, -125) - 8)
    r = np.floor(a / step) * step
    return np.where(x < 0, -r, r)


MUTATIONS = {
    "query_norm_over_all_heads": {"query_norm": _query_norm_joint},
    "partial_fp8_scale_over_all_dims": {"quantize_rows_e4m3_rope_bf16": _partial_fp8_scale_all_dims},
    "bf16_truncating_round": {"round_bf16": _round_bf16_truncate},
    "rope_sign": {"rope": lambda x, pos, r, th, inverse=False: _rope(x, pos, r, th, not inverse)},
    "rope_pairing_rotate_half": {"rope": _rope_half},
    "rope_frequency_exponent": {"rope_inv_freq": lambda r, th: np.power(float(th), -np.arange(r // 2) / r)},
    "rope_first_dims": {"rope": _rope_first_dims},
    "rope_fp32_angle": {"rope": _rope_fp32_angle},
    "softmax_over_channels": {"gated_window_sum": _gws_channel_axis},
    "bias_by_position": {"compressed_entry": _entry_bias_by_position},
    "anchor_at_last_token": {"compressed_entry": _entry_anchor_last},
    "rope_before_norm": {"compressed_entry": _entry_rope_before_norm},
    "eps_outside_sqrt": {"rms_norm": _rms_eps_outside},
    "norm_without_gain": {"rms_norm": lambda x, g, eps: _rms(x, np.ones(np.shape(x)[-1]), eps)},
    "no_inverse_rope": {"attention": _attn_no_inverse},
    "scale_squared": {"attention": _attn_scale_squared},
    "merge_without_rescale": {"merge_partials": _merge_no_rescale},
    "ties_to_higher_index": {"topk_select": _topk_ties_high},
    "visible_at_last_token": {"is_visible": lambda i, p, r, w: O.window_span(i, r, w)[1] <= p,
                              "n_visible": lambda p, r, w: 0 if p < w - 1 else (p - w + 1) // r + 1},
    "indexer_without_relu": {"indexer_scores": lambda q, w, k: (np.asarray(k, float) @ np.asarray(q, float).T)
                             @ np.asarray(w, float)},
    "indexer_without_weights": {"indexer_scores": lambda q, w, k: np.maximum(
        np.asarray(k, float) @ np.asarray(q, float).T, 0).sum(axis=1)},
    "e4m3_subnormal_binade": {"E4M3_TABLE": np.array([_e4m3_value_subnormal(c) for c in range(256)])},
    "e4m3_truncating_round": {"round_e4m3": _round_e4m3_truncate},
    "e2m1_step": {"round_e2m1": _round_e2m1_step},
    "e2m1_nibble_order": {"quantize_nvfp4": _quant_nibbles_swapped},
    "nvfp4_scale_constant": {"E2M1_MAX": 4.0},
    "window_of_127_rows": {"swa_positions": lambda p, swa=128: range(max(0, p - swa + 2), p + 1)},
    "block_of_128_positions": {"BLOCK_POSITIONS": 128},
    "window_stride_from_window": {"window_span": lambda i, r, w: (w * i, w * i + w - 1)},
}


def _pin_cases():
    for name in sorted(dir(P)):
        fn = getattr(P, name)
        if not name.startswith("test_") or not callable(fn):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            yield name, fn, {}
            continue
        names = [a.strip() for a in marks[0].args[0].split(",")]
        for v in marks[0].args[1]:
            yield name, fn, dict(zip(names, v if isinstance(v, tuple) else (v,)))


def _failing_pins():
    failed = []
    for name, fn, kw in _pin_cases():
        try:
            fn(**kw)
        except Exception:  # an assertion, or an error the mutation provokes
            failed.append(name)
    return failed


def test_pins_pass_on_the_oracle_as_it_is():
    assert _failing_pins() == []


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_a_planted_mistake_fails_a_pin(mutation, monkeypatch):
    for attr, value in MUTATIONS[mutation].items():
        monkeypatch.setattr(O, attr, value)
    assert _failing_pins(), f"no pin catches {mutation}"
