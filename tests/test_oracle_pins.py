"""Pins of the oracle against things other than itself: the pages' figures,
closed forms, library routines, invariants and brute force on tiny inputs.

Each test names the mistake it would catch.  CPU only.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import csa_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fig(name):
    with open(os.path.join(GOLDEN, "pages_figures.json")) as f:
        figs = {d["name"]: d["value"] for d in json.load(f)["figures"]}
    return figs[name]


# ------------------------------------------------------------------ RoPE


def test_rope_hand_values_pin_pairing_frequency_and_sign():
    # D=6, r=4, theta=1e4: frequencies theta^(0/4)=1 and theta^(-2/4)=0.01.
    # x = [7, -3, 1, 0, 1, 0] at p=100: dims 0,1 untouched; pair (2,3) turns by
    # 100 rad, pair (4,5) by 1 rad, counter-clockwise.
    x = np.array([7.0, -3.0, 1.0, 0.0, 1.0, 0.0])
    y = O.rope(x, 100, 4, 10000.0)
    want = [7.0, -3.0, math.cos(100.0), math.sin(100.0), math.cos(1.0), math.sin(1.0)]
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-13)
    # (0, 1) input turns to (-sin, cos)
    y2 = O.rope(np.array([0.0, 1.0]), 0.5, 2, 10000.0)
    np.testing.assert_allclose(y2, [-math.sin(0.5), math.cos(0.5)], atol=1e-15)


def test_rope_matches_complex_multiplication():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 32))
    pos = np.array([0, 3, 1000, 65537, 1 << 20])
    y = O.rope(x, pos, 16, 10000.0)
    z = x[:, 16::2] + 1j * x[:, 17::2]
    f = 10000.0 ** (-np.arange(8) * 2.0 / 16)
    zr = z * np.exp(1j * pos[:, None] * f[None, :])
    np.testing.assert_allclose(y[:, 16::2], zr.real, atol=1e-12)
    np.testing.assert_allclose(y[:, 17::2], zr.imag, atol=1e-12)
    np.testing.assert_array_equal(y[:, :16], x[:, :16])


def test_rope_inverse_undoes_rope_and_preserves_norm():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((8, 512))
    for p in (0, 1, 4095, 131072, (1 << 20) + 77):
        y = O.rope(x, p, 64, 10000.0)
        np.testing.assert_allclose(O.rope(y, p, 64, 10000.0, inverse=True), x, atol=1e-12)
        np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_dot_product_depends_on_offset_only():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    base = O.rope(q, 1000, 64, 1e4) @ O.rope(k, 900, 64, 1e4)
    for d in (256, 4096, 1 << 20):
        np.testing.assert_allclose(O.rope(q, 1000 + d, 64, 1e4) @ O.rope(k, 900 + d, 64, 1e4), base, rtol=1e-9)


# ------------------------------------------------------------------ RMSNorm


def test_rms_norm_hand_value():
    # mean(9, 16) = 12.5 -> rms = sqrt(12.5); gamma = (1, 2)
    y = O.rms_norm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    r = math.sqrt(12.5)
    np.testing.assert_allclose(y, [3.0 / r, 8.0 / r], rtol=1e-15)
    # eps enters under the root: x=(1,1), eps=3 -> 1/sqrt(1+3) = 0.5
    np.testing.assert_allclose(O.rms_norm(np.ones(2), np.ones(2), 3.0), [0.5, 0.5], rtol=1e-15)


def test_rms_norm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 512))
    y = O.rms_norm(x, np.ones(512), 1e-12)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-9)
    np.testing.assert_allclose(O.rms_norm(7.5 * x, np.ones(512), 1e-12), y, rtol=1e-9)


def test_query_norm_is_per_head():
    # heads are normalised one by one, not over H*D: scaling one head changes no other
    # head's output, and a head of (3, 4) with gamma (1, 2) gives the hand value above
    q = np.array([[[3.0, 4.0], [30.0, -40.0], [1.0, 1.0]]])  # [1, H=3, D=2]
    y = O.query_norm(q, np.array([1.0, 2.0]), 0.0)
    r = math.sqrt(12.5)
    np.testing.assert_allclose(y[0, 0], [3.0 / r, 8.0 / r], rtol=1e-15)
    np.testing.assert_allclose(y[0, 1], [3.0 / r, -8.0 / r], rtol=1e-15)
    np.testing.assert_allclose(y[0, 2], [1.0, 2.0], rtol=1e-15)
    assert y.shape == q.shape


# ------------------------------------------------------------------ geometry (pages' figures)


def test_block_geometry_matches_pages():
    assert O.BLOCK_POSITIONS == _fig("block_native_positions")
    assert O.entries_per_block(_fig("c4a_stride")) == _fig("c4a_entries_per_block")
    assert O.entries_per_block(_fig("c128a_stride")) == _fig("c128a_entries_per_block")
    assert O.window_span(0, 4, 8) == (_fig("c4a_entry0_first_token"), _fig("c4a_entry0_last_token"))
    assert O.window_span(5, 4, 8) == (20, 27)
    assert O.window_span(3, 128, 128) == (384, 511)


def test_entry_counts_at_one_million_match_pages():
    # "about 250k" c4a entries and "fewer than 8k" c128a entries for a 1M-token context
    for ctx in (10 ** 6, 1 << 20):
        n4 = O.n_visible(ctx, 4, 8)
        n128 = O.n_visible(ctx, 128, 128)
        assert abs(n4 - _fig("c4a_entries_at_1M_approx")) / _fig("c4a_entries_at_1M_approx") < 0.05
        assert n128 <= 8192
    assert O.n_visible(10 ** 6, 4, 8) == 249999
    assert O.n_visible(10 ** 6, 128, 128) == 7812 < _fig("c128a_entries_at_1M_upper")
    assert O.n_visible(1 << 20, 4, 8) == 262143
    assert O.n_visible(1 << 20, 128, 128) == 8192


@pytest.mark.parametrize("ratio,window", [(4, 8), (128, 128)])
def test_visibility_brute_force(ratio, window):
    # brute force: count entries whose every raw token lies before p
    for p in range(0, 700):
        brute = sum(1 for i in range(p + 1) if all(t < p for t in range(ratio * i, ratio * i + window)))
        assert O.n_visible(p, ratio, window) == brute
        assert all(O.is_visible(i, p, ratio, window) == (i < brute) for i in range(brute + 3))


def test_causal_boundary_c4a():
    # the entry over [4i, 4i+7] appears exactly when the query passes 4i+7
    for i in (0, 1, 9, 1000):
        assert not O.is_visible(i, 4 * i + 7, 4, 8)
        assert O.is_visible(i, 4 * i + 8, 4, 8)


@pytest.mark.parametrize("ratio,window", [(4, 8), (128, 128)])
def test_closing_entry_enumeration(ratio, window):
    closed = {}
    for t in range(0, 3000):
        i = O.closing_entry(t, ratio, window)
        if i is not None:
            assert i not in closed
            closed[i] = t
    for i, t in closed.items():
        assert t == ratio * i + window - 1
    assert sorted(closed) == list(range(len(closed)))


def test_swa_positions():
    assert list(O.swa_positions(1000)) == list(range(873, 1001))
    assert len(O.swa_positions(1000)) == _fig("swa_window")
    assert list(O.swa_positions(5)) == list(range(0, 6))


# ------------------------------------------------------------------ compressor


def test_uniform_gate_gives_window_mean():
    rng = np.random.default_rng(5)
    kv = rng.standard_normal((8, 16))
    c = O.gated_window_sum(kv, np.zeros((8, 16)), np.zeros((8, 16)))
    np.testing.assert_allclose(c, kv.mean(axis=0), rtol=1e-14)


def test_one_hot_bias_copies_chosen_offset_per_channel():
    # bias[j*(d), d] = +60 selects offset j*(d) in channel d (weight 1 - O(e^-60))
    rng = np.random.default_rng(6)
    kv = rng.standard_normal((8, 32))
    jstar = rng.integers(0, 8, size=32)
    bias = np.zeros((8, 32))
    bias[jstar, np.arange(32)] = 60.0
    c = O.gated_window_sum(kv, 0.01 * rng.standard_normal((8, 32)), bias)
    np.testing.assert_allclose(c, kv[jstar, np.arange(32)], atol=1e-20 + 1e-12)


def test_gate_shift_per_channel_is_invisible():
    # the softmax runs over offsets: a per-channel constant added to every offset cancels
    rng = np.random.default_rng(7)
    kv, z, b = rng.standard_normal((3, 128, 24))
    c0 = O.gated_window_sum(kv, z, b)
    c1 = O.gated_window_sum(kv, z + 5.0 * rng.standard_normal(24)[None, :], b)
    np.testing.assert_allclose(c1, c0, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("ratio,window,i,D", [(4, 8, 3, 64), (4, 8, 0, 64), (128, 128, 1, 320)])
def test_entry_window_geometry_by_one_hot_rows(ratio, window, i, D):
    # raw row t is the basis vector e_t: with a uniform gate the entry's support is its window
    T = ratio * i + window
    kv = np.eye(T, D)
    e = O.compressed_entry(kv, np.zeros((T, D)), 0, i, ratio, window, np.zeros((window, D)),
                           np.ones(D), 0.0, 0, 1e4)
    support = np.nonzero(np.abs(e) > 1e-9)[0]
    assert list(support) == list(range(ratio * i, ratio * i + window))
    np.testing.assert_allclose(e[support], math.sqrt(D / window), rtol=1e-9)


def test_entry_is_rotated_at_anchor_after_norm():
    # un-rotating the entry at its anchor 4i gives the normalised gated sum (non-uniform gain)
    rng = np.random.default_rng(8)
    D, i = 128, 5
    kv, z = rng.standard_normal((2, 40, D))
    bias = 0.1 * rng.standard_normal((8, D))
    gam = 1 + 0.3 * rng.standard_normal(D)
    e = O.compressed_entry(kv, z, 0, i, 4, 8, bias, gam, 1e-6, 64, 1e4)
    c = O.gated_window_sum(kv[20:28], z[20:28], bias)
    np.testing.assert_allclose(O.rope(e, 20, 64, 1e4, inverse=True), O.rms_norm(c, gam, 1e-6), atol=1e-12)
    # the anchor is the window's first token, not its last
    assert not np.allclose(O.rope(e, 27, 64, 1e4, inverse=True), O.rms_norm(c, gam, 1e-6), atol=1e-6)


def test_bias_is_indexed_by_offset_not_position():
    # moving the same raw rows four positions later gives the next entry the same pre-rotation value
    rng = np.random.default_rng(9)
    D = 32
    kv, z = rng.standard_normal((2, 12, D))
    bias = rng.standard_normal((8, D))
    e0 = O.compressed_entry(kv, z, 0, 0, 4, 8, bias, np.ones(D), 1e-6, 0, 1e4)
    kv2 = np.concatenate([rng.standard_normal((4, D)), kv])
    z2 = np.concatenate([rng.standard_normal((4, D)), z])
    e1 = O.compressed_entry(kv2, z2, 0, 1, 4, 8, bias, np.ones(D), 1e-6, 0, 1e4)
    np.testing.assert_allclose(e1, e0, rtol=1e-13)


# ------------------------------------------------------------------ indexer and top-k


def test_indexer_hand_value():
    # q = [[1,2],[-1,1]], w = [0.5, 2]
    # k0=[1,1]: dots (3, 0)  -> 0.5*3 + 2*0       = 1.5
    # k1=[2,-1]: dots (0,-3) -> relu -> 0         = 0
    # k2=[-1,2]: dots (3, 3) -> 0.5*3 + 2*3       = 7.5
    s = O.indexer_scores(np.array([[1.0, 2.0], [-1.0, 1.0]]), np.array([0.5, 2.0]),
                         np.array([[1.0, 1.0], [2.0, -1.0], [-1.0, 2.0]]))
    np.testing.assert_allclose(s, [1.5, 0.0, 7.5], rtol=0, atol=0)


def test_indexer_one_hot_weight_is_relu_of_one_head():
    rng = np.random.default_rng(10)
    q, k = rng.standard_normal((4, 16)), rng.standard_normal((50, 16))
    w = np.zeros(4)
    w[2] = 1.0
    np.testing.assert_allclose(O.indexer_scores(q, w, k), np.maximum(k @ q[2], 0), rtol=1e-14)


def test_topk_ties_go_to_lower_index():
    s = np.array([1.0, 3.0, 3.0, 2.0, 3.0])
    assert list(O.topk_select(s, 2)) == [1, 2]
    assert list(O.topk_select(s, 4)) == [1, 2, 4, 3]
    assert list(O.topk_select(s, 99)) == [1, 2, 4, 3, 0]
    assert list(O.topk_select(np.array([]), 5)) == []


def test_topk_against_python_sorted():
    rng = np.random.default_rng(11)
    for n, k in [(1, 1), (10, 3), (300, 64), (1000, 512), (40, 64)]:
        s = np.round(rng.standard_normal(n), 1)  # rounding makes many ties
        brute = sorted(range(n), key=lambda i: (-s[i], i))[:k]
        assert list(O.topk_select(s, k)) == brute


# ------------------------------------------------------------------ attention


def test_attention_against_torch_sdpa():
    rng = np.random.default_rng(12)
    H, D, m, p = 4, 64, 37, 12345
    q, keys = rng.standard_normal((H, D)), rng.standard_normal((m, D))
    got = O.attention(q, p, keys, 1 / math.sqrt(D), 16, 1e4)
    qr = torch.tensor(O.rope(q, p, 16, 1e4))[None, :, None, :]  # [1, H, 1, D]
    K = torch.tensor(keys)[None, None].expand(1, H, m, D)
    ref = torch.nn.functional.scaled_dot_product_attention(qr, K, K).squeeze(0).squeeze(1).numpy()
    np.testing.assert_allclose(got, O.rope(ref, p, 16, 1e4, inverse=True), atol=1e-12)


def test_single_key_returns_its_unrotated_value():
    rng = np.random.default_rng(13)
    x = rng.standard_normal(128)
    p = 777777
    out = O.attention(rng.standard_normal((3, 128)), p, O.rope(x, p, 64, 1e4)[None], 0.1, 64, 1e4)
    np.testing.assert_allclose(out, np.broadcast_to(x, (3, 128)), atol=1e-12)


def test_joint_softmax_equals_merge_of_parts():
    rng = np.random.default_rng(14)
    q, a, b = rng.standard_normal((4, 64)), rng.standard_normal((30, 64)), rng.standard_normal((9, 64))
    p = 4242
    joint = O.attention(q, p, np.concatenate([a, b]), 0.2, 16, 1e4)
    merged = O.merge_partials([O.attention_partial(q, p, a, 0.2, 16, 1e4),
                               O.attention_partial(q, p, b, 0.2, 16, 1e4)], p, 16, 1e4)
    np.testing.assert_allclose(merged, joint, atol=1e-12)


def test_keys_are_values_and_order_free():
    rng = np.random.default_rng(15)
    q1 = rng.standard_normal(64)
    keys = rng.standard_normal((20, 64))
    o = O.attention(np.stack([q1, q1]), 50, keys, 0.125, 16, 1e4)
    np.testing.assert_allclose(o[0], o[1], atol=0)
    o2 = O.attention(np.stack([q1, q1]), 50, keys[rng.permutation(20)], 0.125, 16, 1e4)
    np.testing.assert_allclose(o2, o, atol=1e-13)


def _chain_output(shift, seed=16):
    """Compress + window + attention for one query from raw rows at positions shift + t."""
    rng = np.random.default_rng(seed)
    D, r, T = 64, 16, 300
    kv, z = rng.standard_normal((2, T, D))
    bias = 0.1 * rng.standard_normal((8, D))
    gc, gs = 1 + 0.02 * rng.standard_normal((2, D))
    q = rng.standard_normal((4, D))
    p = shift + T - 1
    n = O.n_visible(p, 4, 8)
    ents = [O.compressed_entry(kv, z, shift, i, 4, 8, bias, gc, 1e-6, r, 1e4)
            for i in range(shift // 4, n)]
    swa = [O.swa_row(kv[t - shift], t, gs, 1e-6, r, 1e4) for t in O.swa_positions(p)]
    return O.attention(q, p, np.array(ents + swa), 1 / 8.0, r, 1e4)


def test_inverse_rope_makes_output_translation_invariant():
    base = _chain_output(0)
    for shift in (256, 4096, 1 << 20):
        np.testing.assert_allclose(_chain_output(shift), base, atol=1e-9)


def test_translation_invariance_fails_without_inverse_rope():
    # guards the test above: the un-inverted output does depend on absolute position
    rng = np.random.default_rng(17)
    x, q = rng.standard_normal(64), rng.standard_normal((1, 64))
    keys0 = O.rope(np.stack([x, -x]), np.array([3, 5]), 16, 1e4)
    keys1 = O.rope(np.stack([x, -x]), np.array([259, 261]), 16, 1e4)
    o0 = O.rope(O.attention(q, 7, keys0, 0.1, 16, 1e4), 7, 16, 1e4)
    o1 = O.rope(O.attention(q, 263, keys1, 0.1, 16, 1e4), 263, 16, 1e4)
    assert not np.allclose(o0, o1, atol=1e-6)


# ------------------------------------------------------------------ e4m3 codec


def test_e4m3_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(O.E4M3_TABLE), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(O.E4M3_TABLE[ok], ref[ok])
    assert np.nanmax(O.E4M3_TABLE) == 448.0


def test_e4m3_rounding_matches_torch_cast_incl_midpoints():
    finite = np.sort(np.unique(np.abs(O.E4M3_TABLE[~np.isnan(O.E4M3_TABLE)])))
    mids = (finite[1:] + finite[:-1]) / 2
    rng = np.random.default_rng(18)
    x = np.concatenate([finite, mids, -mids, rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 1e-2])
    x = x.astype(np.float32)
    ref = torch.tensor(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_e4m3(x), ref)


def test_e4m3_encode_roundtrip_and_saturation():
    for c in range(256):
        v = O.E4M3_TABLE[c]
        if not np.isnan(v):
            assert int(O.e4m3_encode(np.array([v]))[0]) == c
    np.testing.assert_array_equal(O.round_e4m3(np.array([500.0, 1e9, -465.0, 464.0])), [448, 448, -448, 448])


def test_row_quantisation_maps_amax_to_448():
    rng = np.random.default_rng(19)
    x = rng.standard_normal((50, 512)).astype(np.float32)
    codes, scale = O.quantize_rows_e4m3(x)
    amax_pos = np.argmax(np.abs(x), axis=1)
    assert np.all(np.abs(O.e4m3_decode(codes[np.arange(50), amax_pos])) == 448.0)
    np.testing.assert_allclose(scale, np.abs(x).max(axis=1) / 448.0, rtol=1e-7)
    err = np.abs(O.dequantize_rows_e4m3(codes, scale) - x)
    # half an e4m3 step: 2^-4 relative for normals, half of 2^-9 * scale below
    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scale[:, None]) * 1.0001)
    c0, s0 = O.quantize_rows_e4m3(np.zeros((1, 16), np.float32))
    assert s0[0] == 0 and np.all(O.e4m3_decode(c0) == 0)


# ------------------------------------------------------------------ e2m1 codec


def test_e2m1_table_is_the_format():
    # e2m1: magnitudes 0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6; bit 3 is the sign
    np.testing.assert_array_equal(O.E2M1_TABLE[:8], [0, 0.5, 1, 1.5, 2, 3, 4, 6])
    np.testing.assert_array_equal(O.E2M1_TABLE[8:], -O.E2M1_TABLE[:8])


def test_e2m1_round_half_even_and_saturation():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -0.74, -5.01])
    want = np.array([0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, -0.5, -6.0])
    np.testing.assert_array_equal(O.round_e2m1(x), want)
    # every grid value is kept, and values off the midpoints go to the nearer neighbour
    np.testing.assert_array_equal(O.round_e2m1(O.E2M1_TABLE), O.E2M1_TABLE)
    x = np.array([0.2, 0.3, 1.2, 1.3, 2.4, 2.6, 3.4, 3.6, 4.9, 5.1, 5.9])
    want = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 3.0, 4.0, 4.0, 6.0, 6.0])
    np.testing.assert_array_equal(O.round_e2m1(x), want)


def test_nvfp4_hand_example_packing_and_scale():
    # group of 16: [1, 2, 0 x 13, 6] -> amax 6 -> scale e4m3(1) = 1 -> codes 2, 4, 0..., 7
    x = np.zeros(16, np.float32)
    x[0], x[1], x[15] = 1.0, 2.0, 6.0
    packed, sc = O.quantize_nvfp4(x[None])
    assert packed.shape == (1, 8) and sc.shape == (1, 1)
    assert packed[0, 0] == 0x42 and packed[0, 7] == 0x70 and O.e4m3_decode(sc)[0, 0] == 1.0
    np.testing.assert_array_equal(O.dequantize_nvfp4(packed, sc)[0], x)


def test_nvfp4_error_bound_and_zero_group():
    rng = np.random.default_rng(20)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    x[3, 16:32] = 0
    packed, sc = O.quantize_nvfp4(x)
    d = O.dequantize_nvfp4(packed, sc)
    assert np.all(d[3, 16:32] == 0) and O.e4m3_decode(sc)[3, 1] == 0
    s = np.repeat(O.e4m3_decode(sc), 16, axis=1)
    # per group the error is at most one e2m1 step (2 units) plus the scale's own rounding
    assert np.all(np.abs(d - x) <= s * 1.0 + np.abs(x) * 0.0625 + 1e-12)


# ------------------------------------------------------------------ KV arithmetic (pages' figures)


def test_kv_per_sequence_at_1m_matches_pages():
    ctx = 1 << 20
    gib = 2.0 ** 30
    v4 = O.kv_bytes_per_sequence(ctx, _fig("c4a_layers"), _fig("c128a_layers"), 512, 128,
                                 entry_bytes=512 * 2, idx_entry_bytes=128 * 2) / gib
    assert round(v4, 2) == _fig("kv_gib_per_seq_1M_bf16")
    # a V3.2-style stack keeps every token: 576 latent+rope dims and a 128-dim indexer key, bf16
    v32 = _fig("total_layers") * ctx * (576 + 128) * 2 / gib
    assert round(v32, 1) == _fig("v32_kv_gib_61_layers")
    assert round(v32 / v4, 1) == _fig("reduction_vs_v32")
    # fp8 entries (512 B + fp32 scale) and fp4 indexer keys (64 B + 8 e4m3 scales)
    q = O.kv_bytes_per_sequence(ctx, 30, 31, 512, 128, entry_bytes=516, idx_entry_bytes=72) / gib
    assert 1.8 < v4 / q < 2.4 and round(v4 / q, 2) == 2.17


# ------------------------------------------------------------ partial token-wise fp8 (e4m3 + bf16 rotary dims)


def test_bf16_rounding_matches_torch_cast_incl_midpoints():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -130, 0.0])])
    x32 = x.astype(np.float32)
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_bf16(x32), want)


def test_partial_fp8_keeps_rotary_dims_in_bf16_and_scales_the_rest():
    """Rotary dims come back as their bf16 rounding whatever their size; the
    scale is the amax of the non-rotary dims only (large rotary values must not
    coarsen the fp8 part); the fp8 part is torch's e4m3 cast of x * 448 / amax."""
    rng = np.random.default_rng(4)
    D, r = 512, 64
    x = rng.standard_normal((6, D)).astype(np.float32)
    x[:, D - r:] *= 50.0  # rotary dims far larger than the rest
    codes, scale, rope = O.quantize_rows_e4m3_rope_bf16(x, r)
    assert codes.shape == (6, D - r) and rope.shape == (6, r)
    np.testing.assert_array_equal(rope, torch.from_numpy(x[:, D - r:]).to(torch.bfloat16).double().numpy())
    np.testing.assert_allclose(scale, np.abs(x[:, : D - r]).max(axis=1) / 448.0, rtol=1e-7)
    y = torch.from_numpy(x[:, : D - r] * (448.0 / np.abs(x[:, : D - r]).max(axis=1, keepdims=True)))
    want_codes = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes, want_codes)
    back = O.dequantize_rows_e4m3_rope_bf16(codes, scale, rope)
    assert back.shape == (6, D)
    # the fp8 part is within half an e4m3 step of x (relative 1/16 of the value's binade)
    err = np.abs(back[:, : D - r] - x[:, : D - r])
    assert np.all(err <= np.abs(x[:, : D - r]) / 16 + scale[:, None] * 2.0 ** -10)
    assert np.all(back[:, D - r:] == rope)

