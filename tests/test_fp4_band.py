"""The e2m1 band comparison used by the indexer-key compressor's GPU test,
pinned on the CPU: it accepts the bytes fp32 arithmetic can produce for the
oracle's entries and rejects planted mistakes of the kinds a kernel makes."""

import numpy as np
import pytest

import fp4_band
import synth
from oracle import csa_oracle as O

RATIO, WINDOW, DIM, ROPE, THETA, EPS = 4, 8, 128, 64, 10000.0, 1e-6


@pytest.fixture(scope="module")
def ref():
    case = synth.index_key_case(5, (300, 129))
    x = np.concatenate([O.complete_entries(case["kv"][b].astype(np.float64), case["gate"][b].astype(np.float64),
                                           RATIO, WINDOW, case["bias"], case["gamma"], EPS, ROPE, THETA)
                        for b in range(2)])
    return case, x


def _fp32_bytes(x, seed=0, rel=1e-6):
    """Bytes of the codec applied to x perturbed as fp32 arithmetic would perturb it."""
    rng = np.random.default_rng(seed)
    x32 = (x * (1.0 + rel * rng.standard_normal(x.shape))).astype(np.float32)
    return O.quantize_nvfp4(x32)


def test_complete_entries_count_and_first_entry(ref):
    case, x = ref
    assert x.shape == ((300 - 8) // 4 + 1 + (129 - 8) // 4 + 1, DIM)
    kv, gate = case["kv"][0].astype(np.float64), case["gate"][0].astype(np.float64)
    np.testing.assert_array_equal(x[0], O.compressed_entry(kv, gate, 0, 0, RATIO, WINDOW, case["bias"],
                                                           case["gamma"], EPS, ROPE, THETA))
    assert O.complete_entries(kv[:7], gate[:7], RATIO, WINDOW, case["bias"], case["gamma"], EPS, ROPE,
                              THETA).shape == (0, DIM)


def test_accepts_fp32_arithmetic(ref):
    _, x = ref
    for seed in range(3):
        p, s = _fp32_bytes(x, seed)
        amb_s, amb_c = fp4_band.check_nvfp4(p, s, x)
        assert amb_s < 0.01 and amb_c < 0.01
    p, s = O.quantize_nvfp4(x)  # the exact value's own bytes
    fp4_band.check_nvfp4(p, s, x)


def _unambiguous_code(x, s):
    """(entry, element) whose code is fixed by the band, with the rounding interval's middle far from 0."""
    codes = fp4_band.unpack_codes(O.quantize_nvfp4(x)[0]).astype(int)
    sc = np.repeat(O.e4m3_decode(s), 16, axis=1)
    y = np.abs(x) / sc
    ok = (y > 1.2) & (y < 5.5) & (np.abs(y - np.round(y * 2) / 2) > 0.1)
    i, j = np.argwhere(ok)[0]
    return i, j, codes


@pytest.mark.parametrize("mistake", ["code_step", "scale_step", "nibble_order", "sign", "no_rope",
                                     "window_shift", "scale_rule"])
def test_rejects_planted_mistakes(ref, mistake):
    case, x = ref
    p, s = _fp32_bytes(x)
    if mistake == "code_step":
        i, j, codes = _unambiguous_code(x, s)
        c = codes[i, j]
        codes[i, j] = (c & 8) | ((c & 7) + (1 if (c & 7) < 7 else -1))
        p = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    elif mistake == "scale_step":
        s = s.copy()
        s[3, 2] += 1
    elif mistake == "nibble_order":
        p = ((p >> 4) | (p << 4)).astype(np.uint8)
    elif mistake == "sign":
        i, j, codes = _unambiguous_code(x, s)
        codes[i, j] ^= 8
        p = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    else:
        kv, gate = case["kv"][0].astype(np.float64), case["gate"][0].astype(np.float64)
        bias, rope = case["bias"], ROPE
        if mistake == "no_rope":
            rope = 0
        if mistake == "window_shift":
            bias = np.roll(bias, 1, axis=0)
        y = O.complete_entries(kv, gate, RATIO, WINDOW, bias, case["gamma"], EPS, rope, THETA)
        if mistake == "scale_rule":
            y = y * (6.0 / 4.0)  # amax mapped to 4 instead of 6
        p, s = O.quantize_nvfp4(y)
        x = x[: len(y)]
    with pytest.raises(AssertionError):
        fp4_band.check_nvfp4(p, s, x)
