"""Comparison of e2m1 cache bytes written from fp32 arithmetic with the
oracle's fp64 values (test helper; uses only the oracle's codec).

The kernel computes an entry in fp32, so near a rounding decision its code
may differ from the one the exact value gets.  Each decision is therefore
checked against the interval [x - e, x + e], e = rel * |x| + abs, around the
oracle's value x:
  * the group scale (e4m3 of amax/6) must be one that some amax in the
    interval rounds to;
  * with the kernel's own scale s, each code must decode to a value between
    the e2m1 roundings of (x - e)/s and (x + e)/s;
  * a zero scale must come with zero codes.
Where the interval holds a single rounding the byte must match exactly; the
fraction of decisions that fell inside a wider interval is returned, so a
caller can bound how much the band was used.
"""

import numpy as np

from oracle import csa_oracle as O


def unpack_codes(packed) -> np.ndarray:
    """[..., d/2] bytes -> [..., d] codes, element 2j in the low nibble of byte j."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def check_nvfp4(packed, scale_codes, x_ref, rel: float = 2e-5, abs_: float = 2e-5):
    """Raise AssertionError on a byte outside the band; return (fraction of
    ambiguous scales, fraction of ambiguous codes)."""
    x = np.asarray(x_ref, dtype=np.float64)
    n, d = x.shape
    g = O.NVFP4_GROUP
    codes = unpack_codes(packed).reshape(n, d // g, g)
    sc = np.asarray(scale_codes, dtype=np.uint8).reshape(n, d // g)
    xg = x.reshape(n, d // g, g)
    err = rel * np.abs(xg) + abs_

    assert np.all(sc < 0x80), "negative group scale"
    s = O.e4m3_decode(sc)
    amax = np.max(np.abs(xg), axis=-1)
    amax_e = np.max(err, axis=-1)
    s_lo = O.round_e4m3(np.maximum(amax - amax_e, 0.0) / O.E2M1_MAX)
    s_hi = O.round_e4m3((amax + amax_e) / O.E2M1_MAX)
    bad = (s < s_lo) | (s > s_hi)
    assert not np.any(bad), f"{int(bad.sum())} group scales outside the band, first at {np.argwhere(bad)[0]}"

    v = O.E2M1_TABLE[codes]
    zero = s == 0
    assert np.all(v[zero] == 0), "codes under a zero scale"
    sd = np.where(zero, 1.0, s)[..., None]
    lo = O.round_e2m1((xg - err) / sd)
    hi = O.round_e2m1((xg + err) / sd)
    live = ~np.broadcast_to(zero[..., None], v.shape)
    bad = live & ((v < lo) | (v > hi))
    assert not np.any(bad), (f"{int(bad.sum())} codes outside the band, first at {np.argwhere(bad)[0]}: "
                             f"{v[bad][0]} not in [{lo[bad][0]}, {hi[bad][0]}]")
    return float(np.mean(s_lo != s_hi)), float(np.mean(live & (lo != hi)))
