"""Oracle for compressed sparse attention (c4a / c128a): plain fp64 numpy.

TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the CPU
baseline leg of the benchmark may import this package.  The library never
does, and this file shares no code, table or helper with the CUDA path.

Sources, cited as (page, section):
  [Support]  "vLLM DeepSeek V4 Support: Efficient Long-context Attention"
             (agentlenshq.com)
  [部署]     "vLLM解密：DeepSeek-V4本地部署為何如此困難" (yhxrc.cn)
  [延迟]     "DeepSeek V4 inference latency optimization" (blog.hotdry.top)

What the pages fix, and the readings taken where they leave a step open:
  * c4a entry i is a weighted sum of raw tokens [4i, 4i+7] (window 8, stride 4),
    rotated at anchor 4i; c128a entry i sums [128i, 128i+127] at anchor 128i
    ([延迟] "KV 缓存压缩"; [Support] "DeepSeek V4 Attention Architecture").
    Reading: the weights are, per channel, a softmax over the window offsets j
    of the token's gate logit plus a learned bias indexed by the offset j.
  * right after compression the entry goes through RMSNorm, then RoPE, then
    into the cache ([部署] §3.2, first fusion).  Reading: RMSNorm over all D
    dims with eps = 1e-6; RoPE on the last r dims.
  * RoPE reading: theta = 10000, interleaved pairs (D-r+2k, D-r+2k+1) turned
    by pos * theta^(-2k/r); no frequency scaling.  Angles are formed in fp64.
  * keys and values are one shared vector, and the attention output gets an
    inverse RoPE so that it carries relative position only ([Support]
    "DeepSeek V4 Attention Architecture", first bullet; [部署] §二 item 1).
  * an entry may not contain future tokens ([延迟] "注意力计算剪枝").  Reading:
    entry i is visible to a query at p iff its last token is before p.
  * raw sliding window of 128 tokens ([Support] "Short Sliding Window").
    Reading: rows [p-127, p], each RMS-normalised with its own gain and rotated
    at its own position; one softmax over the selected entries and the window.
  * DSA top-k over the compressed entries, k = 512 on c4a ([部署] §二 item 3).
    Reading: score_i = sum_h w_h * relu(q_h . k_i) with no extra scale; ties
    go to the lower entry index; fewer than k visible entries -> all of them.
  * c128a layers attend densely to every visible entry ([延迟] "注意力计算剪枝").
  * logical block of 256 native positions: 64 c4a or 2 c128a entries per block
    ([Support] "KV Cache Memory Management"; [部署] §3.1 (1)).
  * fp8 attention cache / fp4 indexer cache ([Support] "DeepSeek V4 Attention
    Architecture", last paragraph).  Reading: e4m3 with one fp32 scale per row
    (amax / 448); e2m1 with one e4m3 scale per 16 elements (amax16 / 6, rounded
    to e4m3).  The codec's rounding decisions are taken in fp32, the precision
    the kernels take them in.
  * decode reads a "partial token-wise fp8" cache ([部署] §二).  Reading: per
    row, e4m3 codes with one fp32 scale (amax / 448) for the non-rotary dims and
    bf16 for the rotary dims (`quantize_rows_e4m3_rope_bf16`).
  * the indexer K cache has its own compress + RMSNorm + RoPE + insert kernel
    ([部署] §3.2, first fusion).  Reading: the same compressor (c4a stride and
    window) over the indexer's own raw streams at its dim, with its own bias and
    gain, RoPE on its last 64 dims, no sliding window (`complete_entries`).
"""

from __future__ import annotations

import math

import numpy as np

BLOCK_POSITIONS = 256
E4M3_MAX = 448.0
E2M1_MAX = 6.0
NVFP4_GROUP = 16

# ============================================================ RoPE


def rope_inv_freq(rope_dim: int, theta: float) -> np.ndarray:
    """Frequencies theta^(-2k/r), k < r/2, in fp64 (reading of RoPE; see header)."""
    k = np.arange(rope_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * k / rope_dim)


def rope(x, pos, rope_dim: int, theta: float, inverse: bool = False) -> np.ndarray:
    """Rotate the last `rope_dim` dims of x[..., D] at position(s) `pos`.

    Pair k is (D - r + 2k, D - r + 2k + 1), turned by the angle pos * theta^(-2k/r)
    (by its negative when `inverse`).  `pos` broadcasts against x[..., 0].
    [延迟] "KV 缓存压缩" (RoPE at the anchor; inverse RoPE on the output).
    """
    x = np.array(x, dtype=np.float64, copy=True)
    if rope_dim == 0:
        return x
    D = x.shape[-1]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(rope_dim, theta)
    if inverse:
        ang = -ang
    c, s = np.cos(ang), np.sin(ang)
    a = x[..., D - rope_dim::2].copy()
    b = x[..., D - rope_dim + 1::2].copy()
    x[..., D - rope_dim::2] = a * c - b * s
    x[..., D - rope_dim + 1::2] = a * s + b * c
    return x


# ============================================================ RMSNorm


def rms_norm(x, gamma, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gamma over the last axis.  [部署] §3.2, first fusion."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)


def query_norm(q, gamma_q, eps: float) -> np.ndarray:
    """RMSNorm of every query head on its own: q [..., H, D] -> same shape, each
    [D] vector divided by its own root mean square and scaled by gamma_q [D].
    The Q half of the third fusion of "vLLM解密" §3.2 (Q norm + KV RoPE + K
    insert); no RoPE here, the attention rotates the query."""
    return rms_norm(q, gamma_q, eps)


# ============================================================ compressor geometry


def window_span(i: int, ratio: int, window: int):
    """First and last raw position summed into compressed entry i; the anchor is the first.
    [延迟] "KV 缓存压缩": entry i of c4a covers [4i, 4i+7] and is rotated at 4i."""
    return ratio * i, ratio * i + window - 1


def is_visible(i: int, p: int, ratio: int, window: int) -> bool:
    """Entry i may be read by a query at p iff all its tokens lie before p.  [延迟] "注意力计算剪枝"."""
    return window_span(i, ratio, window)[1] < p


def n_visible(p: int, ratio: int, window: int) -> int:
    """Number of entries visible at query position p (they are entries 0 .. n-1)."""
    if p < window:
        return 0
    return (p - window) // ratio + 1


def entries_per_block(ratio: int) -> int:
    """Compressed entries in one 256-position logical block: 64 for c4a, 2 for c128a.
    [Support] "KV Cache Memory Management" item 1."""
    return BLOCK_POSITIONS // ratio


def closing_entry(t: int, ratio: int, window: int):
    """Index of the entry whose window ends at raw position t, or None."""
    if t < window - 1 or (t - window + 1) % ratio:
        return None
    return (t - window + 1) // ratio


# ============================================================ compressor


def gated_window_sum(kv_win, gate_win, bias) -> np.ndarray:
    """Weighted sum of the window's raw rows, weights = per-channel softmax over offsets.

    kv_win, gate_win, bias: [window, D].  Row j is the token at offset j of the
    window; bias[j] is the learned bias of offset j.
    [Support] "DeepSeek V4 Attention Architecture" (c4a / c128a bullets).
    """
    logits = np.asarray(gate_win, np.float64) + np.asarray(bias, np.float64)
    logits = logits - logits.max(axis=0, keepdims=True)
    e = np.exp(logits)
    weights = e / e.sum(axis=0, keepdims=True)
    return (weights * np.asarray(kv_win, np.float64)).sum(axis=0)


def compressed_entry(kv, gate, first_pos: int, i: int, ratio: int, window: int, bias,
                     gamma_c, eps: float, rope_dim: int, theta: float) -> np.ndarray:
    """Entry i: gated window sum -> RMSNorm -> RoPE at anchor ratio*i.

    kv, gate: raw rows [n, D] for positions first_pos .. first_pos + n - 1.
    [部署] §3.2 first fusion (compressor, RMSNorm, RoPE, cache write).
    """
    lo, hi = window_span(i, ratio, window)
    if lo < first_pos or hi - first_pos >= len(kv):
        raise IndexError(f"entry {i} needs raw rows {lo}..{hi}")
    c = gated_window_sum(kv[lo - first_pos:hi - first_pos + 1],
                         gate[lo - first_pos:hi - first_pos + 1], bias)
    y = rms_norm(c, gamma_c, eps)
    return rope(y, lo, rope_dim, theta)



def complete_entries(kv, gate, ratio: int, window: int, bias, gamma_c, eps: float, rope_dim: int,
                     theta: float) -> np.ndarray:
    """Every entry whose window lies inside the raw rows kv, gate (positions 0 .. n-1):
    entries 0 .. (n - window) // ratio, each `compressed_entry`.  [D] rows, [0, D] if none.

    The indexer's keys are this at the indexer's dim with their own gate, bias and
    gain: [部署] §3.2 first fusion (compress, RMSNorm, RoPE and the write into the
    attention or the indexer K cache; the indexer K cache keeps its own kernel).
    """
    n = len(kv)
    m = (n - window) // ratio + 1 if n >= window else 0
    rows = [compressed_entry(kv, gate, 0, i, ratio, window, bias, gamma_c, eps, rope_dim, theta) for i in range(m)]
    return np.stack(rows) if rows else np.zeros((0, np.shape(kv)[1]))


def swa_row(kv_t, t: int, gamma_swa, eps: float, rope_dim: int, theta: float) -> np.ndarray:
    """Sliding-window row of raw token t: RMSNorm with its own gain, RoPE at t.
    [部署] §3.2 third fusion (KV RoPE + K insert for the uncompressed window)."""
    return rope(rms_norm(kv_t, gamma_swa, eps), t, rope_dim, theta)


def swa_positions(p: int, swa: int = 128):
    """Raw positions in the window of a query at p: [max(0, p - swa + 1), p]."""
    return range(max(0, p - swa + 1), p + 1)


# ============================================================ indexer and top-k


def indexer_scores(q_idx, w, k_idx) -> np.ndarray:
    """s_i = sum_h w_h * relu(q_idx_h . k_i).  q_idx [H_I, d_I], w [H_I], k_idx [n, d_I].
    [部署] §二 item 3 (DSA picks the top-k compressed tokens)."""
    dots = np.asarray(k_idx, np.float64) @ np.asarray(q_idx, np.float64).T  # [n, H_I]
    return np.maximum(dots, 0.0) @ np.asarray(w, np.float64)


def topk_select(scores, k: int) -> np.ndarray:
    """Indices of the min(k, n) largest scores; equal scores go to the lower index.
    Returned in descending score order."""
    s = np.asarray(scores, np.float64)
    order = np.lexsort((np.arange(len(s)), -s))
    return order[: min(k, len(s))].astype(np.int64)


# ============================================================ attention


def attention(q, p: int, keys, scale: float, rope_dim: int, theta: float) -> np.ndarray:
    """Shared-K=V attention of one query row, then inverse RoPE at p.

    q: [H, D] (un-rotated); keys: [m, D], each row both key and value.
    o_h = softmax_j(RoPE(q_h, p) . K_j * scale) @ K, then RoPE^-1(o_h, p).
    [Support] "DeepSeek V4 Attention Architecture" (shared K/V, inverse RoPE).
    """
    qr = rope(q, p, rope_dim, theta)
    K = np.asarray(keys, np.float64)
    logits = (qr @ K.T) * scale
    logits = logits - logits.max(axis=1, keepdims=True)
    e = np.exp(logits)
    a = e / e.sum(axis=1, keepdims=True)
    return rope(a @ K, p, rope_dim, theta, inverse=True)


def attention_partial(q, p: int, keys, scale: float, rope_dim: int, theta: float):
    """Un-normalised pieces of `attention` over a subset of keys, before inverse RoPE:
    (row max m [H], sum l [H], weighted sum acc [H, D]); used to state the merge rule."""
    qr = rope(q, p, rope_dim, theta)
    K = np.asarray(keys, np.float64)
    logits = (qr @ K.T) * scale
    m = logits.max(axis=1)
    e = np.exp(logits - m[:, None])
    return m, e.sum(axis=1), e @ K


def merge_partials(parts, p: int, rope_dim: int, theta: float) -> np.ndarray:
    """Combine partial softmaxes over disjoint key sets into the joint result."""
    m = np.max(np.stack([pt[0] for pt in parts]), axis=0)
    l = sum(pt[1] * np.exp(pt[0] - m) for pt in parts)
    acc = sum(pt[2] * np.exp(pt[0] - m)[:, None] for pt in parts)
    return rope(acc / l[:, None], p, rope_dim, theta, inverse=True)


# ============================================================ e4m3 codec


def e4m3_value(code: int) -> float:
    """Value of an e4m3 (fn) byte: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;
    exponent 0 is subnormal; S.1111.111 is NaN; no infinities."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def round_e4m3(x) -> np.ndarray:
    """Round to the nearest e4m3 value, ties to even, saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)  # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)  # binade exponent, clamped to the subnormal binade
    step = np.ldexp(1.0, e - 3)
    r = np.minimum(np.rint(a / step) * step, E4M3_MAX)
    return np.where(x < 0, -r, r)


def e4m3_encode(x) -> np.ndarray:
    """Bytes of round_e4m3(x); the sign bit follows the sign of x (so -0 stays -0)."""
    x = np.asarray(x, dtype=np.float64)
    r = np.abs(round_e4m3(x))
    _, ex = np.frexp(r)
    normal = r >= 2.0 ** -6
    e = np.where(normal, ex - 1, -6)
    mant = np.where(normal, r / np.ldexp(1.0, e) - 1.0, r / 2.0 ** -9)  # normal: fraction; subnormal: integer
    m = np.where(normal, mant * 8.0, mant).astype(np.int64)
    code = np.where(normal, ((e + 7) << 3) | m, m)
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.int64)]


def quantize_rows_e4m3(x):
    """Per-row e4m3 with an fp32 scale: scale = amax/448, code = e4m3(x * (448/amax)).
    All arithmetic in fp32 (the rounding decisions are the kernel's).  An all-zero
    row gets scale 0 and zero codes.  Returns (codes uint8 [n, D], scale fp32 [n])."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, np.float32(E4M3_MAX) / amax, np.float32(0)).astype(np.float32)
    y = (x * inv[..., None]).astype(np.float32)
    return e4m3_encode(y), scale


def dequantize_rows_e4m3(codes, scale) -> np.ndarray:
    return e4m3_decode(codes) * np.asarray(scale, np.float64)[..., None]


def round_bf16(x) -> np.ndarray:
    """Round to the nearest bfloat16 value (8 significant bits, fp32's exponent
    range), ties to even."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)  # a = f * 2^ex, f in [0.5, 1)
    step = np.ldexp(1.0, np.maximum(ex, -125) - 8)
    r = np.rint(a / step) * step
    return np.where(x < 0, -r, r)


def quantize_rows_e4m3_rope_bf16(x, rope_dim: int):
    """The decode cache's "partial token-wise fp8" ([部署] §二: the same
    attention kernel reads a bf16 cache in prefill and a partial token-wise fp8
    cache in decode).  Reading: per row (token-wise), the non-rotary dims
    [0, D-r) as e4m3 with one fp32 scale = their amax / 448 (the e4m3 row codec
    above on those dims alone); the r rotary dims kept in bf16.  Rounding
    decisions in fp32, as the kernels take them.
    Returns (codes uint8 [n, D-r], scale fp32 [n], rope fp64 [n, r] holding bf16 values)."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    codes, scale = quantize_rows_e4m3(x[..., : d - rope_dim])
    return codes, scale, round_bf16(x[..., d - rope_dim:])


def dequantize_rows_e4m3_rope_bf16(codes, scale, rope) -> np.ndarray:
    return np.concatenate([dequantize_rows_e4m3(codes, scale), np.asarray(rope, np.float64)], axis=-1)


# ============================================================ e2m1 (fp4) codec

# e2m1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is subnormal.
E2M1_TABLE = np.array([((-1.0) ** (c >> 3)) * ((c & 1) * 0.5 if ((c >> 1) & 3) == 0
                                               else (1.0 + (c & 1) / 2.0) * 2.0 ** (((c >> 1) & 3) - 1))
                       for c in range(16)], dtype=np.float64)


def round_e2m1(x) -> np.ndarray:
    """Round to the nearest e2m1 value (0, .5, 1, 1.5, 2, 3, 4, 6), ties to even, saturating at 6."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.minimum(np.rint(a / step) * step, E2M1_MAX)
    return np.where(x < 0, -r, r)


def e2m1_encode(x) -> np.ndarray:
    r = round_e2m1(x)
    mag = np.searchsorted(E2M1_TABLE[:8], np.abs(r))
    return (mag | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def quantize_nvfp4(x):
    """e2m1 codes with one e4m3 scale per 16 elements along the last axis.

    scale = e4m3(amax16 / 6); a zero scale gives zero codes; code = e2m1(x / scale).
    The division and both roundings are fp32, as in the kernel.  Codes are
    packed two per byte, element 2j in the low nibble.
    Returns (packed uint8 [..., d/2], scale bytes uint8 [..., d/16])."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    g = x.reshape(*x.shape[:-1], d // NVFP4_GROUP, NVFP4_GROUP)
    amax = np.max(np.abs(g), axis=-1)
    s_val = round_e4m3((amax / np.float32(E2M1_MAX)).astype(np.float32)).astype(np.float32)
    s_code = e4m3_encode(s_val)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(s_val[..., None] > 0, (g / s_val[..., None]).astype(np.float32), np.float32(0))
    codes = e2m1_encode(y).reshape(*x.shape[:-1], d)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed, s_code


def dequantize_nvfp4(packed, s_code) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    lo = E2M1_TABLE[packed & 0xF]
    hi = E2M1_TABLE[packed >> 4]
    vals = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.float64)
    vals[..., 0::2] = lo
    vals[..., 1::2] = hi
    d = vals.shape[-1]
    g = vals.reshape(*vals.shape[:-1], d // NVFP4_GROUP, NVFP4_GROUP)
    return (g * e4m3_decode(s_code)[..., None]).reshape(vals.shape)


# ============================================================ KV-size arithmetic


def kv_bytes_per_sequence(context: int, c4a_layers: int, c128a_layers: int, dim: int,
                          idx_dim: int, entry_bytes: float, idx_entry_bytes: float,
                          swa_layers: int = 0, swa: int = 128, swa_row_bytes: float = 0.0) -> float:
    """Cache bytes one sequence holds at `context` tokens.

    c4a layers keep every entry (main + indexer key); c128a layers keep main
    entries only; optional sliding-window rows per layer.
    [Support] "DeepSeek V4 Attention Architecture" (9.62 GiB at 1M).
    """
    n4 = context // 4
    n128 = context // 128
    total = c4a_layers * n4 * (entry_bytes + idx_entry_bytes) + c128a_layers * n128 * entry_bytes
    return total + swa_layers * swa * swa_row_bytes
