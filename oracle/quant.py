"""Column-block FP8 quantiser (the transpose + cast step), float64 reference.

Test infrastructure only (see the package docstring).

What it computes
----------------
The weight gradient ``dw = dy^T x`` reduces over tokens, so the tokens are the
GEMM's K axis and every ``gran_k`` consecutive tokens of one column must share
one scale factor, applied after accumulation ("Is DeepGEMM directly applicable
to backward in training?", qijiaxing's comment of 26 Mar 2025; the DeepSeek-V3
workflow quoted by hxdtest on 4 May 2025: activations are read out, transposed
and re-quantised into 128x1 tiles).  So for a BF16/FP32 matrix ``x[T, C]``
(tokens x channels), for each token block ``kb`` and column ``c``:

    amax   = max_{k in block kb} |x[k, c]|
    e      = clamp(ceil(log2(amax / 448)), -127, 127)   (amax = 0 -> -127)
    sf     = e + 127                                     (UE8M0 byte, value 2^e)
    q[k,c] = E4M3_RNE(x[k, c] * 2^-e)

448 is the largest E4M3 magnitude, so ``|x * 2^-e| <= 448`` and the cast never
saturates.  ``gran_k`` is 128 (the 1x1x128 recipe) or 32, the two values the
API accepts (How to Use DeepGEMM Weight Gradient Kernels..., "FP8
Implementation Example": ``gran_k`` must be 32 or 128).

``ceil(log2(r))`` is taken exactly from ``frexp``: r = f * 2^p with f in
[0.5, 1), so ceil(log2 r) = p - 1 when f == 0.5 and p otherwise.

Layouts: ``q`` token-major ``[T, C]`` (what a TN weight-gradient GEMM reads) or
channel-major ``[C, T]`` (the physical transpose); ``sf`` is ``[T/gran_k, C]``.
"""
import numpy as np

from .e4m3 import E4M3_MAX, e4m3_encode

SCALE_EXP_MIN = -127
SCALE_EXP_MAX = 127


def scale_exponent(amax) -> np.ndarray:
    """Exact clamp(ceil(log2(amax / 448)), -127, 127); -127 for amax == 0."""
    amax = np.asarray(amax, dtype=np.float64)
    r = amax / E4M3_MAX
    f, p = np.frexp(r)
    e = np.where(f == 0.5, p - 1, p).astype(np.int64)
    e = np.where(amax == 0.0, SCALE_EXP_MIN, e)
    return np.clip(e, SCALE_EXP_MIN, SCALE_EXP_MAX)


def quant_colblock(x, gran_k: int = 128, layout: str = "token"):
    """Quantise ``x[T, C]`` (any float dtype; converted to float64 exactly).

    Returns ``(q, sf)``: ``q`` uint8 E4M3 codes, ``[T, C]`` for
    ``layout="token"`` or ``[C, T]`` for ``layout="channel"``; ``sf`` uint8
    UE8M0 bytes ``[T // gran_k, C]``.
    """
    if gran_k not in (32, 128):
        raise ValueError("gran_k must be 32 or 128")
    x = np.asarray(x, dtype=np.float64)
    T, C = x.shape
    if T % gran_k:
        raise ValueError("T must be a multiple of gran_k")
    nb = T // gran_k
    q = np.empty((T, C), dtype=np.uint8)
    sf = np.empty((nb, C), dtype=np.uint8)
    step = max(1, (1 << 22) // max(1, gran_k * C))      # blocks per chunk, bounds memory
    for b0 in range(0, nb, step):
        b1 = min(nb, b0 + step)
        xb = x[b0 * gran_k:b1 * gran_k].reshape(b1 - b0, gran_k, C)
        amax = np.abs(xb).max(axis=1)                    # [blocks, C]
        e = scale_exponent(amax)
        sf[b0:b1] = (e + 127).astype(np.uint8)
        y = np.ldexp(xb, -e[:, None, :])                 # exact power-of-two scaling
        q[b0 * gran_k:b1 * gran_k] = e4m3_encode(y).reshape(-1, C)
    if layout == "token":
        return q, sf
    if layout == "channel":
        return np.ascontiguousarray(q.T), sf
    raise ValueError("layout must be 'token' or 'channel'")


# --------------------------------------------------------------------------
# Re-quantisation of stored FP8 activations, and the MoE token layout.
#
# The forward pass stores activations as E4M3 in 1 x 128 tiles: one scale per
# token per 128 consecutive channels.  The weight gradient needs 128 x 1 tiles
# (one scale per channel per 128 tokens), so the backward pass reads the
# stored tensor back, dequantises it, and quantises it again by columns
# ("Is DeepGEMM directly applicable to backward in training?", hxdtest,
# 4 May 2025, quoting the DeepSeek-V3 workflow: read out, dequantise,
# transpose, re-quantise into 128x1 tiles; the same thread, 12 Mar 2025: the
# FP8 weight-gradient GEMM lets activations be stored in FP8 for the backward
# pass).  The weight-gradient kernels also want the MoE layout: tokens grouped
# by expert, each expert's slice padded to whole 128-token blocks (LyricZhao,
# 26 Feb 2025: casting fused with the MoE layout; NiuMa, 18 Mar 2025: the FP8
# weight-gradient input must be a multiple of 128 tokens).
#
# Readings where the pages are silent: the stored scales are UE8M0 bytes
# (powers of two, the SM100 scale format of "UE8M0 Format in DeepGEMM"),
# laid out [T, C / 128]; the forward cast uses the same scale rule as the
# column-block cast, applied along channels; padding rows are zeros.

ROW_TILE = 128


def quant_rowtile(x):
    """The forward pass's 1 x 128 cast of ``x[T, C]``: per token and per 128
    consecutive channels, the scale rule of ``quant_colblock``.  Returns
    ``(q [T, C] uint8, sf [T, C / 128] uint8)``.  A 1 x 128 tile of x is a
    128 x 1 block of x^T, so this is the column-block cast of the transpose."""
    x = np.asarray(x, dtype=np.float64)
    T, C = x.shape
    if C % ROW_TILE:
        raise ValueError("C must be a multiple of 128")
    qt, sft = quant_colblock(x.T, ROW_TILE)              # q^T [C, T], sf^T [C/128, T]
    return np.ascontiguousarray(qt.T), np.ascontiguousarray(sft.T)


def dequant_rowtile(q, sf):
    """x[t, c] = e4m3(q[t, c]) * 2^(sf[t, c // 128] - 127), exact in float64."""
    from .e4m3 import e4m3_decode, ue8m0_to_float
    q = np.asarray(q, dtype=np.uint8)
    sf = np.asarray(sf, dtype=np.uint8)
    T, C = q.shape
    if C % ROW_TILE or sf.shape != (T, C // ROW_TILE):
        raise ValueError("sf must be [T, C / 128]")
    return e4m3_decode(q) * np.repeat(ue8m0_to_float(sf), ROW_TILE, axis=1)


def requant_colblock(q, sf_row, gran_k: int = 128, layout: str = "token"):
    """Stored 1 x 128 FP8 tiles -> 128 x 1 (gran_k x 1) column-block FP8:
    dequantise exactly, then the column-block cast."""
    return quant_colblock(dequant_rowtile(q, sf_row), gran_k, layout)


def gather_rows(x, src_rows):
    """MoE layout: row i of the result is ``x[src_rows[i]]``, or a row of
    zeros where ``src_rows[i] == -1`` (an expert's padding)."""
    x = np.asarray(x)
    src = np.asarray(src_rows, dtype=np.int64)
    if src.ndim != 1 or np.any(src < -1) or np.any(src >= x.shape[0]):
        raise ValueError("src_rows entries must lie in [-1, rows of x)")
    out = np.zeros((src.shape[0],) + x.shape[1:], dtype=x.dtype)
    keep = src >= 0
    out[keep] = x[src[keep]]
    return out


def moe_layout_cast(x, src_rows, gran_k: int = 128, layout: str = "token", sf_row=None):
    """Column-block cast of the MoE-layout rows of x.  ``x`` is a float matrix
    (BF16 values), or, with ``sf_row`` given, stored E4M3 codes with 1 x 128
    scales (re-quantised).  Padding rows are zeros before the cast."""
    src = dequant_rowtile(x, sf_row) if sf_row is not None else np.asarray(x, dtype=np.float64)
    return quant_colblock(gather_rows(src, src_rows), gran_k, layout)


def moe_layout_plan(topk_idx, G: int, align: int = 128):
    """The MoE token layout from top-k routing ``topk_idx[T, topk]`` (expert of
    each (token, slot) pair, or -1 for an unused slot): expert e's slice holds
    its pairs in (token, slot) order, then ``-1`` padding rows up to a multiple
    of ``align``; slices follow in expert order.  Returns ``(ks, src_rows,
    pair_rows)``: padded rows per expert, the source token of each row and the
    pair index ``t * topk + j`` of each row (-1 on padding)."""
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, topk = idx.shape
    if np.any(idx < -1) or np.any(idx >= G):
        raise ValueError("routing entries must lie in [-1, G)")
    flat = idx.reshape(-1)                       # entry t * topk + j
    ks, pair = [], []
    for e in range(G):
        pairs = np.nonzero(flat == e)[0]             # increasing pair index
        pad = (-len(pairs)) % align
        ks.append(len(pairs) + pad)
        pair.append(np.concatenate([pairs, -np.ones(pad, dtype=np.int64)]))
    pair = np.concatenate(pair) if pair else np.zeros(0, dtype=np.int64)
    src = np.where(pair >= 0, pair // topk, -1)
    return np.array(ks, dtype=np.int64), src.astype(np.int64), pair.astype(np.int64)
