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
