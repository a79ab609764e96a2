"""M-grouped data-gradient GEMM (the other GEMM of a MoE expert's backward),
float64 reference.

Test infrastructure only (see the package docstring).

What it computes
----------------
A linear layer's backward is two GEMMs ("Is DeepGEMM directly applicable to
backward in training?", YouJiacheng's opening post of 26 Feb 2025): the weight
gradient (the K-grouped GEMM of ``wgrad``) and the data gradient, which the
library already ships (LyricZhao's reply of the same day).  For a MoE expert
``e`` with weight ``W_e [h_out, h_in]`` and the upstream gradients ``dy_e`` of
its tokens, the data gradient is ``dx_e = dy_e W_e``.  The experts' token rows
are contiguous (the padded MoE layout): expert ``e`` owns rows
``[off_e, off_e + M_e)`` of ``dy [sum_m, K]`` (K = h_out) and of
``dx [sum_m, N]`` (N = h_in), so the GEMM is grouped along M.

The pages print no scale recipe for this GEMM.  The reading taken: both
operands carry one power-of-two (UE8M0) scale per ``gran_k`` elements along
the contraction axis K -- dy one per token per ``gran_k`` channels (the 1 x 128
tile in which the forward pass stores activations), the weight one per column
per ``gran_k`` rows (a 128 x 128 block scale is this with each block's scale
repeated over its columns) -- which is the form the block-scaled tensor-core
MMA consumes ("UE8M0 Format in DeepGEMM": packed UE8M0 scales on SM100):

    D[t, n] = sum_{k < K} fp8(A[t, k]) 2^(sfa[t, k // g] - 127)
                          * fp8(W[e, k, n]) 2^(sfw[e, k // g, n] - 127)

for every row t of expert e.  Experts with M_e = 0 own no rows.  As in
``wgrad``, the sum is one float64 matrix product of the dequantised operands
per expert (a library matmul used as a step; every product is exact in
float64), and ``S = sum_k |a w s|`` is returned for the tolerances
(``wgrad.fp32_bound`` / ``wgrad.bf16_bound``).
"""
import numpy as np

from .e4m3 import e4m3_decode, ue8m0_to_float
from .wgrad import expert_offsets


def _check(ms, sum_m, K, gran_k):
    off = expert_offsets(ms)
    if off[-1] != sum_m:
        raise ValueError("sum of ms does not match the rows of a")
    if K % gran_k:
        raise ValueError("K must be whole scale blocks")
    return off


def dequant_rows(codes, sf, gran_k: int):
    """fp8(codes[t, k]) * 2^(sf[t, k // gran_k] - 127): scales along each row."""
    codes = np.asarray(codes)
    sf = np.asarray(sf)
    v = e4m3_decode(codes)
    blk = np.arange(codes.shape[1]) // gran_k
    return v * ue8m0_to_float(sf[:, blk])


def dequant_weight(codes, sf, gran_k: int):
    """fp8(W[k, n]) * 2^(sf[k // gran_k, n] - 127) for one expert's [K, N]."""
    codes = np.asarray(codes)
    sf = np.asarray(sf)
    v = e4m3_decode(codes)
    blk = np.arange(codes.shape[0]) // gran_k
    return v * ue8m0_to_float(sf[blk])


def mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, gran_k: int = 128):
    """Full ``(D, S)``, float64 ``[sum_m, N]``.

    a: uint8 E4M3 codes [sum_m, K]; sfa: uint8 UE8M0 [sum_m, K / gran_k];
    w: uint8 E4M3 [G, K, N]; sfw: uint8 UE8M0 [G, K / gran_k, N];
    ms: G token counts (any non-negative values here).
    """
    a = np.asarray(a)
    w = np.asarray(w)
    G, K, N = w.shape
    if len(ms) != G:
        raise ValueError("ms must have G entries")
    off = _check(ms, a.shape[0], K, gran_k)
    D = np.zeros((a.shape[0], N))
    S = np.zeros((a.shape[0], N))
    for e in range(G):
        if ms[e] == 0:
            continue
        r0, r1 = off[e], off[e + 1]
        ad = dequant_rows(a[r0:r1], sfa[r0:r1], gran_k)
        wd = dequant_weight(w[e], sfw[e], gran_k)
        D[r0:r1] = ad @ wd
        S[r0:r1] = np.abs(ad) @ np.abs(wd)
    return D, S


def mgrouped_fp8_dgrad_rows(a, sfa, w, sfw, ms, rows, gran_k: int = 128):
    """Rows ``rows`` (global token rows) of D and S: ``(D_rows, S_rows)``."""
    a = np.asarray(a)
    G, K, N = np.asarray(w).shape
    off = _check(ms, a.shape[0], K, gran_k)
    rows = np.asarray(rows, dtype=np.int64)
    owner = np.searchsorted(np.asarray(off[1:]), rows, side="right")
    D = np.zeros((len(rows), N))
    S = np.zeros((len(rows), N))
    for e in np.unique(owner):
        sel = np.nonzero(owner == e)[0]
        ad = dequant_rows(a[rows[sel]], np.asarray(sfa)[rows[sel]], gran_k)
        wd = dequant_weight(np.asarray(w[e]), np.asarray(sfw[e]), gran_k)
        D[sel] = ad @ wd
        S[sel] = np.abs(ad) @ np.abs(wd)
    return D, S
