"""K-grouped weight-gradient GEMM, float64 reference.

Test infrastructure only (see the package docstring).

What it computes
----------------
Expert ``e`` owns the contiguous token slice ``[off_e, off_e + K_e)`` of the
token-concatenated operands ``A[sum K, M]`` (upstream gradients dy of the
expert's output, M = h_out) and ``B[sum K, N]`` (its input activations x,
N = h_in).  Its weight gradient is ``dw_e = dy_e^T x_e``, a GEMM with K = tokens
("Is DeepGEMM directly applicable to backward in training?", qijiaxing's
comment of 26 Mar 2025; How to Use DeepGEMM Weight Gradient Kernels for
Training Backward Passes, "FP8 Implementation Example": A is [sum(K_i), M], B is
[sum(K_i), N], one K slice per expert).  With FP8 operands every ``gran_k``-token
block of each column carries one power-of-two scale, applied to the block's
contribution (same comment: the scale is shared along k and applied after
accumulation):

    D[e, m, n] = Cterm[e, m, n]
               + sum_{k = off_e}^{off_e + K_e - 1}
                   fp8(A[k, m]) 2^(sfa[k // g, m] - 127) * fp8(B[k, n]) 2^(sfb[k // g, n] - 127)

with ``Cterm = C`` when an accumulator is given, else 0.  An expert with
K_e = 0 gets ``D[e] = Cterm[e]`` (zero-size groups are skipped: "Dispatch and
Tensor-Map Handling", "Integration Best Practices for MoE Training").  The BF16
variant ("BF16 Alternative") is the same sum without scales.

The sum is computed per expert as one float64 matrix product of the dequantised
slices (a library matmul used as a step).  Every product is exact in float64 (3
mantissa bits times 3 mantissa bits times a power of two, or 8 x 8 bits for
BF16), so the only rounding is float64 summation, about 1e-16 relative: the
result is exact for every comparison made against it.

Alongside D the oracle returns ``S[e, m, n] = sum_k |a b s|`` (the same sum of
absolute terms), from which the comparison tolerances are built:

    FP32 output:  |D_gpu - D| <= 1e-5 * S + 1e-6
    BF16 output:  |D_gpu - D| <= 2^-7 |D| + 1e-5 * S + 1e-6
"""
import numpy as np

from .e4m3 import e4m3_decode, ue8m0_to_float

FP32_REL = 1e-5
ABS = 1e-6
BF16_REL = 2.0 ** -7


def expert_offsets(ks):
    """off_e = sum_{j<e} K_j, as a list of length G + 1."""
    off = [0]
    for k in ks:
        if k < 0:
            raise ValueError("negative expert size")
        off.append(off[-1] + int(k))
    return off


def dequant_colblock(codes, sf, gran_k: int, rows=None):
    """fp8(codes[k, c]) * 2^(sf[k // gran_k, c] - 127) as float64.

    ``rows`` optionally selects a contiguous token range ``(k0, k1)``.
    """
    codes = np.asarray(codes)
    sf = np.asarray(sf)
    k0, k1 = (0, codes.shape[0]) if rows is None else rows
    v = e4m3_decode(codes[k0:k1])
    blk = np.arange(k0, k1) // gran_k
    return v * ue8m0_to_float(sf[blk])


def _check_ks(ks, sum_k):
    off = expert_offsets(ks)
    if off[-1] != sum_k:
        raise ValueError("sum of ks does not match the operands' row count")
    return off


def kgrouped_fp8_wgrad(a, sfa, b, sfb, ks, gran_k: int = 128, c=None):
    """Full ``(D, S)`` for the FP8 K-grouped weight gradient.

    a: uint8 E4M3 codes [sum_k, M]; sfa: uint8 UE8M0 [sum_k / gran_k, M];
    b, sfb likewise with N; ks: G expert sizes (multiples of gran_k);
    c: optional float array [G, M, N] (the accumulator).
    Returns float64 arrays D, S of shape [G, M, N].
    """
    a = np.asarray(a)
    b = np.asarray(b)
    G, M, N = len(ks), a.shape[1], b.shape[1]
    off = _check_ks(ks, a.shape[0])
    D = np.zeros((G, M, N)) if c is None else np.array(c, dtype=np.float64, copy=True)
    S = np.zeros((G, M, N))
    for e in range(G):
        if ks[e] == 0:
            continue
        if ks[e] % gran_k or off[e] % gran_k:
            raise ValueError("FP8 expert slices must be whole scale blocks")
        ad = dequant_colblock(a, sfa, gran_k, (off[e], off[e + 1]))
        bd = dequant_colblock(b, sfb, gran_k, (off[e], off[e + 1]))
        D[e] += ad.T @ bd
        S[e] = np.abs(ad).T @ np.abs(bd)
    return D, S


def kgrouped_fp8_wgrad_rows(a, sfa, b, sfb, ks, rows, gran_k: int = 128, c=None, experts=None):
    """Rows ``rows`` (indices into M) of D and S for the experts in
    ``experts`` (default: all).  Returns dict e -> (D_rows [R, N], S_rows)."""
    a = np.asarray(a)
    b = np.asarray(b)
    off = _check_ks(ks, a.shape[0])
    rows = np.asarray(rows)
    out = {}
    for e in (range(len(ks)) if experts is None else experts):
        base = np.zeros((len(rows), b.shape[1])) if c is None else \
            np.asarray(c[e])[rows].astype(np.float64)
        if ks[e] == 0:
            out[e] = (base, np.zeros_like(base))
            continue
        ad = dequant_colblock(a[:, rows], sfa[:, rows], gran_k, (off[e], off[e + 1]))
        bd = dequant_colblock(b, sfb, gran_k, (off[e], off[e + 1]))
        out[e] = (base + ad.T @ bd, np.abs(ad).T @ np.abs(bd))
    return out


def kgrouped_bf16_wgrad(a, b, ks, c=None):
    """Full ``(D, S)`` for the BF16-input variant: a [sum_k, M], b [sum_k, N]
    (any float dtype, read exactly as float64); ks arbitrary non-negative."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    G, M, N = len(ks), a.shape[1], b.shape[1]
    off = _check_ks(ks, a.shape[0])
    D = np.zeros((G, M, N)) if c is None else np.array(c, dtype=np.float64, copy=True)
    S = np.zeros((G, M, N))
    for e in range(G):
        if ks[e] == 0:
            continue
        ad = a[off[e]:off[e + 1]]
        bd = b[off[e]:off[e + 1]]
        D[e] += ad.T @ bd
        S[e] = np.abs(ad).T @ np.abs(bd)
    return D, S


def kgrouped_bf16_wgrad_rows(a, b, ks, rows, c=None, experts=None):
    """Sampled rows of the BF16 variant, as ``kgrouped_fp8_wgrad_rows``."""
    off = _check_ks(ks, a.shape[0])
    rows = np.asarray(rows)
    out = {}
    for e in (range(len(ks)) if experts is None else experts):
        base = np.zeros((len(rows), b.shape[1])) if c is None else \
            np.asarray(c[e])[rows].astype(np.float64)
        if ks[e] == 0:
            out[e] = (base, np.zeros_like(base))
            continue
        ad = np.asarray(a[off[e]:off[e + 1]][:, rows], dtype=np.float64)
        bd = np.asarray(b[off[e]:off[e + 1]], dtype=np.float64)
        out[e] = (base + ad.T @ bd, np.abs(ad).T @ np.abs(bd))
    return out


def fp32_bound(S):
    """Per-element tolerance for an FP32-output result."""
    return FP32_REL * np.asarray(S) + ABS


def bf16_bound(D, S):
    """Per-element tolerance for a BF16-output result."""
    return BF16_REL * np.abs(np.asarray(D)) + FP32_REL * np.asarray(S) + ABS
