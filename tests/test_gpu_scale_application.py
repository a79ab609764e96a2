"""Where the block scales are applied: inside the tensor-core MMA (the kernel's
block-scaled E4M3 instruction) or by the alternative that scale-less tensor
cores need, an FP32 rescale of each block's partial sum into an FP32
accumulator.  Both are measured here against the float64 oracle on the same
outlier-heavy operands (1 % of the values x100, as in the down-projection
workload).

fp32_rescale below is that alternative in its best case: each 128-token
block's sum of code products is exact (every product of two E4M3 values has
at most 8 significant bits and lies in [2^-18, 2^18), so 128 of them sum
exactly in float64) and is rounded once to FP32, multiplied by the block's two
power-of-two scales (exact) and added into the FP32 accumulator (one rounding
per block).  A real implementation also rounds inside each block.
"""
import numpy as np
import pytest
import torch

import oracle
from grouped_fp8_weight_gb300 import workloads
from oracle.e4m3 import e4m3_decode, e4m3_encode
from gpu_helpers import assert_close, fp8_operands, run_fp8


def fp32_rescale(qa, sa, qb, sb, ks, gran_k=128):
    """[G, M, N] float32 result of the per-block FP32 rescale (best case)."""
    av = e4m3_decode(np.asarray(qa))
    bv = e4m3_decode(np.asarray(qb))
    G, M, N = len(ks), av.shape[1], bv.shape[1]
    out = np.zeros((G, M, N), dtype=np.float32)
    off = 0
    for e, k in enumerate(ks):
        acc = np.zeros((M, N), dtype=np.float32)
        for kb in range(off // gran_k, (off + k) // gran_k):
            rows = slice(kb * gran_k, (kb + 1) * gran_k)
            part = (av[rows].T @ bv[rows]).astype(np.float32)   # exact sum, one rounding
            scale = (np.ldexp(1.0, sa[kb].astype(np.int64) - 127)[:, None] *
                     np.ldexp(1.0, sb[kb].astype(np.int64) - 127)[None, :]).astype(np.float32)
            acc = acc + part * scale                            # exact product, one rounding
        out[e] = acc
        off += k
    return out


def test_fp32_rescale_is_exact_on_small_integers():
    """Integer codes 0..8 under scale bytes 125..129: every partial sum and
    every accumulation is an exact FP32 value, so the emulation equals the
    oracle's float64 result; a dropped block or a transposed scale breaks it."""
    rng = np.random.default_rng(5)
    ks = [256, 0, 384]
    M, N = 16, 24
    sk = sum(ks)
    qa = e4m3_encode(rng.integers(-8, 9, size=(sk, M)).astype(np.float64))
    qb = e4m3_encode(rng.integers(-8, 9, size=(sk, N)).astype(np.float64))
    sa = rng.integers(125, 130, size=(sk // 128, M)).astype(np.uint8)
    sb = rng.integers(125, 130, size=(sk // 128, N)).astype(np.uint8)
    D, _ = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    got = fp32_rescale(qa, sa, qb, sb, ks).astype(np.float64)
    assert np.array_equal(got, D)


def _outlier_operands(sk, M, N, seed):
    a = workloads.randn((sk, M), seed).numpy()
    b = workloads.randn((sk, N), seed + 1).numpy()
    rng = np.random.default_rng(seed)
    a = np.where(rng.random(a.shape) < 0.01, a * 100.0, a)
    b = np.where(rng.random(b.shape) < 0.01, b * 100.0, b)
    return fp8_operands(a, b)


@pytest.mark.gpu
@pytest.mark.parametrize("N", [448, 1792])
def test_block_scaled_against_fp32_rescale(N):
    """The block-scaled kernel within the FP32 tolerance of the oracle, and its
    error beside the FP32-rescale alternative's on the same operands (long
    experts: up to 32 scale blocks accumulated)."""
    ks = [128 * 32, 128 * 16, 128 * 8, 128 * 4]
    M = 256
    qa, sa, qb, sb = _outlier_operands(sum(ks), M, N, 71 + N)
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    d = run_fp8(qa, sa, qb, sb, ks, 128).double().cpu().numpy()
    assert_close(d, D, S, what=f"block-scaled, N = {N}")
    r = fp32_rescale(qa, sa, qb, sb, ks).astype(np.float64)
    nz = S > 0
    e_blk = np.abs(d - D)[nz] / S[nz]
    e_res = np.abs(r - D)[nz] / S[nz]
    # the alternative's own first-order bound (one rounding per block sum and
    # one per accumulation, at most 32 blocks): a check of the emulation
    assert e_res.max() <= 2 * 32 * 2.0 ** -24
    print(f"\nscale application, N = {N}: max |D - D64| / S  block-scaled {e_blk.max():.3e}, "
          f"FP32 rescale {e_res.max():.3e}; rms  block-scaled {np.sqrt(np.mean(e_blk ** 2)):.3e}, "
          f"FP32 rescale {np.sqrt(np.mean(e_res ** 2)):.3e}")
