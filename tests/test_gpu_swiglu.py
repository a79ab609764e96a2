"""GPU parity of dg_swiglu_backward_quant_fp8 against the float64 oracle.

The kernel evaluates the SwiGLU backward in FP32 (expf for e^-|g|, the
hardware reciprocal, then explicitly rounded products), so its values differ
from the exact ones by a few FP32 ulp.  The bound used here follows the
operation count: expf is within 2 ulp (CUDA's documented bound), the
reciprocal within 1 ulp, each other operation within 1/2 ulp, which gives at
most 16 ulp of |da u s| (1 + |g (1 - s)|) for dg and 8 ulp of |du| and |a|;
the tests allow twice that, 2^-19 relative.  Where sigma(g) or a product falls into FP32's subnormal range the
error is absolute instead: a few units of 2^-149 in sigma, carried by the
factors that multiply it, so the bound adds 2^-146 |da u| (1 + |g|) for dg,
2^-146 |da g| and 2^-146 |g u| for du and a, and 2^-145 for a rounded
subnormal product.  A scale or code is
accepted when it is the one of some value within that bound (check_cast_bound);
everywhere else the comparison is exact."""
import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import workloads
import oracle
from gpu_helpers import assert_close, check_cast_bound

pytestmark = pytest.mark.gpu

REL = 2.0 ** -19
SUB = 2.0 ** -146
ABS = 2.0 ** -145


def _bounds(h, da):
    h = np.asarray(h, dtype=np.float64)
    da = np.asarray(da, dtype=np.float64)
    I = h.shape[1] // 2
    g, u = h[:, :I], h[:, I:]
    s = oracle.sigmoid(g)
    b_dg = (REL * np.abs(da * u * s) * (1 + np.abs(g * (1 - s)))
            + SUB * np.abs(da * u) * (1 + np.abs(g)) + ABS)
    b_du = REL * np.abs(da * g * s) + SUB * np.abs(da * g) + ABS
    b_a = REL * np.abs(g * s * u) + SUB * np.abs(g * u) + ABS
    return np.concatenate([b_dg, b_du], axis=1), b_a


def _run(h, da, gran_k, with_a=True):
    T, I2 = h.shape
    I = I2 // 2
    q = torch.empty(T, I2, dtype=torch.uint8, device="cuda")
    sf = torch.empty(T // gran_k, I2, dtype=torch.uint8, device="cuda")
    qa = torch.empty(T, I, dtype=torch.uint8, device="cuda") if with_a else None
    sfa = torch.empty(T // gran_k, I, dtype=torch.uint8, device="cuda") if with_a else None
    dg.dg_swiglu_backward_quant_fp8(h.cuda(), da.cuda(), q, sf, qa, sfa, gran_k)
    dg.dg_sync_check()
    return q, sf, qa, sfa


def _check(h, da, gran_k, with_a=True, max_ambiguous=1e-3):
    q, sf, qa, sfa = _run(h, da, gran_k, with_a)
    hf, df = h.float().numpy(), da.float().numpy()
    dh, a = oracle.swiglu_backward(hf, df)
    b_dh, b_a = _bounds(hf, df)
    check_cast_bound(q, sf, dh, b_dh, gran_k, "dh", max_ambiguous)
    if with_a:
        check_cast_bound(qa, sfa, a, b_a, gran_k, "a", max_ambiguous)


@pytest.mark.parametrize("gran_k", [128, 32])
@pytest.mark.parametrize("T,I", [(128, 128), (256, 2048 // 8), (384, 144), (512, 16), (128, 1040)])
def test_swiglu_random(T, I, gran_k):
    h = workloads.randn((T, 2 * I), seed=T + I, dtype=torch.bfloat16)
    da = workloads.randn((T, I), seed=T + I + 1, dtype=torch.bfloat16)
    _check(h, da, gran_k)


@pytest.mark.parametrize("T,I", [(160, 80), (32 * 37, 208)])
def test_swiglu_ragged_token_tiles(T, I):
    # gran_k 32: the last 128-token tile is partial (its rows past T arrive
    # as zeros) and I is not a multiple of the 64-channel tile
    h = workloads.randn((T, 2 * I), seed=T + 3 * I, dtype=torch.bfloat16)
    da = workloads.randn((T, I), seed=T + 3 * I + 1, dtype=torch.bfloat16)
    _check(h, da, 32)


def test_swiglu_without_activation_output():
    h = workloads.randn((256, 512), seed=5, dtype=torch.bfloat16)
    da = workloads.randn((256, 256), seed=6, dtype=torch.bfloat16)
    _check(h, da, 128, with_a=False)


@pytest.mark.parametrize("gran_k", [128, 32])
def test_swiglu_special_values(gran_k):
    """Both tails of the sigmoid, exact zeros, the zero of silu' (g near
    -2.3994), huge and tiny magnitudes that keep FP32 values finite."""
    T, I = 256, 64
    rng = np.random.default_rng(7)
    g = rng.standard_normal((T, I)).astype(np.float32) * 3
    u = rng.standard_normal((T, I)).astype(np.float32)
    d = rng.standard_normal((T, I)).astype(np.float32)
    g[:, 0] = 100.0
    g[:, 1] = -100.0
    g[:, 2] = 0.0
    u[:, 3] = 0.0
    d[:, 4] = 0.0
    g[:, 5] = np.linspace(-2.45, -2.35, T)          # silu' changes sign here
    g[:, 6] = 1e4
    g[:, 7] = -1e4
    u[:, 8] *= 1e15
    d[:, 8] *= 1e15                                 # |dg| up to ~1e31, finite
    u[:, 9] *= 1e-20
    d[:, 9] *= 1e-20                                # tiny products
    g[:, 10] = 89.0                                 # e^-g below FP32's normal range
    g[:, 11] = -89.0                                # e^-g above FP32's range: s = 0
    h = torch.from_numpy(np.concatenate([g, u], axis=1)).to(torch.bfloat16)
    da = torch.from_numpy(d).to(torch.bfloat16)
    # Columns 1, 7, 9 and 11 hold values in FP32's subnormal range on purpose,
    # where the bound is absolute and admits two codes far more often.
    _check(h, da, gran_k, max_ambiguous=0.05)


def test_swiglu_full_size_sampled():
    """The up/gate shape of the bench (T = 32768 tokens, I = 2048: dh is the
    [32768, 4096] A operand) in the bench's launch configuration; sampled
    token blocks checked against the oracle."""
    T, I = 32768, 2048
    gen = torch.Generator(device="cuda").manual_seed(12)
    h = torch.randn(T, 2 * I, generator=gen, device="cuda").to(torch.bfloat16)
    da = torch.randn(T, I, generator=gen, device="cuda").to(torch.bfloat16)
    q = torch.empty(T, 2 * I, dtype=torch.uint8, device="cuda")
    sf = torch.empty(T // 128, 2 * I, dtype=torch.uint8, device="cuda")
    qa = torch.empty(T, I, dtype=torch.uint8, device="cuda")
    sfa = torch.empty(T // 128, I, dtype=torch.uint8, device="cuda")
    dg.dg_swiglu_backward_quant_fp8(h, da, q, sf, qa, sfa)
    dg.dg_sync_check()
    for kb in [0, 77, 255]:
        rows = slice(kb * 128, (kb + 1) * 128)
        hf, df = h[rows].float().cpu().numpy(), da[rows].float().cpu().numpy()
        dh, a = oracle.swiglu_backward(hf, df)
        b_dh, b_a = _bounds(hf, df)
        check_cast_bound(q[rows], sf[kb:kb + 1], dh, b_dh, 128, f"dh block {kb}")
        check_cast_bound(qa[rows], sfa[kb:kb + 1], a, b_a, 128, f"a block {kb}")


def test_swiglu_feeds_the_weight_gradient():
    """dh cast by the kernel as the up/gate A operand, X cast as B: the FP8
    GEMM on them against the oracle's GEMM on the same operands."""
    ks = [256, 0, 128, 384]
    T, I, N = sum(ks), 128, 256
    h = workloads.randn((T, 2 * I), seed=31, dtype=torch.bfloat16)
    da = workloads.randn((T, I), seed=32, dtype=torch.bfloat16)
    x = workloads.randn((T, N), seed=33, dtype=torch.bfloat16)
    q, sf, _, _ = _run(h, da, 128, with_a=False)
    qb = torch.empty(T, N, dtype=torch.uint8, device="cuda")
    sb = torch.empty(T // 128, N, dtype=torch.uint8, device="cuda")
    dg.dg_quant_transpose_fp8(x.cuda(), qb, sb)
    d = torch.full((len(ks), 2 * I, N), float("nan"), device="cuda")
    dg.dg_k_grouped_fp8_wgrad(q, sf, qb, sb, d, None, ks,
                              torch.tensor(ks, dtype=torch.int32, device="cuda"), 128)
    dg.dg_sync_check()
    D, S = oracle.kgrouped_fp8_wgrad(q.cpu().numpy(), sf.cpu().numpy(), qb.cpu().numpy(),
                                     sb.cpu().numpy(), ks, 128)
    assert_close(d, D, S, "f32", "SwiGLU cast -> GEMM")
