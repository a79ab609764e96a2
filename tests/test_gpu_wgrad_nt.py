"""GPU parity of dg_k_grouped_fp8_wgrad_nt (K-major operands a [M, sum_k],
b [N, sum_k]) against the float64 oracle, with the tolerances of the TN form
(FP32 |D_gpu - D| <= 1e-5 S + 1e-6; BF16 2^-7 |D| + 1e-5 S + 1e-6; empty
experts in place bit-identical; integer-valued problems bit-exact), and the
chain from the channel-major cast output."""
import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import workloads
import oracle
from tests.gpu_helpers import fp8_operands, assert_close, DEV

pytestmark = pytest.mark.gpu


def _case(ks, M, N, seed, gran_k=128, scale_noise=False):
    sk = sum(ks)
    A = workloads.randn((sk, M), seed).numpy()
    B = workloads.randn((sk, N), seed + 1).numpy()
    qa, sa, qb, sb = fp8_operands(A, B, gran_k)
    if scale_noise:
        rng = np.random.default_rng(seed)
        sa = (sa.astype(np.int64) + rng.integers(-6, 7, sa.shape)).astype(np.uint8)
        sb = (sb.astype(np.int64) + rng.integers(-6, 7, sb.shape)).astype(np.uint8)
    return qa, sa, qb, sb


def run_nt(qa, sa, qb, sb, ks, gran_k=128, out="f32", c=None, c_mode="none"):
    """The oracle's token-major operands, transposed to [M, sum_k] / [N, sum_k]."""
    G, M, N = len(ks), qa.shape[1], qb.shape[1]
    dt = torch.float32 if out == "f32" else torch.bfloat16
    at = torch.from_numpy(np.ascontiguousarray(qa.T)).to(DEV)
    bt = torch.from_numpy(np.ascontiguousarray(qb.T)).to(DEV)
    ks_dev = torch.tensor(ks, dtype=torch.int32, device=DEV)
    if c_mode == "inplace":
        d = torch.from_numpy(c).to(DEV).float().clone()
        cc = d
    elif c_mode == "separate":
        d = torch.full((G, M, N), float("nan"), dtype=dt, device=DEV)
        cc = torch.from_numpy(c).to(DEV).float()
    else:
        d = torch.full((G, M, N), float("nan"), dtype=dt, device=DEV)
        cc = None
    dg.dg_k_grouped_fp8_wgrad_nt(at, torch.from_numpy(sa).to(DEV), bt,
                                 torch.from_numpy(sb).to(DEV), d, cc, ks, ks_dev, gran_k)
    dg.dg_sync_check()
    return d


@pytest.mark.parametrize("gran_k", [128, 32])
@pytest.mark.parametrize("out,c_mode", [("f32", "none"), ("f32", "inplace"),
                                        ("f32", "separate"), ("bf16", "none")])
def test_nt_modes(gran_k, out, c_mode):
    ks = [256, 0, 384, 128]
    M, N = 256, 448
    qa, sa, qb, sb = _case(ks, M, N, 11, gran_k, scale_noise=True)
    C = workloads.randn((len(ks), M, N), 99).numpy()
    d = run_nt(qa, sa, qb, sb, ks, gran_k, out, C if c_mode != "none" else None, c_mode)
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, gran_k,
                                     C if c_mode != "none" else None)
    assert_close(d, D, S, out, what=f"nt {out}/{c_mode}/g{gran_k}")
    if c_mode == "inplace":
        assert torch.equal(d[1].cpu(), torch.from_numpy(C[1]))


@pytest.mark.parametrize("M,N", [(144, 240), (16, 16), (272, 896), (128, 224 * 3 + 16)])
def test_nt_ragged_shapes(M, N):
    ks = [128, 256, 0, 128]
    qa, sa, qb, sb = _case(ks, M, N, M + N)
    d = run_nt(qa, sa, qb, sb, ks)
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    assert_close(d, D, S, what=f"nt {M}x{N}")


@pytest.mark.parametrize("gran_k", [128, 32])
def test_nt_lanes_and_rotated_k_loops(gran_k):
    ks = [128 * 82, 128 * 41, 128 * 13, 0, 128 * 2, 128]
    M, N = 2048, 1792
    qa, sa, qb, sb = _case(ks, M, N, 21, gran_k, scale_noise=True)
    d = run_nt(qa, sa, qb, sb, ks, gran_k)
    rows = np.sort(np.random.default_rng(21).choice(M, 24, replace=False))
    part = oracle.kgrouped_fp8_wgrad_rows(qa, sa, qb, sb, ks, rows, gran_k)
    dr = d[:, torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    for e, (De, Se) in part.items():
        assert_close(dr[e], De, Se, what=f"nt lanes expert {e}")
    assert torch.count_nonzero(d[3]).item() == 0


def test_nt_integer_valued_is_bit_exact():
    rng = np.random.default_rng(1)
    ks, M, N = [256, 128, 0, 384], 128, 448
    sk = sum(ks)
    qa = oracle.e4m3_encode(rng.integers(-8, 9, size=(sk, M)).astype(np.float64))
    qb = oracle.e4m3_encode(rng.integers(-8, 9, size=(sk, N)).astype(np.float64))
    sa = np.full((sk // 128, M), 127, np.uint8)
    sb = np.full((sk // 128, N), 127, np.uint8)
    d = run_nt(qa, sa, qb, sb, ks).cpu().numpy()
    D, _ = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    assert np.array_equal(d.astype(np.float64), D)


def test_nt_from_channel_major_cast():
    """BF16 dY and X cast channel-major ([C, T] codes) feed the NT GEMM
    directly; the result matches the oracle on the oracle's own cast."""
    ks = [256, 128, 0, 384]
    T, M, N = sum(ks), 256, 448
    dy = workloads.randn((T, M), seed=41, dtype=torch.bfloat16)
    x = workloads.randn((T, N), seed=42, dtype=torch.bfloat16)
    qa = torch.empty(M, T, dtype=torch.uint8, device=DEV)
    sa = torch.empty(T // 128, M, dtype=torch.uint8, device=DEV)
    qb = torch.empty(N, T, dtype=torch.uint8, device=DEV)
    sb = torch.empty(T // 128, N, dtype=torch.uint8, device=DEV)
    dg.dg_quant_transpose_fp8(dy.to(DEV), qa, sa, "channel")
    dg.dg_quant_transpose_fp8(x.to(DEV), qb, sb, "channel")
    d = torch.full((len(ks), M, N), float("nan"), device=DEV)
    dg.dg_k_grouped_fp8_wgrad_nt(qa, sa, qb, sb, d, None, ks,
                                 torch.tensor(ks, dtype=torch.int32, device=DEV), 128)
    dg.dg_sync_check()
    ra, rsa = oracle.quant_colblock(dy.float().numpy(), 128)
    rb, rsb = oracle.quant_colblock(x.float().numpy(), 128)
    assert np.array_equal(qa.cpu().numpy(), ra.T) and np.array_equal(qb.cpu().numpy(), rb.T)
    D, S = oracle.kgrouped_fp8_wgrad(ra, rsa, rb, rsb, ks, 128)
    assert_close(d, D, S, what="channel-major cast -> NT GEMM")


@pytest.mark.slow
def test_nt_full_size_upgate_sampled():
    """The up/gate workload (G = 32, 4096 x 7168, sum K = 32768) with K-major
    operands; every expert on 48 seeded rows x all N."""
    name = "moe_upgate_fp8_g32"
    w = workloads.WORKLOADS[name]
    ks, A, B, _ = workloads.draw_operands(name)
    qa, sa, qb, sb = fp8_operands(A.numpy(), B.numpy())
    del A, B
    d = run_nt(qa, sa, qb, sb, ks)
    rows = np.sort(np.random.default_rng(w.seed).choice(w.M, 48, replace=False))
    part = oracle.kgrouped_fp8_wgrad_rows(qa, sa, qb, sb, ks, rows, 128)
    dr = d[:, torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    for e, (De, Se) in part.items():
        assert_close(dr[e], De, Se, what=f"nt {name} expert {e}")


@pytest.mark.parametrize("out,c_mode", [("f32", "none"), ("f32", "inplace"), ("bf16", "none")])
def test_nt_transposed_tiles(out, c_mode):
    """K-major operands with M a multiple of 224 and N not: transposed tiles."""
    ks = [256, 0, 384, 128]
    M, N = 448, 272
    qa, sa, qb, sb = _case(ks, M, N, 17, 128, scale_noise=True)
    C = workloads.randn((len(ks), M, N), 97).numpy()
    d = run_nt(qa, sa, qb, sb, ks, 128, out, C if c_mode != "none" else None, c_mode)
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128, C if c_mode != "none" else None)
    assert_close(d, D, S, out, what=f"nt transposed {out}/{c_mode}")


def test_nt_inplace_long_expert_is_split():
    ks = [128 * 70, 128, 0, 128 * 3]
    M, N = 256, 224
    qa, sa, qb, sb = _case(ks, M, N, 33, 128, scale_noise=True)
    C = workloads.randn((len(ks), M, N), 95).numpy()
    d = run_nt(qa, sa, qb, sb, ks, 128, "f32", C, "inplace")
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128, C)
    assert_close(d, D, S, what="nt split")
