"""GPU parity of dg_k_grouped_fp8_wgrad against the float64 oracle.

Operands are drawn by the seeded generators and quantised by the oracle, so the
GPU and the oracle see the same bytes.  FP32 output must satisfy
|D_gpu - D| <= 1e-5 * S + 1e-6 element-wise (S = sum |a b s|); BF16 output
2^-7 |D| + 1e-5 * S + 1e-6; empty experts under in-place accumulation must be
bit-identical to C; integer-valued problems must be bit-exact.
"""
import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import workloads
import oracle
from tests.gpu_helpers import fp8_operands, run_fp8, assert_close, DEV

pytestmark = pytest.mark.gpu


def _case(ks, M, N, seed, gran_k=128, scale_noise=False):
    sk = sum(ks)
    A = workloads.randn((sk, M), seed).numpy()
    B = workloads.randn((sk, N), seed + 1).numpy()
    qa, sa, qb, sb = fp8_operands(A, B, gran_k)
    if scale_noise:            # distinct per-row/column scales exercise the scale layout
        rng = np.random.default_rng(seed)
        sa = (sa.astype(np.int64) + rng.integers(-6, 7, sa.shape)).astype(np.uint8)
        sb = (sb.astype(np.int64) + rng.integers(-6, 7, sb.shape)).astype(np.uint8)
    return qa, sa, qb, sb


def test_tiny_workload_inplace():
    w = workloads.WORKLOADS["fp8_tiny_g4"]
    ks, A, B, C = workloads.draw_operands("fp8_tiny_g4")
    qa, sa, qb, sb = fp8_operands(A.numpy(), B.numpy())
    d = run_fp8(qa, sa, qb, sb, ks, c=C.numpy(), c_mode="inplace")
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128, C.numpy())
    assert_close(d, D, S, what=w.name)
    assert torch.equal(d[1].cpu(), C[1])       # K = 0 expert: untouched, bitwise


@pytest.mark.parametrize("gran_k", [128, 32])
@pytest.mark.parametrize("out,c_mode", [("f32", "none"), ("f32", "inplace"),
                                        ("f32", "separate"), ("bf16", "none")])
def test_modes_two_ntiles(gran_k, out, c_mode):
    ks = [256, 0, 384, 128]
    M, N = 256, 448                     # N = 2 x 224
    qa, sa, qb, sb = _case(ks, M, N, 11, gran_k, scale_noise=True)
    C = workloads.randn((len(ks), M, N), 99).numpy()
    d = run_fp8(qa, sa, qb, sb, ks, gran_k, out, C if c_mode != "none" else None, c_mode)
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, gran_k,
                                     C if c_mode != "none" else None)
    assert_close(d, D, S, out, what=f"{out}/{c_mode}/g{gran_k}")
    if c_mode == "inplace":
        assert torch.equal(d[1].cpu(), torch.from_numpy(C[1]))


@pytest.mark.parametrize("M,N", [(144, 240), (16, 16), (272, 7168 // 8), (128, 224 * 3 + 16)])
def test_ragged_shapes(M, N):
    ks = [128, 256, 0, 128]
    qa, sa, qb, sb = _case(ks, M, N, M + N)
    d = run_fp8(qa, sa, qb, sb, ks)
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    assert_close(d, D, S, what=f"{M}x{N}")


def test_long_expert_many_stages():
    ks = [128 * 40, 128]
    qa, sa, qb, sb = _case(ks, 128, 224, 5, scale_noise=True)
    d = run_fp8(qa, sa, qb, sb, ks)
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    assert_close(d, D, S, what="long")


@pytest.mark.parametrize("gran_k", [128, 32])
def test_lanes_and_rotated_k_loops(gran_k):
    """Several tiles per CTA pair: long experts (82, 41 k-blocks) are split into
    lane chunks interleaved with short and output-only tiles, and their k loops
    are rotated; every expert checked on sampled rows x all N."""
    ks = [128 * 82, 128 * 41, 128 * 13, 0, 128 * 2, 128]
    M, N = 2048, 1792
    qa, sa, qb, sb = _case(ks, M, N, 21, gran_k, scale_noise=True)
    d = run_fp8(qa, sa, qb, sb, ks, gran_k)
    rows = np.sort(np.random.default_rng(21).choice(M, 24, replace=False))
    part = oracle.kgrouped_fp8_wgrad_rows(qa, sa, qb, sb, ks, rows, gran_k)
    dr = d[:, torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    for e, (De, Se) in part.items():
        assert_close(dr[e], De, Se, what=f"lanes expert {e}")
    assert torch.count_nonzero(d[3]).item() == 0


def test_integer_valued_is_bit_exact():
    """E4M3 integers in [-8, 8] with unit scales: every partial sum is an
    integer below 2^24, so the FP32 result is exact."""
    rng = np.random.default_rng(1)
    ks, M, N = [256, 128, 0, 384], 128, 448
    sk = sum(ks)
    vals = rng.integers(-8, 9, size=(sk, M)).astype(np.float64)
    valsb = rng.integers(-8, 9, size=(sk, N)).astype(np.float64)
    qa = oracle.e4m3_encode(vals)
    qb = oracle.e4m3_encode(valsb)
    sa = np.full((sk // 128, M), 127, np.uint8)
    sb = np.full((sk // 128, N), 127, np.uint8)
    d = run_fp8(qa, sa, qb, sb, ks).cpu().numpy()
    D, _ = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    assert np.array_equal(d.astype(np.float64), D)


def test_deterministic_rerun():
    ks = [512, 128, 0, 256]
    qa, sa, qb, sb = _case(ks, 256, 448, 21)
    d1 = run_fp8(qa, sa, qb, sb, ks)
    d2 = run_fp8(qa, sa, qb, sb, ks)
    assert torch.equal(d1, d2)


def test_all_experts_empty():
    ks, M, N = [0, 0, 0], 128, 224
    qa = np.zeros((0, M), np.uint8)
    qb = np.zeros((0, N), np.uint8)
    sa = np.zeros((0, M), np.uint8)
    sb = np.zeros((0, N), np.uint8)
    C = workloads.randn((3, M, N), 4).numpy()
    ks_dev = torch.tensor(ks, dtype=torch.int32, device=DEV)
    e = torch.empty(0, device=DEV, dtype=torch.uint8)
    d = torch.full((3, M, N), float("nan"), device=DEV)
    dg.dg_k_grouped_fp8_wgrad(e.view(0, M), e.view(0, M), e.view(0, N), e.view(0, N), d, None,
                              ks, ks_dev, 128)
    dg.dg_sync_check()
    assert torch.count_nonzero(d).item() == 0
    d2 = torch.from_numpy(C).to(DEV)
    dg.dg_k_grouped_fp8_wgrad(e.view(0, M), e.view(0, M), e.view(0, N), e.view(0, N), d2, d2,
                              ks, ks_dev, 128)
    dg.dg_sync_check()
    assert torch.equal(d2.cpu(), torch.from_numpy(C))
    sep = torch.from_numpy(C).to(DEV)
    d3 = torch.full((3, M, N), float("nan"), device=DEV)
    dg.dg_k_grouped_fp8_wgrad(e.view(0, M), e.view(0, M), e.view(0, N), e.view(0, N), d3, sep,
                              ks, ks_dev, 128)
    dg.dg_sync_check()
    assert torch.equal(d3.cpu(), torch.from_numpy(C))


def test_ks_dev_mismatch_is_reported():
    ks = [128, 256]
    qa, sa, qb, sb = _case(ks, 128, 224, 2)
    ks_dev = torch.tensor([256, 128], dtype=torch.int32, device=DEV)
    d = torch.empty(2, 128, 224, device=DEV)
    dg.dg_k_grouped_fp8_wgrad(torch.from_numpy(qa).to(DEV), torch.from_numpy(sa).to(DEV),
                              torch.from_numpy(qb).to(DEV), torch.from_numpy(sb).to(DEV),
                              d, None, ks, ks_dev, 128)
    with pytest.raises(dg.DGError) as ei:
        dg.dg_sync_check()
    assert ei.value.status == dg.DG_ERR_INVALID_ARG
    dg.dg_sync_check()                      # the status word was cleared


def _full_size_sampled(name, out):
    """Full-size workload in the bench's launch configuration; every expert
    checked on 48 seeded rows x all N, plus the smallest non-empty expert in full."""
    w = workloads.WORKLOADS[name]
    ks, A, B, _ = workloads.draw_operands(name)
    qa, sa, qb, sb = fp8_operands(A.numpy(), B.numpy())
    del A, B
    d = run_fp8(qa, sa, qb, sb, ks, 128, out)
    rng = np.random.default_rng(w.seed)
    rows = np.sort(rng.choice(w.M, 48, replace=False))
    part = oracle.kgrouped_fp8_wgrad_rows(qa, sa, qb, sb, ks, rows, 128)
    dr = d[:, torch.from_numpy(rows).to(DEV)].float().cpu().double().numpy()
    for e, (De, Se) in part.items():
        assert_close(dr[e], De, Se, out, what=f"{name} expert {e}")
    small = min((k, e) for e, k in enumerate(ks) if k > 0)[1]
    full = oracle.kgrouped_fp8_wgrad_rows(qa, sa, qb, sb, ks, np.arange(w.M), 128,
                                          experts=[small])
    assert_close(d[small].float().cpu().double().numpy(), *full[small], out,
                 what=f"{name} expert {small} full")
    for e, k in enumerate(ks):
        if k == 0:
            assert torch.count_nonzero(d[e]).item() == 0


@pytest.mark.slow
def test_full_size_upgate_sampled():
    _full_size_sampled("moe_upgate_fp8_g32", "f32")


@pytest.mark.slow
def test_full_size_down_bf16_sampled():
    _full_size_sampled("moe_down_fp8_g32", "bf16")


@pytest.mark.parametrize("gran_k", [128, 32])
@pytest.mark.parametrize("out,c_mode", [("f32", "none"), ("f32", "inplace"),
                                        ("f32", "separate"), ("bf16", "none")])
def test_transposed_tiles_modes(gran_k, out, c_mode):
    """M a multiple of 224 and N not (the down-projection's orientation): the
    library computes D^T tiles and writes them transposed."""
    ks = [256, 0, 384, 128]
    M, N = 448, 272
    qa, sa, qb, sb = _case(ks, M, N, 13, gran_k, scale_noise=True)
    C = workloads.randn((len(ks), M, N), 98).numpy()
    d = run_fp8(qa, sa, qb, sb, ks, gran_k, out, C if c_mode != "none" else None, c_mode)
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, gran_k,
                                     C if c_mode != "none" else None)
    assert_close(d, D, S, out, what=f"transposed {out}/{c_mode}/g{gran_k}")
    if c_mode == "inplace":
        assert torch.equal(d[1].cpu(), torch.from_numpy(C[1]))
    if c_mode == "none":
        assert torch.count_nonzero(d[1]).item() == 0


@pytest.mark.parametrize("M,N", [(224, 16), (672, 2048 // 8), (224 * 5, 80)])
def test_transposed_tiles_shapes(M, N):
    ks = [128, 256, 0, 128]
    qa, sa, qb, sb = _case(ks, M, N, M + 3 * N)
    d = run_fp8(qa, sa, qb, sb, ks, 128, "bf16")
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    assert_close(d, D, S, "bf16", what=f"transposed {M}x{N}")


def test_transposed_tiles_lanes():
    """Long and short experts across several tiles per CTA pair, transposed."""
    ks = [128 * 60, 128 * 17, 0, 128 * 3, 128]
    M, N = 2240, 1024
    qa, sa, qb, sb = _case(ks, M, N, 23, 128, scale_noise=True)
    d = run_fp8(qa, sa, qb, sb, ks, 128, "bf16")
    rows = np.sort(np.random.default_rng(23).choice(M, 24, replace=False))
    part = oracle.kgrouped_fp8_wgrad_rows(qa, sa, qb, sb, ks, rows, 128)
    dr = d[:, torch.from_numpy(rows).to(DEV)].float().cpu().double().numpy()
    for e, (De, Se) in part.items():
        assert_close(dr[e], De, Se, "bf16", what=f"transposed lanes expert {e}")
    assert torch.count_nonzero(d[2]).item() == 0


@pytest.mark.parametrize("gran_k", [128, 32])
@pytest.mark.parametrize("M,N", [(256, 224), (448, 272)])
def test_inplace_long_expert_is_split(gran_k, M, N):
    """In place, one expert far longer than a CTA pair's share of the work (a
    one- or two-tile grid): it runs as several K parts that each add into D.
    (448 x 272 also takes the transposed tiles.)"""
    ks = [128 * 70, 128, 0, 128 * 3]
    qa, sa, qb, sb = _case(ks, M, N, 31, gran_k, scale_noise=True)
    C = workloads.randn((len(ks), M, N), 96).numpy()
    d = run_fp8(qa, sa, qb, sb, ks, gran_k, "f32", C, "inplace")
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, gran_k, C)
    assert_close(d, D, S, what=f"split {M}x{N} g{gran_k}")
    assert torch.equal(d[2].cpu(), torch.from_numpy(C[2]))
