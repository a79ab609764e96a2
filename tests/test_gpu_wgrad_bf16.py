"""GPU parity of dg_k_grouped_bf16_wgrad (BF16 operands, arbitrary per-expert
token counts) against the float64 oracle."""
import numpy as np
import pytest
import torch

from grouped_fp8_weight_gb300 import workloads
import oracle
from tests.gpu_helpers import run_bf16, assert_close

pytestmark = pytest.mark.gpu


def _ops(ks, M, N, seed):
    sk = sum(ks)
    a = workloads.randn((sk, M), seed, torch.bfloat16)
    b = workloads.randn((sk, N), seed + 1, torch.bfloat16)
    return a, b


@pytest.mark.parametrize("ks", [[5, 0, 77, 130, 1], [64, 64], [1], [200, 0, 0, 63]])
@pytest.mark.parametrize("out,c_mode", [("f32", "none"), ("f32", "inplace"),
                                        ("f32", "separate"), ("bf16", "none")])
def test_unaligned_counts(ks, out, c_mode):
    M, N = 256, 512
    a, b = _ops(ks, M, N, len(ks) + sum(ks))
    C = workloads.randn((len(ks), M, N), 7, std=0.1).numpy()
    cc = C if c_mode != "none" else None
    d = run_bf16(a, b, ks, out, cc, c_mode)
    D, S = oracle.kgrouped_bf16_wgrad(a.float().numpy(), b.float().numpy(), ks, cc)
    assert_close(d, D, S, out, what=f"{ks}/{out}/{c_mode}")


@pytest.mark.parametrize("M,N", [(136, 264), (8, 8), (1024, 1024), (128, 128)])
def test_ragged_shapes(M, N):
    ks = [100, 0, 29, 300]
    a, b = _ops(ks, M, N, M * 3 + N)
    d = run_bf16(a, b, ks)
    D, S = oracle.kgrouped_bf16_wgrad(a.float().numpy(), b.float().numpy(), ks)
    assert_close(d, D, S, what=f"{M}x{N}")


def test_tail_masking_ignores_next_expert():
    """Expert 0 ends mid-stage; expert 1's rows hold huge values that must
    not leak into expert 0."""
    ks = [70, 58]
    M = N = 128
    a, b = _ops(ks, M, N, 3)
    a[70:] = 1e4
    b[70:] = -1e4
    d = run_bf16(a, b, ks)
    D, S = oracle.kgrouped_bf16_wgrad(a.float().numpy(), b.float().numpy(), ks)
    assert_close(d, D, S, what="tail")


def test_fine_grained_workload_full():
    """The fine-grained BF16 workload at full size (256 experts, token-level
    counts, ~30% empty, accumulated in place); every expert on 32 seeded rows,
    plus three experts in full."""
    w = workloads.WORKLOADS["bf16_fine_g256"]
    ks, A, B, C = workloads.draw_operands(w.name)
    d = run_bf16(A, B, ks, "f32", C.numpy(), "inplace")
    a32, b32 = A.float().numpy(), B.float().numpy()
    rows = np.sort(np.random.default_rng(3).choice(w.M, 32, replace=False))
    part = oracle.kgrouped_bf16_wgrad_rows(a32, b32, ks, rows, C.numpy())
    dr = d[:, torch.from_numpy(rows).cuda()].cpu().double().numpy()
    for e, (De, Se) in part.items():
        assert_close(dr[e], De, Se, what=f"expert {e}")
    nz = [e for e, k in enumerate(ks) if k > 0]
    for e in [nz[0], nz[len(nz) // 2], nz[-1]]:
        full = oracle.kgrouped_bf16_wgrad_rows(a32, b32, ks, np.arange(w.M), C.numpy(), [e])
        assert_close(d[e].cpu().double().numpy(), *full[e], what=f"expert {e} full")
    for e, k in enumerate(ks):
        if k == 0:
            assert torch.equal(d[e].cpu(), C[e])


def test_inplace_long_expert_is_split():
    """In place on a one-tile grid, an expert of 5000 tokens (78 full stages of
    64 and a tail of 8) runs as several K parts, the last one with the tail."""
    ks = [5000, 3, 0, 130]
    M = N = 256
    a, b = _ops(ks, M, N, 41)
    C = workloads.randn((len(ks), M, N), 8, std=0.1).numpy()
    d = run_bf16(a, b, ks, "f32", C, "inplace")
    D, S = oracle.kgrouped_bf16_wgrad(a.float().numpy(), b.float().numpy(), ks, C)
    assert_close(d, D, S, what="bf16 split")
    assert torch.equal(d[2].cpu(), torch.from_numpy(C[2]))
