"""GPU parity with more schedule entries than the kernel keeps in shared memory
(256 entries, 223 for K-major operands): the schedule is then read from the
kernel parameters.  Covers the TN and NT FP8 weight gradients (with output-only
entries for empty experts), the BF16 weight gradient and the M-grouped data
gradient, each against the float64 oracle with the usual tolerances."""
import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import workloads
import oracle
from tests.gpu_helpers import fp8_operands, run_fp8, run_bf16, assert_close, DEV

pytestmark = pytest.mark.gpu


def _ks(G, live, unit, seed):
    rng = np.random.default_rng(seed)
    ks = [0] * G
    for e in rng.choice(G, size=live, replace=False):
        ks[int(e)] = unit * int(rng.integers(1, 3))
    return ks


def test_fp8_tn_schedule_from_parameters():
    ks = _ks(300, 220, 128, 1)                 # 220 GEMM entries + 80 output-only = 300
    M, N = 128, 224
    A = workloads.randn((sum(ks), M), 71).numpy()
    B = workloads.randn((sum(ks), N), 72).numpy()
    qa, sa, qb, sb = fp8_operands(A, B, 128)
    d = run_fp8(qa, sa, qb, sb, ks)
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    assert_close(d, D, S, what="tn, 300 entries")


def test_fp8_nt_schedule_from_parameters():
    ks = _ks(240, 240, 128, 2)                 # above the K-major limit of 223
    M, N = 128, 224
    A = workloads.randn((sum(ks), M), 73).numpy()
    B = workloads.randn((sum(ks), N), 74).numpy()
    qa, sa, qb, sb = fp8_operands(A, B, 128)
    d = torch.full((len(ks), M, N), float("nan"), device=DEV)
    at = torch.from_numpy(np.ascontiguousarray(qa.T)).to(DEV)
    bt = torch.from_numpy(np.ascontiguousarray(qb.T)).to(DEV)
    dg.dg_k_grouped_fp8_wgrad_nt(at, torch.from_numpy(sa).to(DEV), bt, torch.from_numpy(sb).to(DEV),
                                 d, None, ks, torch.tensor(ks, dtype=torch.int32, device=DEV), 128)
    dg.dg_sync_check()
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    assert_close(d, D, S, what="nt, 240 entries")


def test_bf16_schedule_from_parameters():
    rng = np.random.default_rng(3)
    ks = [int(k) for k in rng.integers(0, 90, size=300)]
    M, N = 64, 128
    a = workloads.randn((sum(ks), M), 75, torch.bfloat16)
    b = workloads.randn((sum(ks), N), 76, torch.bfloat16)
    C = workloads.randn((len(ks), M, N), 77).numpy()
    d = run_bf16(a.to(DEV), b.to(DEV), ks, "f32", C, "inplace")
    D, S = oracle.kgrouped_bf16_wgrad(a.float().numpy(), b.float().numpy(), ks, C)
    assert_close(d, D, S, what="bf16, 300 experts in place")


def test_dgrad_schedule_from_parameters():
    ms = [128] * 280 + [0] * 20 + [256] * 4   # 284 entries with tokens
    K, N = 128, 224
    gen = torch.Generator().manual_seed(78)
    a = workloads.random_codes((sum(ms), K), gen).numpy()
    sfa = torch.randint(118, 138, (sum(ms), 1), generator=gen, dtype=torch.uint8).numpy()
    w = workloads.random_codes((len(ms), K, N), gen).numpy()
    sfw = torch.randint(110, 130, (len(ms), 1, N), generator=gen, dtype=torch.uint8).numpy()
    d = torch.full((sum(ms), N), float("nan"), dtype=torch.bfloat16, device=DEV)
    t = lambda x: torch.from_numpy(x).to(DEV)
    dg.dg_m_grouped_fp8_dgrad(t(a), t(sfa), t(w), t(sfw), d, ms,
                              torch.tensor(ms, dtype=torch.int32, device=DEV), 128)
    dg.dg_sync_check()
    D, S = oracle.mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, 128)
    assert_close(d, D, S, "bf16", what="dgrad, 284 entries")
