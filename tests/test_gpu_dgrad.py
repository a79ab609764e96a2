"""GPU parity of dg_m_grouped_fp8_dgrad and dg_m_grouped_fp8_dgrad_nt (the
M-grouped FP8 data gradient dx_e = dy_e W_e, weights [G, K, N] or K-major
[G, N, K]) against the float64 oracle, with the weight gradient's
tolerances (FP32 |D_gpu - D| <= 1e-5 S + 1e-6; BF16 2^-7 |D| + 1e-5 S + 1e-6;
integer-valued problems bit-exact).  Cases span several tiles, ragged N
tiles, experts whose token count is an odd multiple of 128 (the second half
of their last 256-row chunk is not stored), empty experts, partial scale
groups along K, long k loops, and the full-size up/gate workload on
sampled rows."""
import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import workloads
import oracle
from tests.gpu_helpers import assert_close, DEV

pytestmark = pytest.mark.gpu


def _case(ms, K, N, seed, gran_k=128):
    gen = torch.Generator().manual_seed(seed)
    sm, G = sum(ms), len(ms)
    a = workloads.random_codes((sm, K), gen).numpy()
    sfa = torch.randint(118, 138, (sm, K // gran_k), generator=gen, dtype=torch.uint8).numpy()
    w = workloads.random_codes((G, K, N), gen).numpy()
    sfw = torch.randint(110, 130, (G, K // gran_k, N), generator=gen, dtype=torch.uint8).numpy()
    return a, sfa, w, sfw


def run_dgrad(a, sfa, w, sfw, ms, gran_k=128, out="bf16", w_kmajor=False):
    """w is the oracle's [G, K, N]; with w_kmajor it is passed as [G, N, K]
    to the K-major entry point."""
    dt = torch.float32 if out == "f32" else torch.bfloat16
    d = torch.full((a.shape[0], w.shape[2]), float("nan"), dtype=dt, device=DEV)
    ms_dev = torch.tensor(ms, dtype=torch.int32, device=DEV)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    if w_kmajor:
        dg.dg_m_grouped_fp8_dgrad_nt(t(a), t(sfa), t(np.swapaxes(w, 1, 2)), t(sfw), d, ms, ms_dev,
                                     gran_k)
    else:
        dg.dg_m_grouped_fp8_dgrad(t(a), t(sfa), t(w), t(sfw), d, ms, ms_dev, gran_k)
    dg.dg_sync_check()
    return d


@pytest.mark.parametrize("w_kmajor", [False, True])
@pytest.mark.parametrize("gran_k", [128, 32])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_dgrad_modes(gran_k, out, w_kmajor):
    ms, K, N = [256, 0, 384, 128], 512, 448
    a, sfa, w, sfw = _case(ms, K, N, 31, gran_k)
    d = run_dgrad(a, sfa, w, sfw, ms, gran_k, out, w_kmajor)
    D, S = oracle.mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, gran_k)
    assert_close(d, D, S, out, what=f"dgrad {out}/g{gran_k}/kmajor={w_kmajor}")


@pytest.mark.parametrize("w_kmajor", [False, True])
@pytest.mark.parametrize("K,N", [(128, 240), (384, 16), (640, 224 * 3 + 16), (1280, 96)])
def test_dgrad_ragged_shapes(K, N, w_kmajor):
    ms = [128, 384, 0, 256, 128]
    a, sfa, w, sfw = _case(ms, K, N, K + N)
    d = run_dgrad(a, sfa, w, sfw, ms, 128, "f32", w_kmajor)
    D, S = oracle.mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, 128)
    assert_close(d, D, S, "f32", what=f"dgrad K={K} N={N} kmajor={w_kmajor}")


@pytest.mark.parametrize("w_kmajor", [False, True])
@pytest.mark.parametrize("gran_k", [128, 32])
def test_dgrad_many_tiles_and_long_k_loops(gran_k, w_kmajor):
    """More tiles than CTA pairs (both lanes busy), 16-stage k loops, one
    expert of a single 128-row half."""
    ms, K, N = [128 * 21, 128 * 7, 0, 128 * 3, 128], 2048, 896
    a, sfa, w, sfw = _case(ms, K, N, 41, gran_k)
    d = run_dgrad(a, sfa, w, sfw, ms, gran_k, "bf16", w_kmajor)
    D, S = oracle.mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, gran_k)
    assert_close(d, D, S, "bf16", what=f"dgrad lanes g{gran_k} kmajor={w_kmajor}")


@pytest.mark.parametrize("w_kmajor", [False, True])
def test_dgrad_integer_valued_is_bit_exact(w_kmajor):
    """E4M3 integers in [-8, 8] with unit scales: every partial sum is an
    integer below 2^24, so the FP32 result is exact."""
    rng = np.random.default_rng(2)
    ms, K, N = [256, 128, 0, 384], 512, 448
    sm = sum(ms)
    a = oracle.e4m3_encode(rng.integers(-8, 9, size=(sm, K)).astype(np.float64))
    w = oracle.e4m3_encode(rng.integers(-8, 9, size=(len(ms), K, N)).astype(np.float64))
    sfa = np.full((sm, K // 128), 127, np.uint8)
    sfw = np.full((len(ms), K // 128, N), 127, np.uint8)
    d = run_dgrad(a, sfa, w, sfw, ms, 128, "f32", w_kmajor).cpu().numpy()
    D, _ = oracle.mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, 128)
    assert np.array_equal(d.astype(np.float64), D)


def test_dgrad_deterministic_rerun():
    ms = [384, 0, 256]
    a, sfa, w, sfw = _case(ms, 512, 448, 51)
    d1 = run_dgrad(a, sfa, w, sfw, ms)
    d2 = run_dgrad(a, sfa, w, sfw, ms)
    assert torch.equal(d1, d2)


def test_dgrad_no_rows():
    """Every expert empty: nothing to write (d keeps its contents)."""
    ms, K, N = [0, 0, 0], 256, 224
    e = torch.empty(0, dtype=torch.uint8, device=DEV)
    w = torch.zeros(3, K, N, dtype=torch.uint8, device=DEV)
    sfw = torch.full((3, K // 128, N), 127, dtype=torch.uint8, device=DEV)
    d = torch.empty(0, N, dtype=torch.bfloat16, device=DEV)
    ms_dev = torch.tensor(ms, dtype=torch.int32, device=DEV)
    dg.dg_m_grouped_fp8_dgrad(e.view(0, K), e.view(0, K // 128), w, sfw, d, ms, ms_dev, 128)
    dg.dg_sync_check()


def test_dgrad_ms_dev_mismatch_is_reported():
    ms = [128, 256]
    a, sfa, w, sfw = _case(ms, 256, 224, 61)
    ms_dev = torch.tensor([256, 128], dtype=torch.int32, device=DEV)
    d = torch.empty(sum(ms), 224, dtype=torch.bfloat16, device=DEV)
    t = lambda x: torch.from_numpy(x).to(DEV)
    dg.dg_m_grouped_fp8_dgrad(t(a), t(sfa), t(w), t(sfw), d, ms, ms_dev, 128)
    with pytest.raises(dg.DGError) as ei:
        dg.dg_sync_check()
    assert ei.value.status == dg.DG_ERR_INVALID_ARG
    dg.dg_sync_check()                      # the status word was cleared


@pytest.mark.parametrize("w_kmajor", [False, True])
def test_dgrad_full_size_upgate_sampled(w_kmajor):
    """The bench's data-gradient workload (G = 32, K = 4096, N = 7168, 32768
    tokens, BF16 out) in the bench's launch configuration, weights [G, K, N]
    or K-major [G, N, K]; eight experts (the largest, the smallest non-empty,
    six seeded others) checked on 24 seeded rows each plus the smallest
    non-empty expert's rows in full."""
    name = "moe_upgate_dgrad_fp8_g32"
    ms, a, sfa, w, sfw = workloads.draw_dgrad_operands(name)
    d = torch.empty(a.shape[0], w.shape[2], dtype=torch.bfloat16, device=DEV)
    ms_dev = torch.tensor(ms, dtype=torch.int32, device=DEV)
    if w_kmajor:
        dg.dg_m_grouped_fp8_dgrad_nt(a.to(DEV), sfa.to(DEV), w.to(DEV).transpose(1, 2).contiguous(),
                                     sfw.to(DEV), d, ms, ms_dev, 128)
    else:
        dg.dg_m_grouped_fp8_dgrad(a.to(DEV), sfa.to(DEV), w.to(DEV), sfw.to(DEV), d, ms, ms_dev,
                                  128)
    dg.dg_sync_check()
    a, sfa, w, sfw = a.numpy(), sfa.numpy(), w.numpy(), sfw.numpy()
    off = oracle.expert_offsets(ms)
    live = [e for e in range(len(ms)) if ms[e] > 0]
    small = min(live, key=lambda e: ms[e])
    rng = np.random.default_rng(6)
    pick = {max(live, key=lambda e: ms[e]), small}
    pick |= set(rng.choice(live, size=6, replace=False).tolist())
    rows = []
    for e in sorted(pick):
        rows += (off[e] + rng.choice(ms[e], size=min(24, ms[e]), replace=False)).tolist()
    rows = sorted(set(rows) | set(range(off[small], off[small + 1])))
    D, S = oracle.mgrouped_fp8_dgrad_rows(a, sfa, w, sfw, ms, rows, 128)
    got = d[torch.tensor(rows, device=DEV)]
    assert_close(got, D, S, "bf16", what="dgrad full-size sampled")
    assert not torch.isnan(d.float()).any()
