"""GPU parity of the mixed-width FP8 weight gradient.

When the kernel's N is a multiple of both 256 and 224 (N = 1792 k), the
schedule cuts the longest experts into 256 x 256 tiles, which only the first
accumulator holds, and the rest into 256 x 224 tiles; the second accumulator
takes narrow tiles only, and the tensor memory keeps two scale slots instead
of five.  Each case checks against the float64 oracle at the tolerances of the
other FP8 tests, with the plan read from the DG_LOG line (so that the wide
tiles are known to have run), and again with DG_MIXED_TILES=0 (224 columns
only).  DG_MIXED_TILES=1000 makes every entry wide, so lane 1 gets nothing
but output-only tiles and lane 0 runs the rest alone.
"""
import re

import numpy as np
import pytest
import torch

from grouped_fp8_weight_gb300 import workloads
import oracle
from tests.gpu_helpers import DEV, assert_close, fp8_operands, run_fp8
from tests.test_gpu_wgrad_nt import run_nt

pytestmark = pytest.mark.gpu

_PLAN = re.compile(r"\((\d+) entries of 256 x 256 tiles")


def _case(ks, M, N, seed, gran_k=128):
    sk = sum(ks)
    qa, sa, qb, sb = fp8_operands(workloads.randn((sk, M), seed).numpy(),
                                  workloads.randn((sk, N), seed + 1).numpy(), gran_k)
    rng = np.random.default_rng(seed)    # distinct per-row / per-column scales
    sa = (sa.astype(np.int64) + rng.integers(-6, 7, sa.shape)).astype(np.uint8)
    sb = (sb.astype(np.int64) + rng.integers(-6, 7, sb.shape)).astype(np.uint8)
    return qa, sa, qb, sb


def _run_logged(monkeypatch, capfd, mixed, *args, run=run_fp8, **kw):
    """run_fp8 (or run_nt) with DG_LOG on; returns (D, number of wide entries
    in the plan)."""
    monkeypatch.setenv("DG_LOG", "1")
    if mixed is None:
        monkeypatch.delenv("DG_MIXED_TILES", raising=False)
    else:
        monkeypatch.setenv("DG_MIXED_TILES", str(mixed))
    capfd.readouterr()
    d = run(*args, **kw)
    err = capfd.readouterr().err
    m = _PLAN.findall(err)
    assert m, f"no plan line in {err!r}"
    monkeypatch.delenv("DG_LOG")
    return d, int(m[-1])


@pytest.mark.parametrize("gran_k", [128, 32])
@pytest.mark.parametrize("out,c_mode", [("f32", "none"), ("f32", "inplace"),
                                        ("f32", "separate"), ("bf16", "none")])
def test_mixed_modes(monkeypatch, capfd, gran_k, out, c_mode):
    ks = [128 * 12, 128 * 6, 0, 256, 128]
    M, N = 256, 1792
    qa, sa, qb, sb = _case(ks, M, N, 41, gran_k)
    C = workloads.randn((len(ks), M, N), 42).numpy()
    c = C if c_mode != "none" else None
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, gran_k, c)
    for mixed in (None, 0):
        d, n_wide = _run_logged(monkeypatch, capfd, mixed, qa, sa, qb, sb, ks, gran_k, out, c,
                                c_mode)
        assert (n_wide > 0) == (mixed is None), n_wide
        assert_close(d, D, S, out, what=f"{out}/{c_mode}/g{gran_k}/mixed={mixed}")
        if c_mode == "inplace":
            assert torch.equal(d[2].cpu(), torch.from_numpy(C[2]))
        elif c_mode == "none" and out == "f32":
            assert torch.count_nonzero(d[2]).item() == 0


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_mixed_transposed(monkeypatch, capfd, out):
    # N = 256 is no multiple of 224 but M = 1792 is: D^T tiles, whose 256- and
    # 224-wide sides run along M.
    ks = [128 * 10, 128 * 3, 128, 0]
    M, N = 1792, 256
    qa, sa, qb, sb = _case(ks, M, N, 43)
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    d, n_wide = _run_logged(monkeypatch, capfd, None, qa, sa, qb, sb, ks, 128, out)
    assert n_wide > 0
    assert_close(d, D, S, out, what=f"transposed {out}")


def test_mixed_all_wide_lane0_alone(monkeypatch, capfd):
    # 7 x 28 wide tiles and 4 output-only ones over 76 CTA pairs: lane 1 finds
    # wide tiles at the tail of its list and leaves them to lane 0.
    ks = [128 * 9, 128 * 4, 0, 256, 128 * 6, 384, 128, 128 * 5]
    M, N = 1024, 1792
    qa, sa, qb, sb = _case(ks, M, N, 45)
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128)
    d, n_wide = _run_logged(monkeypatch, capfd, 1000, qa, sa, qb, sb, ks, 128)
    assert n_wide == 7
    assert_close(d, D, S, what="every entry wide")


@pytest.mark.parametrize("gran_k", [128, 32])
def test_mixed_many_tiles_per_pair(monkeypatch, capfd, gran_k):
    """Several wide and narrow tiles per CTA pair, lane chunks of the longest
    experts (82 and 41 k-blocks) interleaved with narrow and output-only tiles;
    every expert checked on sampled rows x all N."""
    ks = [128 * 82, 128 * 41, 128 * 13, 0, 128 * 5, 128 * 2, 128, 128 * 3]
    M, N = 2048, 3584
    qa, sa, qb, sb = _case(ks, M, N, 47, gran_k)
    d, n_wide = _run_logged(monkeypatch, capfd, None, qa, sa, qb, sb, ks, gran_k)
    assert 0 < n_wide < 7
    rows = np.sort(np.random.default_rng(47).choice(M, 16, replace=False))
    part = oracle.kgrouped_fp8_wgrad_rows(qa, sa, qb, sb, ks, rows, gran_k)
    dr = d[:, torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    for e, (De, Se) in part.items():
        assert_close(dr[e], De, Se, what=f"expert {e} (K = {ks[e]})")
    assert torch.count_nonzero(d[3]).item() == 0


@pytest.mark.parametrize("gran_k", [128, 32])
@pytest.mark.parametrize("out,c_mode", [("f32", "none"), ("f32", "inplace"), ("bf16", "none")])
def test_mixed_k_major(monkeypatch, capfd, gran_k, out, c_mode):
    # K-major (NT) operands a [M, sum_k], b [N, sum_k]: the same widths
    ks = [128 * 12, 128 * 6, 0, 256, 128]
    M, N = 256, 1792
    qa, sa, qb, sb = _case(ks, M, N, 49, gran_k)
    C = workloads.randn((len(ks), M, N), 50).numpy()
    c = C if c_mode != "none" else None
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, gran_k, c)
    d, n_wide = _run_logged(monkeypatch, capfd, None, qa, sa, qb, sb, ks, gran_k, out, c, c_mode,
                            run=run_nt)
    assert n_wide > 0
    assert_close(d, D, S, out, what=f"K-major {out}/{c_mode}/g{gran_k}")
    if c_mode == "inplace":
        assert torch.equal(d[2].cpu(), torch.from_numpy(C[2]))


def test_mixed_k_major_transposed_many_tiles(monkeypatch, capfd):
    # D^T tiles on K-major operands (M = 3584 along the tiles' widths), several
    # wide and narrow tiles per CTA pair; sampled rows x all N
    ks = [128 * 40, 128 * 17, 128 * 5, 0, 128 * 2, 128]
    M, N = 3584, 512
    qa, sa, qb, sb = _case(ks, M, N, 51)
    d, n_wide = _run_logged(monkeypatch, capfd, None, qa, sa, qb, sb, ks, 128, run=run_nt)
    assert n_wide > 0
    rows = np.sort(np.random.default_rng(51).choice(M, 16, replace=False))
    part = oracle.kgrouped_fp8_wgrad_rows(qa, sa, qb, sb, ks, rows, 128)
    dr = d[:, torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    for e, (De, Se) in part.items():
        assert_close(dr[e], De, Se, what=f"K-major transposed expert {e}")


def test_mixed_many_experts_schedule_from_parameters(monkeypatch, capfd):
    """More schedule entries than shared memory holds (330 experts, 256 kept
    there): wide and narrow tiles with the schedule read from the kernel
    parameters, in place, every expert against the oracle."""
    rng = np.random.default_rng(53)
    ks = [128 * int(k) for k in rng.choice([0, 1, 1, 2, 2, 3], size=330)]
    for e in rng.choice(330, size=8, replace=False):
        ks[int(e)] = 128 * int(rng.integers(12, 33))
    M, N = 128, 1792
    qa, sa, qb, sb = _case(ks, M, N, 53)
    C = workloads.randn((len(ks), M, N), 54).numpy()
    D, S = oracle.kgrouped_fp8_wgrad(qa, sa, qb, sb, ks, 128, C)
    d, n_wide = _run_logged(monkeypatch, capfd, None, qa, sa, qb, sb, ks, 128, "f32", C, "inplace")
    assert n_wide > 0
    assert_close(d, D, S, what="330 experts, mixed widths, in place")
    for e, k in enumerate(ks):
        if k == 0:
            assert torch.equal(d[e].cpu(), torch.from_numpy(C[e]))
