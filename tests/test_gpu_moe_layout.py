"""GPU parity of dg_moe_layout_plan (bit-exact against the oracle's layout),
and the chain it serves: top-k routing -> plan -> casts fused with the MoE
layout (X by source token, dY by routed pair) -> K-grouped FP8 weight
gradient, against the oracle end to end."""
import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import workloads
import oracle
from gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


def _routing(T, topk, G, seed, unused=0.1, zipf=1.2):
    """Top-k routing with Zipf expert popularity, distinct experts per token,
    a fraction of slots unused (-1)."""
    rng = np.random.default_rng(seed)
    p = np.arange(1, G + 1, dtype=np.float64) ** -zipf
    p /= p.sum()
    k = min(topk, G)
    # Gumbel top-k: distinct experts drawn by popularity
    g = np.log(p)[None, :] - np.log(-np.log(rng.random((T, G))))
    idx = np.argsort(-g, axis=1)[:, :k]
    if k < topk:
        idx = np.concatenate([idx, -np.ones((T, topk - k), dtype=np.int64)], axis=1)
    idx[rng.random((T, topk)) < unused] = -1
    return idx.astype(np.int32)


def _plan_gpu(idx, G, align=128):
    ks, src, pair = dg.dg_moe_layout_plan(torch.from_numpy(idx).cuda(), G, align,
                                          with_pairs=True)
    dg.dg_sync_check()
    return ks.cpu().numpy(), src.cpu().numpy(), pair.cpu().numpy()


@pytest.mark.parametrize("T,topk,G,align", [
    (0, 2, 4, 128), (1, 1, 1, 128), (300, 3, 7, 128), (5000, 8, 64, 128),
    (4096 * 3 + 17, 2, 256, 128), (20000, 8, 1024, 128), (999, 4, 32, 32), (777, 2, 16, 1),
])
def test_plan_matches_oracle(T, topk, G, align):
    idx = _routing(T, topk, G, seed=T + G)
    ks, src, pair = _plan_gpu(idx, G, align)
    rk, rsrc, rpair = oracle.moe_layout_plan(idx, G, align)
    assert np.array_equal(ks, rk)
    n = int(rk.sum())
    assert np.array_equal(src[:n], rsrc) and np.array_equal(pair[:n], rpair)
    assert np.all(src[n:] == -1) and np.all(pair[n:] == -1)


def test_plan_large_routing():
    """Pipeline scale: 131072 tokens, top-8 of 64 experts (1 M routing entries)."""
    idx = _routing(131072, 8, 64, seed=3, unused=0.0)
    ks, src, pair = _plan_gpu(idx, 64)
    rk, rsrc, rpair = oracle.moe_layout_plan(idx, 64)
    n = int(rk.sum())
    assert np.array_equal(ks, rk) and np.array_equal(pair[:n], rpair)
    assert np.array_equal(src[:n], rsrc)


def test_plan_out_of_range_entry_is_reported():
    idx = _routing(500, 2, 8, seed=4)
    idx[3, 1] = 8
    ks, src, pair = dg.dg_moe_layout_plan(torch.from_numpy(idx).cuda(), 8, with_pairs=True)
    with pytest.raises(dg.DGError, match="topk_idx"):
        dg.dg_sync_check()
    idx[3, 1] = -1                                  # the entry was skipped
    rk, rsrc, rpair = oracle.moe_layout_plan(idx, 8)
    assert np.array_equal(ks.cpu().numpy(), rk)
    assert np.array_equal(pair.cpu().numpy()[:int(rk.sum())], rpair)
    dg.dg_sync_check()


def test_routing_to_weight_gradient():
    """X [T, N] (BF16, per token) and dY [T * topk, M] (BF16, per routed pair):
    the plan, both casts fused with the layout, and the FP8 GEMM, against the
    oracle's layout, casts and GEMM."""
    T, topk, G, M, N = 900, 2, 6, 256, 384
    idx = _routing(T, topk, G, seed=6)
    x = workloads.randn((T, N), seed=61, dtype=torch.bfloat16)
    dy = workloads.randn((T * topk, M), seed=62, dtype=torch.bfloat16)
    ks_d, src, pair = dg.dg_moe_layout_plan(torch.from_numpy(idx).cuda(), G, with_pairs=True)
    ks = ks_d.cpu().tolist()
    S = sum(ks)
    qa = torch.empty(S, M, dtype=torch.uint8, device="cuda")
    sa = torch.empty(S // 128, M, dtype=torch.uint8, device="cuda")
    qb = torch.empty(S, N, dtype=torch.uint8, device="cuda")
    sb = torch.empty(S // 128, N, dtype=torch.uint8, device="cuda")
    dg.dg_quant_moe_layout_fp8(dy.cuda(), pair[:S].contiguous(), qa, sa)
    dg.dg_quant_moe_layout_fp8(x.cuda(), src[:S].contiguous(), qb, sb)
    d = torch.full((G, M, N), float("nan"), device="cuda")
    dg.dg_k_grouped_fp8_wgrad(qa, sa, qb, sb, d, None, ks, ks_d, 128)
    dg.dg_sync_check()
    rk, rsrc, rpair = oracle.moe_layout_plan(idx, G)
    assert ks == rk.tolist()
    ra, rsa = oracle.moe_layout_cast(dy.float().numpy(), rpair)
    rb, rsb = oracle.moe_layout_cast(x.float().numpy(), rsrc)
    assert np.array_equal(qa.cpu().numpy(), ra) and np.array_equal(sa.cpu().numpy(), rsa)
    assert np.array_equal(qb.cpu().numpy(), rb) and np.array_equal(sb.cpu().numpy(), rsb)
    D, Sb = oracle.kgrouped_fp8_wgrad(ra, rsa, rb, rsb, ks, 128)
    assert_close(d, D, Sb, "f32", "routing -> plan -> casts -> GEMM")
