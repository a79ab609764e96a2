"""The full hot path at the pipeline workload's size: BF16 dY and X are cast
on the GPU, then the K-grouped FP8 GEMM accumulates onto C in place.  The
oracle independently quantises the sampled experts' slices from the same BF16
inputs and computes their gradients; the GPU's cast bytes of those slices must
match bit for bit and the GEMM within tolerance."""
import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import workloads
import oracle
from tests.gpu_helpers import assert_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_pipeline_full_size_sampled_experts():
    w = workloads.WORKLOADS["pipeline_fp8_g64"]
    ks = workloads.counts_for(w.name)
    T, M, N, G = w.sum_k, w.M, w.N, w.G
    gen = torch.Generator(device="cuda").manual_seed(w.seed)
    dy = torch.randn(T, M, generator=gen, device="cuda").to(torch.bfloat16)
    x = torch.randn(T, N, generator=gen, device="cuda").to(torch.bfloat16)
    c = torch.randn(G, M, N, generator=gen, device="cuda") * w.c_std
    c_host = c.cpu()
    qa = torch.empty(T, M, dtype=torch.uint8, device="cuda")
    sa = torch.empty(T // 128, M, dtype=torch.uint8, device="cuda")
    qb = torch.empty(T, N, dtype=torch.uint8, device="cuda")
    sb = torch.empty(T // 128, N, dtype=torch.uint8, device="cuda")
    dg.dg_quant_transpose_fp8(dy, qa, sa)
    dg.dg_quant_transpose_fp8(x, qb, sb)
    ks_dev = torch.tensor(ks, dtype=torch.int32, device="cuda")
    dg.dg_k_grouped_fp8_wgrad(qa, sa, qb, sb, c, c, ks, ks_dev, 128)
    dg.dg_sync_check()

    off = np.cumsum([0] + ks)
    nz = [e for e, k in enumerate(ks) if k > 0]
    pick = sorted({min(nz, key=lambda e: ks[e]), nz[len(nz) // 2]})
    rows = np.sort(np.random.default_rng(4).choice(M, 32, replace=False))
    for e in pick:
        sl = slice(int(off[e]), int(off[e + 1]))
        ra, rsa = oracle.quant_colblock(dy[sl].float().cpu().numpy(), 128)
        rb, rsb = oracle.quant_colblock(x[sl].float().cpu().numpy(), 128)
        assert np.array_equal(qa[sl].cpu().numpy(), ra)
        assert np.array_equal(qb[sl].cpu().numpy(), rb)
        bs = slice(int(off[e]) // 128, int(off[e + 1]) // 128)
        assert np.array_equal(sa[bs].cpu().numpy(), rsa)
        assert np.array_equal(sb[bs].cpu().numpy(), rsb)
        De, Se = oracle.kgrouped_fp8_wgrad(ra[:, rows], rsa[:, rows], rb, rsb, [ks[e]], 128,
                                           c_host[e][rows][None].numpy())
        got = c[e][torch.from_numpy(rows).cuda()].cpu().double().numpy()
        assert_close(got, De[0], Se[0], what=f"pipeline expert {e}")
    for e, k in enumerate(ks):
        if k == 0:
            assert torch.equal(c[e].cpu(), c_host[e])
