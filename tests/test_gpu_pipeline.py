"""The full hot path at the pipeline workload's size: BF16 dY [131072, 4096] and
X [131072, 7168] are cast on the GPU, then the K-grouped FP8 GEMM accumulates
onto C in place (G = 64 experts, 59 with tokens).  The oracle independently
quantises slices of the same BF16 inputs and computes their gradients:

* the expert with the most tokens (38144, the longest K reduction of the
  workload, 298 k-blocks per tile) on 32 sampled rows x all 7168 columns,
  with the cast bytes and scales of its whole X slice and of its sampled dY
  columns compared bit for bit;
* every other expert with tokens on 4 sampled rows x 256 sampled columns,
  with the cast bytes and scales of those columns compared bit for bit
  (columns quantise independently, so a column sample of the oracle's cast
  is exactly that column of the full cast);
* experts without tokens left untouched (bitwise).

For this workload the schedule splits no expert along K: a tile of the
longest expert is 4 % of a CTA pair's share of the work, below the split
threshold of a quarter (the split itself is covered at small size by
test_inplace_long_expert_is_split)."""
import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import workloads
import oracle
from tests.gpu_helpers import assert_close, oracle_quant

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_pipeline_full_size_every_expert():
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
    big = max(nz, key=lambda e: ks[e])
    rng = np.random.default_rng(4)

    def check(e, rows, cols):
        sl = slice(int(off[e]), int(off[e + 1]))
        bs = slice(int(off[e]) // 128, int(off[e + 1]) // 128)
        r_t = torch.from_numpy(rows).cuda()
        c_t = torch.from_numpy(cols).cuda()
        ra, rsa = oracle_quant(dy[sl][:, r_t].float().cpu().numpy(), 128)
        rb, rsb = oracle_quant(x[sl][:, c_t].float().cpu().numpy(), 128)
        assert np.array_equal(qa[sl][:, r_t].cpu().numpy(), ra), f"dY cast, expert {e}"
        assert np.array_equal(sa[bs][:, r_t].cpu().numpy(), rsa), f"dY scales, expert {e}"
        assert np.array_equal(qb[sl][:, c_t].cpu().numpy(), rb), f"X cast, expert {e}"
        assert np.array_equal(sb[bs][:, c_t].cpu().numpy(), rsb), f"X scales, expert {e}"
        c0 = c_host[e][torch.from_numpy(rows)][:, torch.from_numpy(cols)]
        De, Se = oracle.kgrouped_fp8_wgrad(ra, rsa, rb, rsb, [ks[e]], 128, c0[None].numpy())
        got = c[e][r_t][:, c_t].cpu().double().numpy()
        assert_close(got, De[0], Se[0], what=f"pipeline expert {e} (K = {ks[e]})")

    check(big, np.sort(rng.choice(M, 32, replace=False)), np.arange(N))
    for e in nz:
        if e != big:
            check(e, np.sort(rng.choice(M, 4, replace=False)),
                  np.sort(rng.choice(N, 256, replace=False)))
    for e, k in enumerate(ks):
        if k == 0:
            assert torch.equal(c[e].cpu(), c_host[e])
