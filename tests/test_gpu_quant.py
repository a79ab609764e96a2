"""GPU parity of dg_quant_transpose_fp8: bit-exact E4M3 bytes and UE8M0
exponents against the oracle, both layouts and both granularities, ragged
tiles, special values, and sampled blocks of the full-size pipeline input."""
import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import workloads
import oracle

pytestmark = pytest.mark.gpu


def _gpu_quant(x_bf16, gran_k, layout):
    T, C = x_bf16.shape
    x = x_bf16.cuda()
    q = torch.empty((T, C) if layout == "token" else (C, T), dtype=torch.uint8, device="cuda")
    sf = torch.empty(T // gran_k, C, dtype=torch.uint8, device="cuda")
    dg.dg_quant_transpose_fp8(x, q, sf, layout, gran_k)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy()


def _check(x_bf16, gran_k, layout):
    q, sf = _gpu_quant(x_bf16, gran_k, layout)
    rq, rsf = oracle.quant_colblock(x_bf16.float().numpy(), gran_k, layout)
    assert np.array_equal(sf, rsf), np.argwhere(sf != rsf)[:5]
    bad = np.argwhere(q != rq)
    assert bad.size == 0, (bad[:5], q[tuple(bad[0])], rq[tuple(bad[0])])


@pytest.mark.parametrize("layout", ["token", "channel"])
@pytest.mark.parametrize("gran_k", [128, 32])
@pytest.mark.parametrize("T,C", [(128, 256), (512, 768), (384, 272), (256, 16), (1024, 7168 // 4)])
def test_quant_random(T, C, gran_k, layout):
    x = workloads.randn((T, C), seed=T * 7 + C, dtype=torch.bfloat16)
    _check(x, gran_k, layout)


@pytest.mark.parametrize("layout", ["token", "channel"])
def test_quant_gran32_partial_token_tile(layout):
    x = workloads.randn((160, 528), seed=9, dtype=torch.bfloat16)      # 160 = 5 x 32
    _check(x, 32, layout)


@pytest.mark.parametrize("layout", ["token", "channel"])
@pytest.mark.parametrize("gran_k", [128, 32])
def test_quant_special_values(gran_k, layout):
    T, C = 256, 64
    x = workloads.randn((T, C), seed=3).numpy()
    x[:, 0] = 0.0                                   # zero block -> scale byte 0
    x[:, 1] = -0.0
    x[:, 2] *= 1e-39                                # bf16 subnormals
    x[:, 3] = np.where(np.arange(T) % 2, -1e-40, 0.0)
    x[:, 4] = 1.75 * 2.0 ** 3                       # amax exactly 1.75 * 2^q
    x[:, 5] = np.nextafter(np.float32(1.75 * 8), np.float32(np.inf))
    x[:, 6] = 448.0
    x[:, 7] *= 3e38 / 4                             # near the bf16 maximum
    x[:, 8] *= 1e-30
    x[::3, 9] = -2.0 ** -9
    x[:, 10] = np.linspace(-3, 3, T)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    _check(xb, gran_k, layout)


def test_quant_full_size_pipeline_sampled():
    """The pipeline's X [131072, 7168] in the bench's launch configuration;
    sampled token blocks (all channels) checked bit for bit."""
    T, C = 131072, 7168
    gen = torch.Generator(device="cuda").manual_seed(4)
    x = torch.randn(T, C, generator=gen, device="cuda").to(torch.bfloat16)
    q = torch.empty(T, C, dtype=torch.uint8, device="cuda")
    sf = torch.empty(T // 128, C, dtype=torch.uint8, device="cuda")
    dg.dg_quant_transpose_fp8(x, q, sf, "token", 128)
    torch.cuda.synchronize()
    for kb in [0, 1, 517, 1023]:
        rows = slice(kb * 128, (kb + 1) * 128)
        xs = x[rows].float().cpu().numpy()
        rq, rsf = oracle.quant_colblock(xs, 128)
        assert np.array_equal(sf[kb].cpu().numpy(), rsf[0])
        assert np.array_equal(q[rows].cpu().numpy(), rq)
    del x, q, sf
    torch.cuda.empty_cache()
