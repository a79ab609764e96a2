"""GPU parity of dg_requant_transpose_fp8 and dg_quant_moe_layout_fp8: E4M3
bytes and UE8M0 exponents bit-exact against the oracle, both layouts and both
granularities, ragged tiles, the extremes of the stored scale range, padding
rows, an out-of-range row index, and sampled blocks of full-size inputs."""
import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import workloads
import oracle

pytestmark = pytest.mark.gpu


def _out(T, C, gran_k, layout):
    q = torch.empty((T, C) if layout == "token" else (C, T), dtype=torch.uint8, device="cuda")
    sf = torch.empty(T // gran_k, C, dtype=torch.uint8, device="cuda")
    return q, sf


def _requant_gpu(q_in, sf_in, gran_k, layout):
    T, C = q_in.shape
    q, sf = _out(T, C, gran_k, layout)
    dg.dg_requant_transpose_fp8(torch.from_numpy(q_in).cuda(), torch.from_numpy(sf_in).cuda(),
                                q, sf, layout, gran_k)
    dg.dg_sync_check()
    return q.cpu().numpy(), sf.cpu().numpy()


def _assert_same(got, want):
    (q, sf), (rq, rsf) = got, want
    assert np.array_equal(sf, rsf), np.argwhere(sf != rsf)[:5]
    bad = np.argwhere(q != rq)
    assert bad.size == 0, (bad[:5], q[tuple(bad[0])], rq[tuple(bad[0])])


def _stored(T, C, seed):
    """Forward-pass FP8 activations: BF16 N(0, 1) cast in 1 x 128 tiles by the oracle."""
    x = workloads.randn((T, C), seed=seed, dtype=torch.bfloat16).float().numpy()
    return oracle.quant_rowtile(x)


@pytest.mark.parametrize("layout", ["token", "channel"])
@pytest.mark.parametrize("gran_k", [128, 32])
@pytest.mark.parametrize("T,C", [(128, 256), (512, 768), (384, 384), (256, 128), (1024, 1792)])
def test_requant_random(T, C, gran_k, layout):
    q_in, sf_in = _stored(T, C, seed=T + 3 * C)
    _assert_same(_requant_gpu(q_in, sf_in, gran_k, layout),
                 oracle.requant_colblock(q_in, sf_in, gran_k, layout))


@pytest.mark.parametrize("layout", ["token", "channel"])
@pytest.mark.parametrize("gran_k", [128, 32])
def test_requant_scale_extremes(gran_k, layout):
    """Random codes under scale bytes 0..254: blocks whose maximum is below
    2^-118 (a subnormal FP32 intermediate), blocks needing a factor above
    2^127, the top of the range, and blocks mixing huge and tiny tiles."""
    rng = np.random.default_rng(17)
    T, C = 640, 384
    q_in = rng.integers(0, 256, size=(T, C)).astype(np.uint8)
    q_in[(q_in & 0x7F) == 0x7F] = 0x7E                       # no NaN codes
    sf_in = rng.integers(0, 255, size=(T, C // 128)).astype(np.uint8)
    sf_in[0:128, 0] = rng.integers(0, 9, size=128)           # tiny block
    sf_in[128:256, 1] = rng.integers(0, 4, size=128)          # factor 2^(8 - e) > 2^127
    sf_in[128:256, 2] = 0
    sf_in[256:384, 0] = rng.integers(245, 255, size=128)       # top of the range
    sf_in[384:512, :] = np.where(rng.random((128, C // 128)) < 0.5, 250, 2)   # mixed
    q_in[512:640, :64] = 0x80                                  # negative zeros
    q_in[512:640, 64:72] = rng.choice(np.array([0x01, 0x81, 0x07, 0x87], np.uint8), (128, 8))
    sf_in[512:640, 0] = 0                                      # subnormal codes, least scale
    _assert_same(_requant_gpu(q_in, sf_in, gran_k, layout),
                 oracle.requant_colblock(q_in, sf_in, gran_k, layout))


@pytest.mark.parametrize("layout", ["token", "channel"])
@pytest.mark.parametrize("gran_k", [128, 32])
def test_requant_row_scale_spread(gran_k, layout):
    """One row per 128-token block with a scale byte above the rest (by 15 to
    26) and zero codes in some channels: there the block maximum comes from
    rows whose dequantised values, relative to that row's scale, fall to the
    subnormal range or below it, and in the third block small codes put every
    such product below 2^-14."""
    rng = np.random.default_rng(23)
    T, C = 512, 512
    q_in = rng.integers(0, 256, size=(T, C)).astype(np.uint8)
    q_in[(q_in & 0x7F) == 0x7F] = 0x7E                       # no NaN codes
    sf_in = np.zeros((T, C // 128), dtype=np.uint8)
    for blk, spread in enumerate((13, 16, 20, 24)):
        rows = slice(128 * blk, 128 * blk + 128)
        sf_in[rows, :] = 140 - spread
        sf_in[128 * blk + 7, :] = 142                        # one row above the rest
        q_in[128 * blk + 7, : 32 * (blk + 1)] = 0            # ... with zeros in some channels
    q_in[256:384, :64] = rng.integers(1, 0x30, size=(128, 64)).astype(np.uint8)   # |x| < 0.5
    q_in[256 + 7, :64] = 0
    _assert_same(_requant_gpu(q_in, sf_in, gran_k, layout),
                 oracle.requant_colblock(q_in, sf_in, gran_k, layout))


def _moe_src(T_tok, G, topk, seed):
    """An MoE layout from random top-k routing: each expert's (token, slot)
    pairs in token order, padded with -1 to a multiple of 128."""
    rng = np.random.default_rng(seed)
    p = (np.arange(1, G + 1) ** -1.2)
    p /= p.sum()
    ex = np.stack([rng.choice(G, size=topk, replace=False, p=p) for _ in range(T_tok)])
    rows, ks = [], []
    for e in range(G):
        toks = np.nonzero((ex == e).any(axis=1))[0]
        pad = (-len(toks)) % 128
        rows.append(np.concatenate([toks, -np.ones(pad, dtype=np.int64)]))
        ks.append(len(toks) + pad)
    return np.concatenate(rows).astype(np.int32), ks


def _moe_gpu(x, src, gran_k, layout, x_sf=None):
    T = src.shape[0]
    C = x.shape[1]
    q, sf = _out(T, C, gran_k, layout)
    xd = torch.from_numpy(x).cuda() if isinstance(x, np.ndarray) else x.cuda()
    dg.dg_quant_moe_layout_fp8(xd, torch.from_numpy(src).cuda(), q, sf,
                               None if x_sf is None else torch.from_numpy(x_sf).cuda(),
                               layout, gran_k)
    dg.dg_sync_check()
    return q.cpu().numpy(), sf.cpu().numpy()


@pytest.mark.parametrize("layout", ["token", "channel"])
@pytest.mark.parametrize("gran_k", [128, 32])
@pytest.mark.parametrize("src_kind", ["bf16", "fp8"])
def test_moe_layout_cast(src_kind, gran_k, layout):
    T_tok, C, G, topk = 700, 384, 6, 2
    src, ks = _moe_src(T_tok, G, topk, seed=5)
    xb = workloads.randn((T_tok, C), seed=23, dtype=torch.bfloat16)
    if src_kind == "bf16":
        got = _moe_gpu(xb, src, gran_k, layout)
        want = oracle.moe_layout_cast(xb.float().numpy(), src, gran_k, layout)
    else:
        qs, ss = oracle.quant_rowtile(xb.float().numpy())
        got = _moe_gpu(qs, src, gran_k, layout, x_sf=ss)
        want = oracle.moe_layout_cast(qs, src, gran_k, layout, sf_row=ss)
    _assert_same(got, want)


@pytest.mark.parametrize("T,C", [(160, 208), (32 * 45, 400)])
def test_moe_layout_ragged_tiles(T, C):
    # gran_k 32: the last 128-row tile is partial and C is not a multiple of
    # the 128-channel tile; padding rows scattered through the layout
    rng = np.random.default_rng(T + C)
    T_src = 300
    src = rng.integers(0, T_src, T).astype(np.int32)
    src[rng.random(T) < 0.2] = -1
    xb = workloads.randn((T_src, C), seed=T + C, dtype=torch.bfloat16)
    got = _moe_gpu(xb, src, 32, "token")
    want = oracle.moe_layout_cast(xb.float().numpy(), src, 32, "token")
    _assert_same(got, want)


def test_moe_layout_all_padding_and_empty_source():
    """A layout of padding rows only (T_src = 0) gives zero codes and the
    least scale byte."""
    src = -np.ones(256, dtype=np.int32)
    x = torch.empty(0, 64, dtype=torch.bfloat16)
    q, sf = _moe_gpu(x, src, 128, "token")
    assert not q.any() and not sf.any()


@pytest.mark.parametrize("src_kind", ["bf16", "fp8"])
def test_moe_layout_out_of_range_index_is_reported(src_kind):
    C = 64 if src_kind == "bf16" else 128          # stored E4M3 rows: whole 128-channel tiles
    x = workloads.randn((200, C), seed=4, dtype=torch.bfloat16)
    src = np.arange(256, dtype=np.int32) % 200
    src[7] = 200                                   # one past the end
    q, sf = _out(256, C, 128, "token")
    if src_kind == "bf16":
        dg.dg_quant_moe_layout_fp8(x.cuda(), torch.from_numpy(src).cuda(), q, sf)
    else:
        qs, ss = oracle.quant_rowtile(x.float().numpy())
        dg.dg_quant_moe_layout_fp8(torch.from_numpy(qs).cuda(), torch.from_numpy(src).cuda(), q,
                                   sf, torch.from_numpy(ss).cuda())
    with pytest.raises(dg.DGError, match="src_rows"):
        dg.dg_sync_check()
    src[7] = -1                                    # the row it wrote: zeros
    if src_kind == "bf16":
        want = oracle.moe_layout_cast(x.float().numpy(), src, 128)
    else:
        want = oracle.moe_layout_cast(qs, src, 128, sf_row=ss)
    _assert_same((q.cpu().numpy(), sf.cpu().numpy()), want)
    dg.dg_sync_check()                             # the status word was cleared


def test_requant_full_size_sampled():
    """Stored activations of the pipeline's X shape [131072, 7168] (random
    codes, scale bytes around 127) re-quantised in the launch configuration of
    the bench; sampled token blocks checked bit for bit."""
    T, C = 131072, 7168
    gen = torch.Generator(device="cuda").manual_seed(31)
    q_in = torch.randint(0, 256, (T, C), generator=gen, device="cuda", dtype=torch.uint8)
    q_in[(q_in & 0x7F) == 0x7F] = 0x7E
    sf_in = torch.randint(110, 140, (T, C // 128), generator=gen, device="cuda",
                          dtype=torch.uint8)
    q, sf = _out(T, C, 128, "token")
    dg.dg_requant_transpose_fp8(q_in, sf_in, q, sf)
    dg.dg_sync_check()
    for kb in [0, 3, 600, 1023]:
        rows = slice(kb * 128, (kb + 1) * 128)
        rq, rsf = oracle.requant_colblock(q_in[rows].cpu().numpy(), sf_in[rows].cpu().numpy())
        assert np.array_equal(sf[kb].cpu().numpy(), rsf[0])
        assert np.array_equal(q[rows].cpu().numpy(), rq)
    del q_in, sf_in, q, sf
    torch.cuda.empty_cache()


def test_moe_layout_full_size_sampled():
    """BF16 X [65536, 7168] gathered into a top-2 MoE layout over 64 experts
    (about 131k rows with padding); sampled output blocks checked bit for bit."""
    T_tok, C, G, topk = 65536, 7168, 64, 2
    rng = np.random.default_rng(8)
    p = np.arange(1, G + 1) ** -1.2
    p /= p.sum()
    # top-2 routing drawn per token without replacement, vectorised: the first
    # expert by p, the second by p with the first removed
    e1 = rng.choice(G, size=T_tok, p=p)
    e2 = (e1 + 1 + rng.choice(G - 1, size=T_tok)) % G
    rows = []
    for e in range(G):
        toks = np.nonzero((e1 == e) | (e2 == e))[0]
        rows.append(np.concatenate([toks, -np.ones((-len(toks)) % 128, dtype=np.int64)]))
    src = np.concatenate(rows).astype(np.int32)
    gen = torch.Generator(device="cuda").manual_seed(9)
    x = torch.randn(T_tok, C, generator=gen, device="cuda").to(torch.bfloat16)
    T = src.shape[0]
    q, sf = _out(T, C, 128, "token")
    dg.dg_quant_moe_layout_fp8(x, torch.from_numpy(src).cuda(), q, sf)
    dg.dg_sync_check()
    for kb in [0, 5, T // 256, T // 128 - 1]:
        s = src[kb * 128:(kb + 1) * 128]
        xs = x[torch.from_numpy(np.maximum(s, 0)).cuda().long()].float().cpu().numpy()
        rq, rsf = oracle.moe_layout_cast(xs, np.where(s >= 0, np.arange(128), -1), 128)
        assert np.array_equal(sf[kb].cpu().numpy(), rsf[0])
        assert np.array_equal(q[kb * 128:(kb + 1) * 128].cpu().numpy(), rq)
    del x, q, sf
    torch.cuda.empty_cache()
