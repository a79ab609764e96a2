"""The allocation-free FP8 entry point, dg_k_grouped_fp8_wgrad_noalloc.

It exists for callers that cannot allocate device memory: their memory belongs
to their own caching allocator, or they cannot take the device
synchronisation a cudaMalloc can cause.  It keeps its status record and the
packed scale records in a static device array of the library instead.

Each case is called twice in a row through the C ABI (the two calls share the
static array) and compared with the float64 oracle at the tolerances of the
other tests, and with the ordinary dg_k_grouped_fp8_wgrad on the same inputs
(same schedule and kernels, so equal results; in-place calls of experts split
along K add their parts in a timing-dependent order and are compared within
tolerance).  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import binding, workloads
import oracle
from tests.gpu_helpers import assert_close


def _problem(ks, M, N, seed, gran_k):
    sk = sum(ks)
    qa, sa = oracle.quant_colblock(workloads.randn((sk, M), seed).numpy(), gran_k)
    qb, sb = oracle.quant_colblock(workloads.randn((sk, N), seed + 1).numpy(), gran_k)
    return [torch.from_numpy(x).cuda() for x in (qa, sa, qb, sb)], (qa, sa, qb, sb)


def _noalloc(ops, d, c, ks, ks_dev, gran_k):
    qa, sa, qb, sb = ops
    G, M, N = d.shape
    kh = (ctypes.c_int * len(ks))(*ks)
    st = binding.lib().dg_k_grouped_fp8_wgrad_noalloc(
        qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), d.data_ptr(),
        binding.DG_BF16 if d.dtype == torch.bfloat16 else binding.DG_F32,
        None if c is None else c.data_ptr(), G, M, N, qa.shape[0], kh, ks_dev.data_ptr(),
        gran_k, torch.cuda.current_stream().cuda_stream)
    assert st == binding.DG_OK, binding.dg_last_error()


# (ks, M, N, gran_k, output, accumulator): direct 224-wide tiles, 128-wide
# ragged tiles, transposed tiles (N % 224 != 0, M % 224 == 0), BF16 output,
# a separate C, in place with an expert long enough to be split along K, and
# mixed 256 / 224 widths (N = 1792) with and without an accumulator.
CASES = [
    ([256, 0, 384, 128], 256, 448, 128, "f32", "inplace"),
    ([128, 640, 0], 384, 672, 128, "f32", "none"),
    ([512, 0, 256], 256, 320, 32, "f32", "separate"),
    ([384, 128, 0, 256], 448, 256, 128, "bf16", "none"),
    ([640, 256, 0], 448, 2048, 32, "f32", "inplace"),
    ([128 * 40, 128, 0], 256, 448, 128, "f32", "inplace"),
    ([128 * 12, 0, 128 * 6, 256], 256, 1792, 128, "f32", "none"),
    ([128 * 12, 0, 128 * 6, 256], 512, 1792, 32, "f32", "inplace"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=[f"{c[5]}-{c[4]}-g{c[3]}-{c[1]}x{c[2]}" for c in CASES])
def test_noalloc_matches_oracle_and_ordinary_entry_point(case):
    ks, M, N, gran_k, out, mode = case
    ops, host = _problem(ks, M, N, 7 + M + N, gran_k)
    ks_dev = torch.tensor(ks, dtype=torch.int32, device="cuda")
    dt = torch.float32 if out == "f32" else torch.bfloat16
    C = workloads.randn((len(ks), M, N), 11 + N)
    Cd = C.cuda()
    D, S = oracle.kgrouped_fp8_wgrad(*host, ks, gran_k,
                                     C.numpy() if mode in ("inplace", "separate") else None)

    def fresh():
        return Cd.clone() if mode == "inplace" else torch.full(Cd.shape, float("nan"), dtype=dt,
                                                               device="cuda")

    def acc(d):
        return d if mode == "inplace" else (Cd if mode == "separate" else None)

    d_ref = fresh()
    dg.dg_k_grouped_fp8_wgrad(*ops, d_ref, acc(d_ref), ks, ks_dev, gran_k)
    dg.dg_sync_check()
    for _ in range(2):                      # two calls in a row on the shared static array
        d_new = fresh()
        _noalloc(ops, d_new, acc(d_new), ks, ks_dev, gran_k)
        dg.dg_sync_check()                  # reads (and clears) the entry point's record too
        assert_close(d_new, D, S, out=out, what=f"noalloc {case}")
        if mode == "inplace":
            assert_close(d_new, d_ref.cpu().double().numpy(), S, out=out, what="vs ordinary")
            for e, k in enumerate(ks):
                if k == 0:
                    assert torch.equal(d_new[e], Cd[e])
        else:
            assert torch.equal(d_new, d_ref)


@pytest.mark.gpu
def test_noalloc_timeout_is_reported_by_sync_check(monkeypatch):
    # A wait limit of two microseconds ends the kernel early; the record in the
    # static array carries DG_ERR_TIMEOUT to dg_sync_check, which clears it.
    ks, M, N = [16384, 2048, 0], 256, 448
    ops, host = _problem(ks, M, N, 21, 128)
    ks_dev = torch.tensor(ks, dtype=torch.int32, device="cuda")
    d = torch.zeros(len(ks), M, N, device="cuda")
    dg.dg_sync_check()
    monkeypatch.setenv("DG_WAIT_LIMIT_US", "2")
    _noalloc(ops, d, None, ks, ks_dev, 128)
    with pytest.raises(binding.DGError) as ei:
        dg.dg_sync_check()
    assert ei.value.status == binding.DG_ERR_TIMEOUT
    monkeypatch.delenv("DG_WAIT_LIMIT_US")
    dg.dg_sync_check()
    _noalloc(ops, d, None, ks, ks_dev, 128)
    dg.dg_sync_check()
    D, S = oracle.kgrouped_fp8_wgrad(*host, ks, 128)
    assert_close(d, D, S, what="noalloc after a timed-out call")


def test_noalloc_rejects_too_many_experts_without_a_device():
    L = binding.lib()
    ks = (ctypes.c_int * (binding.DG_MAX_GROUPS + 1))()
    st = L.dg_k_grouped_fp8_wgrad_noalloc(None, None, None, None, 0x10000, binding.DG_F32,
                                          None, binding.DG_MAX_GROUPS + 1, 128, 128, 0, ks,
                                          0x10000, 128, None)
    assert st == binding.DG_ERR_UNSUPPORTED
    assert "maximum" in binding.dg_last_error()


def test_noalloc_rejects_scale_records_beyond_32_mib_without_a_device():
    # 2^20 tokens at gran_k 32 with M = N = 4096: one scale group per k-block,
    # 8192 groups x 64 records x 512 bytes = 256 MiB of packed scale records.
    # The check runs before any CUDA call; the pointers are never touched.
    L = binding.lib()
    G, M, N, sk = 1, 4096, 4096, 1 << 20
    ks = (ctypes.c_int * G)(sk)
    fake = 0x100000
    st = L.dg_k_grouped_fp8_wgrad_noalloc(fake, fake, fake, fake, fake, binding.DG_F32, None,
                                          G, M, N, sk, ks, fake, 32, None)
    assert st == binding.DG_ERR_UNSUPPORTED
    msg = binding.dg_last_error()
    assert "packed scale factors" in msg and "maximum" in msg
    # the same problem at gran_k 128 needs a quarter of that: 64 MiB, still too much
    st = L.dg_k_grouped_fp8_wgrad_noalloc(fake, fake, fake, fake, fake, binding.DG_F32, None,
                                          G, M, N, sk, ks, fake, 128, None)
    assert st == binding.DG_ERR_UNSUPPORTED
