"""The allocation-free FP8 entry point, dg_k_grouped_fp8_wgrad_noalloc.

It exists for callers that cannot allocate device memory (their device memory
is owned by their own caching allocator, or they cannot take the device
synchronisation a cudaMalloc can cause).  Called here through the C ABI on two
problems in a row (sharing the library's static scratch array), each result
is compared with the ordinary dg_k_grouped_fp8_wgrad on the same inputs,
within the FP32 tolerance the other tests use (the kernels are the same, so the
results are also expected to be bitwise equal).  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import binding, workloads
import oracle

pytestmark = pytest.mark.gpu


def _problem(ks, M, N, seed):
    sk = sum(ks)
    qa, sa = oracle.quant_colblock(workloads.randn((sk, M), seed).numpy(), 128)
    qb, sb = oracle.quant_colblock(workloads.randn((sk, N), seed + 1).numpy(), 128)
    return [torch.from_numpy(x).cuda() for x in (qa, sa, qb, sb)], (qa, sa, qb, sb)


def _noalloc(ops, d, c, ks, ks_dev):
    qa, sa, qb, sb = ops
    G, M, N = d.shape
    kh = (ctypes.c_int * len(ks))(*ks)
    st = binding.lib().dg_k_grouped_fp8_wgrad_noalloc(
        qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), d.data_ptr(),
        binding.DG_F32, None if c is None else c.data_ptr(), G, M, N, qa.shape[0], kh,
        ks_dev.data_ptr(), 128, torch.cuda.current_stream().cuda_stream)
    assert st == binding.DG_OK, binding.dg_last_error()


def test_noalloc_matches_ordinary_entry_point_twice():
    cases = [([256, 0, 384, 128], 256, 448, 7, "inplace"),
             ([128, 640, 0], 384, 672, 9, "none")]
    for ks, M, N, seed, mode in cases:
        ops, host = _problem(ks, M, N, seed)
        ks_dev = torch.tensor(ks, dtype=torch.int32, device="cuda")
        C = workloads.randn((len(ks), M, N), seed + 2).cuda()
        d_ref = C.clone() if mode == "inplace" else torch.full_like(C, float("nan"))
        dg.dg_k_grouped_fp8_wgrad(*ops, d_ref, d_ref if mode == "inplace" else None,
                                  ks, ks_dev, 128)
        d_new = C.clone() if mode == "inplace" else torch.full_like(C, float("nan"))
        _noalloc(ops, d_new, d_new if mode == "inplace" else None, ks, ks_dev)
        torch.cuda.synchronize()
        _, S = oracle.kgrouped_fp8_wgrad(*host, ks, 128)
        err = np.abs(d_new.cpu().double().numpy() - d_ref.cpu().double().numpy())
        assert np.all(err <= oracle.fp32_bound(S)), float(np.nanmax(err))
        assert torch.equal(d_new, d_ref)


def test_noalloc_rejects_sizes_beyond_its_limits():
    L = binding.lib()
    ks = (ctypes.c_int * (binding.DG_MAX_GROUPS + 1))()
    st = L.dg_k_grouped_fp8_wgrad_noalloc(None, None, None, None, 0x10000, binding.DG_F32,
                                          None, binding.DG_MAX_GROUPS + 1, 128, 128, 0, ks,
                                          0x10000, 128, None)
    assert st == binding.DG_ERR_UNSUPPORTED
    assert "maximum" in binding.dg_last_error()
