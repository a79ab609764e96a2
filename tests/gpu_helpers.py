"""Shared helpers for the GPU parity tests: operand preparation through the
oracle (CPU), calls through the C-ABI binding, and the tolerance checks."""
import numpy as np
import torch

import grouped_fp8_weight_gb300 as dg
import oracle

DEV = "cuda"


_POOL = None


def _pool():
    """Process pool for the oracle (spawned, so it is safe after CUDA init)."""
    global _POOL
    if _POOL is None:
        import multiprocessing as mp
        import os
        n = max(1, min(16, len(os.sched_getaffinity(0))))
        _POOL = mp.get_context("spawn").Pool(n)
    return _POOL


def _quant_chunk(args):
    x, gran_k = args
    return oracle.quant_colblock(x, gran_k)


def oracle_quant(x, gran_k=128, rows_per_task=2048):
    """oracle.quant_colblock over token-block chunks in parallel (identical
    result: blocks are independent)."""
    x = np.asarray(x)
    T = x.shape[0]
    if T <= rows_per_task:
        return oracle.quant_colblock(x, gran_k)
    step = max(gran_k, rows_per_task // gran_k * gran_k)
    parts = _pool().map(_quant_chunk, [(x[i:i + step], gran_k) for i in range(0, T, step)])
    return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))


def fp8_operands(A_raw, B_raw, gran_k=128):
    """Quantise raw float operands with the ORACLE's quantiser (never the GPU's)."""
    qa, sa = oracle_quant(A_raw, gran_k)
    qb, sb = oracle_quant(B_raw, gran_k)
    return qa, sa, qb, sb


def to_dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x)) if isinstance(x, np.ndarray) else x
    t = t.to(DEV)
    return t if dtype is None else t.to(dtype)


def run_fp8(qa, sa, qb, sb, ks, gran_k=128, out="f32", c=None, c_mode="none"):
    """Run the GPU K-grouped FP8 kernel.  c_mode: none | inplace | separate."""
    G, M, N = len(ks), qa.shape[1], qb.shape[1]
    dt = torch.float32 if out == "f32" else torch.bfloat16
    ks_dev = torch.tensor(ks, dtype=torch.int32, device=DEV)
    A, SA, B_, SB = to_dev(qa), to_dev(sa), to_dev(qb), to_dev(sb)
    if c_mode == "inplace":
        d = to_dev(c, torch.float32).clone()
        cc = d
    elif c_mode == "separate":
        d = torch.full((G, M, N), float("nan"), dtype=dt, device=DEV)
        cc = to_dev(c, torch.float32)
    else:
        d = torch.full((G, M, N), float("nan"), dtype=dt, device=DEV)
        cc = None
    dg.dg_k_grouped_fp8_wgrad(A, SA, B_, SB, d, cc, ks, ks_dev, gran_k)
    dg.dg_sync_check()
    return d


def run_bf16(a, b, ks, out="f32", c=None, c_mode="none"):
    G, M, N = len(ks), a.shape[1], b.shape[1]
    dt = torch.float32 if out == "f32" else torch.bfloat16
    ks_dev = torch.tensor(ks, dtype=torch.int32, device=DEV)
    A, B_ = to_dev(a, torch.bfloat16), to_dev(b, torch.bfloat16)
    if c_mode == "inplace":
        d = to_dev(c, torch.float32).clone()
        cc = d
    elif c_mode == "separate":
        d = torch.full((G, M, N), float("nan"), dtype=dt, device=DEV)
        cc = to_dev(c, torch.float32)
    else:
        d = torch.full((G, M, N), float("nan"), dtype=dt, device=DEV)
        cc = None
    dg.dg_k_grouped_bf16_wgrad(A, B_, d, cc, ks, ks_dev)
    dg.dg_sync_check()
    return d


def assert_close(d_gpu, D, S, out="f32", what=""):
    got = d_gpu.float().cpu().double().numpy() if isinstance(d_gpu, torch.Tensor) else d_gpu
    bound = oracle.fp32_bound(S) if out == "f32" else oracle.bf16_bound(D, S)
    err = np.abs(got - D)
    bad = ~(err <= bound)          # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; first "
            f"{[tuple(i) for i in idx]}: got {got[bad][:5]}, want {D[bad][:5]}, "
            f"bound {bound[bad][:5]}")
    return float(err.max()) if err.size else 0.0


def check_cast_bound(q, sf, X, B, gran_k=128, what="", max_ambiguous=1e-3):
    """A GPU column-block cast (q, sf) of values the GPU computes in FP32, against
    the oracle's float64 values X with elementwise error bounds B: each scale
    byte must be the scale rule's for some block maximum of values within
    X +- B, and each code the RNE E4M3 code of some value within the bound at
    that scale.  Where the bound admits one decision only (all but a small
    fraction of elements) this is an exact comparison."""
    from oracle.e4m3 import e4m3_decode, e4m3_encode
    from oracle.quant import scale_exponent
    q = q.cpu().numpy() if isinstance(q, torch.Tensor) else np.asarray(q)
    sf = sf.cpu().numpy() if isinstance(sf, torch.Tensor) else np.asarray(sf)
    T, C = X.shape
    nb = T // gran_k
    Xb, Bb = X.reshape(nb, gran_k, C), B.reshape(nb, gran_k, C)
    e_lo = scale_exponent(np.max(np.maximum(np.abs(Xb) - Bb, 0.0), axis=1))
    e_hi = scale_exponent(np.max(np.abs(Xb) + Bb, axis=1))
    e = sf.astype(np.int64) - 127
    bad = ~((e_lo <= e) & (e <= e_hi))
    assert not bad.any(), f"{what}: scale bytes out of bound at {np.argwhere(bad)[:5]}"
    scale = np.repeat(np.ldexp(1.0, -e), gran_k, axis=0)
    v_lo = e4m3_decode(e4m3_encode((X - B) * scale))
    v_hi = e4m3_decode(e4m3_encode((X + B) * scale))
    v = e4m3_decode(q)
    bad = ~((v_lo <= v) & (v <= v_hi))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} codes out of bound; first {i}: got "
                             f"{v[i]}, allowed [{v_lo[i]}, {v_hi[i]}], x = {X[i]} +- {B[i]}")
    amb = float(np.mean(v_lo != v_hi))
    assert amb <= max_ambiguous, f"{what}: {amb:.2e} of the codes are undecided by the bound"
    return amb
