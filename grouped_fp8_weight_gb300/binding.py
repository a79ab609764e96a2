"""Thin Python binding of the C ABI in ``include/dg_wgrad.h``.

Argument marshalling only: every function checks shapes and dtypes of torch
tensors, passes their device pointers and the current CUDA stream to the
library of the same name, and raises ``DGError`` on a non-OK status.  All
computation happens in the CUDA kernels of ``libdg.so``; there is no fallback.
If the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdg.so")

DG_OK, DG_ERR_INVALID_ARG, DG_ERR_UNSUPPORTED, DG_ERR_CUDA, DG_ERR_TIMEOUT = range(5)
DG_F32, DG_BF16 = 0, 1
DG_TOKEN_MAJOR, DG_CHANNEL_MAJOR = 0, 1
DG_MAX_GROUPS = 1024
STATUS_NAMES = {0: "DG_OK", 1: "DG_ERR_INVALID_ARG", 2: "DG_ERR_UNSUPPORTED",
                3: "DG_ERR_CUDA", 4: "DG_ERR_TIMEOUT"}

# Every symbol the header declares, with (restype, argtypes).
_VP, _U8P, _FP, _IP = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
_I, _I64 = ctypes.c_int, ctypes.c_int64
SIGNATURES = {
    "dg_k_grouped_fp8_wgrad": (_I, [_VP, _U8P, _VP, _U8P, _VP, _I, _FP, _I, _I, _I, _I64,
                                    _IP, _IP, _I, _VP]),
    "dg_k_grouped_fp8_wgrad_noalloc": (_I, [_VP, _U8P, _VP, _U8P, _VP, _I, _FP, _I, _I, _I,
                                            _I64, _IP, _IP, _I, _VP]),
    "dg_k_grouped_fp8_wgrad_nt": (_I, [_VP, _U8P, _VP, _U8P, _VP, _I, _FP, _I, _I, _I, _I64,
                                       _IP, _IP, _I, _VP]),
    "dg_k_grouped_bf16_wgrad": (_I, [_VP, _VP, _VP, _I, _FP, _I, _I, _I, _I64, _IP, _IP, _VP]),
    "dg_m_grouped_fp8_dgrad": (_I, [_VP, _U8P, _VP, _U8P, _VP, _I, _I, _I, _I, _I64, _IP, _IP,
                                    _I, _VP]),
    "dg_m_grouped_fp8_dgrad_nt": (_I, [_VP, _U8P, _VP, _U8P, _VP, _I, _I, _I, _I, _I64, _IP,
                                       _IP, _I, _VP]),
    "dg_quant_transpose_fp8": (_I, [_VP, _I64, _I, _VP, _U8P, _I, _I, _VP]),
    "dg_requant_transpose_fp8": (_I, [_VP, _U8P, _I64, _I, _VP, _U8P, _I, _I, _VP]),
    "dg_quant_moe_layout_fp8": (_I, [_VP, _U8P, _I64, _I, _IP, _I64, _VP, _U8P, _I, _I, _VP]),
    "dg_moe_layout_plan": (_I, [_IP, _I64, _I, _I, _I, _IP, _IP, _IP, _I64, _VP]),
    "dg_swiglu_backward_quant_fp8": (_I, [_VP, _VP, _I64, _I, _VP, _U8P, _VP, _U8P, _I, _VP]),
    "dg_last_error": (ctypes.c_char_p, []),
    "dg_sync_check": (_I, [_VP]),
    "dg_version": (_I, []),
}


class DGError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None


def lib():
    """The loaded ``libdg.so`` with argument types set (raises if not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run grouped_fp8_weight_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status: int):
    if status != DG_OK:
        raise DGError(status, lib().dg_last_error().decode())


_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, t=None):
    """The CUDA stream handle to launch on: `stream`'s, or the current stream of
    tensor t's device (of the current device when t is None)."""
    if stream is None:
        if _RAW_STREAM is not None:
            idx = t.device.index if t is not None and t.device.index is not None \
                else torch.cuda.current_device()
            return _RAW_STREAM(idx)
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


_KS_CACHE = {}


def _ks_host(ks):
    """ks as a ctypes int array (the host copy the C call reads), with its
    length.  Arrays of recently seen count lists are reused (they are only
    read by the call)."""
    if isinstance(ks, torch.Tensor):
        ks = ks.tolist()
    key = tuple(ks)
    hit = _KS_CACHE.get(key)
    if hit is not None:
        return hit
    arr = (ctypes.c_int * max(1, len(key)))(*[int(k) for k in key])
    if len(_KS_CACHE) >= 64:
        _KS_CACHE.clear()
    _KS_CACHE[key] = (arr, len(key))
    return arr, len(key)


def _dptr(t):
    return None if t is None else t.data_ptr()


def _need(t, dtype, name, ndim):
    if t.dtype != dtype or t.dim() != ndim or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor of rank {ndim}, "
                         f"got {t.dtype} {tuple(t.shape)}")


def dg_k_grouped_fp8_wgrad(a, sfa, b, sfb, d, c, ks_host, ks_dev, gran_k: int = 128,
                           stream=None):
    """D[e] (+)= A_e^T B_e with E4M3 operands and UE8M0 block scales.

    a: uint8/float8_e4m3fn [sum_k, M]; sfa: uint8 [sum_k/gran_k, M]; b, sfb
    likewise with N; d: float32 or bfloat16 [G, M, N]; c: None, d itself (in
    place), or a separate float32 [G, M, N]; ks_host: G ints; ks_dev: int32
    CUDA tensor [G].
    """
    a8 = a.view(torch.uint8) if a.dtype != torch.uint8 else a
    b8 = b.view(torch.uint8) if b.dtype != torch.uint8 else b
    _need(a8, torch.uint8, "a", 2)
    _need(b8, torch.uint8, "b", 2)
    _need(sfa, torch.uint8, "sfa", 2)
    _need(sfb, torch.uint8, "sfb", 2)
    if d.dim() != 3 or d.dtype not in (torch.float32, torch.bfloat16) or not d.is_contiguous():
        raise ValueError("d: expected contiguous float32/bfloat16 [G, M, N]")
    G, M, N = d.shape
    if a8.shape[1] != M or b8.shape[1] != N or a8.shape[0] != b8.shape[0]:
        raise ValueError("operand shapes do not match d")
    if c is not None and c is not d:
        _need(c, torch.float32, "c", 3)
        if tuple(c.shape) != tuple(d.shape):
            raise ValueError("c must have d's shape")
    _need(ks_dev, torch.int32, "ks_dev", 1)
    kh, g = _ks_host(ks_host)
    if g != G or ks_dev.numel() != G:
        raise ValueError("ks must have G entries")
    _check(lib().dg_k_grouped_fp8_wgrad(
        _dptr(a8), _dptr(sfa), _dptr(b8), _dptr(sfb), _dptr(d),
        DG_BF16 if d.dtype == torch.bfloat16 else DG_F32,
        _dptr(c), G, M, N, a8.shape[0], kh, _dptr(ks_dev), gran_k, _stream(stream, d)))


def dg_k_grouped_fp8_wgrad_nt(a, sfa, b, sfb, d, c, ks_host, ks_dev, gran_k: int = 128,
                              stream=None):
    """As dg_k_grouped_fp8_wgrad with K-major operands a [M, sum_k], b [N, sum_k]."""
    a8 = a.view(torch.uint8) if a.dtype != torch.uint8 else a
    b8 = b.view(torch.uint8) if b.dtype != torch.uint8 else b
    _need(a8, torch.uint8, "a", 2)
    _need(b8, torch.uint8, "b", 2)
    _need(sfa, torch.uint8, "sfa", 2)
    _need(sfb, torch.uint8, "sfb", 2)
    if d.dim() != 3 or d.dtype not in (torch.float32, torch.bfloat16) or not d.is_contiguous():
        raise ValueError("d: expected contiguous float32/bfloat16 [G, M, N]")
    G, M, N = d.shape
    if a8.shape[0] != M or b8.shape[0] != N or a8.shape[1] != b8.shape[1]:
        raise ValueError("operand shapes do not match d")
    if c is not None and c is not d:
        _need(c, torch.float32, "c", 3)
        if tuple(c.shape) != tuple(d.shape):
            raise ValueError("c must have d's shape")
    _need(ks_dev, torch.int32, "ks_dev", 1)
    kh, g = _ks_host(ks_host)
    if g != G or ks_dev.numel() != G:
        raise ValueError("ks must have G entries")
    _check(lib().dg_k_grouped_fp8_wgrad_nt(
        _dptr(a8), _dptr(sfa), _dptr(b8), _dptr(sfb), _dptr(d),
        DG_BF16 if d.dtype == torch.bfloat16 else DG_F32,
        _dptr(c), G, M, N, a8.shape[1], kh, _dptr(ks_dev), gran_k, _stream(stream, d)))


def dg_k_grouped_bf16_wgrad(a, b, d, c, ks_host, ks_dev, stream=None):
    """D[e] (+)= A_e^T B_e with BF16 operands (any per-expert token counts)."""
    _need(a, torch.bfloat16, "a", 2)
    _need(b, torch.bfloat16, "b", 2)
    if d.dim() != 3 or d.dtype not in (torch.float32, torch.bfloat16) or not d.is_contiguous():
        raise ValueError("d: expected contiguous float32/bfloat16 [G, M, N]")
    G, M, N = d.shape
    if a.shape[1] != M or b.shape[1] != N or a.shape[0] != b.shape[0]:
        raise ValueError("operand shapes do not match d")
    if c is not None and c is not d:
        _need(c, torch.float32, "c", 3)
    _need(ks_dev, torch.int32, "ks_dev", 1)
    kh, g = _ks_host(ks_host)
    if g != G or ks_dev.numel() != G:
        raise ValueError("ks must have G entries")
    _check(lib().dg_k_grouped_bf16_wgrad(
        _dptr(a), _dptr(b), _dptr(d), DG_BF16 if d.dtype == torch.bfloat16 else DG_F32,
        _dptr(c), G, M, N, a.shape[0], kh, _dptr(ks_dev), _stream(stream, d)))


def dg_m_grouped_fp8_dgrad(a, sfa, w, sfw, d, ms_host, ms_dev, gran_k: int = 128,
                           stream=None, w_kmajor: bool = False):
    """D[t] = dy[t] W_e for the token rows t of expert e (M-grouped, contiguous).

    a: E4M3 [sum_m, K] (or uint8 codes), sfa: uint8 [sum_m, K / gran_k];
    w: E4M3 [G, K, N], sfw: uint8 [G, K / gran_k, N]; d: float32 or bfloat16
    [sum_m, N]; ms_host: G token counts (multiples of 128), ms_dev the same as
    an int32 CUDA tensor.
    """
    a8 = a.view(torch.uint8) if a.dtype != torch.uint8 else a
    w8 = w.view(torch.uint8) if w.dtype != torch.uint8 else w
    _need(a8, torch.uint8, "a", 2)
    _need(w8, torch.uint8, "w", 3)
    _need(sfa, torch.uint8, "sfa", 2)
    _need(sfw, torch.uint8, "sfw", 3)
    if d.dim() != 2 or d.dtype not in (torch.float32, torch.bfloat16) or not d.is_contiguous():
        raise ValueError("d: expected contiguous float32/bfloat16 [sum_m, N]")
    if w_kmajor:
        G, N, K = w8.shape
    else:
        G, K, N = w8.shape
    sum_m = a8.shape[0]
    if a8.shape[1] != K or tuple(d.shape) != (sum_m, N):
        raise ValueError("operand shapes do not match: a [sum_m, K], w [G, K, N] (or [G, N, K] "
                         "K-major), d [sum_m, N]")
    if tuple(sfa.shape) != (sum_m, K // gran_k) or tuple(sfw.shape) != (G, K // gran_k, N):
        raise ValueError("scale shapes: sfa [sum_m, K / gran_k], sfw [G, K / gran_k, N]")
    _need(ms_dev, torch.int32, "ms_dev", 1)
    mh, g = _ks_host(ms_host)
    if g != G or ms_dev.numel() != G:
        raise ValueError("ms must have G entries")
    fn = lib().dg_m_grouped_fp8_dgrad_nt if w_kmajor else lib().dg_m_grouped_fp8_dgrad
    _check(fn(_dptr(a8), _dptr(sfa), _dptr(w8), _dptr(sfw), _dptr(d),
              DG_BF16 if d.dtype == torch.bfloat16 else DG_F32,
              G, K, N, sum_m, mh, _dptr(ms_dev), gran_k, _stream(stream)))


def dg_m_grouped_fp8_dgrad_nt(a, sfa, w, sfw, d, ms_host, ms_dev, gran_k: int = 128,
                              stream=None):
    """As dg_m_grouped_fp8_dgrad with the weights stored K-major: w [G, N, K]
    (scales still sfw [G, K / gran_k, N])."""
    dg_m_grouped_fp8_dgrad(a, sfa, w, sfw, d, ms_host, ms_dev, gran_k, stream, w_kmajor=True)


def dg_quant_transpose_fp8(x, q, sf, layout: str = "token", gran_k: int = 128, stream=None):
    """Column-block E4M3 cast of bf16 x [T, C] into q ([T, C] or [C, T]) and sf [T/gran_k, C]."""
    _need(x, torch.bfloat16, "x", 2)
    q8 = q.view(torch.uint8) if q.dtype != torch.uint8 else q
    _need(q8, torch.uint8, "q", 2)
    _need(sf, torch.uint8, "sf", 2)
    T, C = x.shape
    want = (T, C) if layout == "token" else (C, T)
    if tuple(q8.shape) != want or tuple(sf.shape) != (T // gran_k, C):
        raise ValueError("q / sf shapes do not match x")
    _check(lib().dg_quant_transpose_fp8(
        _dptr(x), T, C, _dptr(q8), _dptr(sf),
        DG_TOKEN_MAJOR if layout == "token" else DG_CHANNEL_MAJOR, gran_k, _stream(stream)))


def _layout(layout):
    if layout not in ("token", "channel"):
        raise ValueError("layout must be 'token' or 'channel'")
    return DG_TOKEN_MAJOR if layout == "token" else DG_CHANNEL_MAJOR


def _check_out(q8, sf, T, C, layout, gran_k):
    _need(q8, torch.uint8, "q", 2)
    _need(sf, torch.uint8, "sf", 2)
    want = (T, C) if layout == "token" else (C, T)
    if tuple(q8.shape) != want or tuple(sf.shape) != (T // gran_k, C):
        raise ValueError("q / sf shapes do not match the output rows")


def dg_requant_transpose_fp8(q_in, sf_in, q, sf, layout: str = "token", gran_k: int = 128,
                             stream=None):
    """Stored E4M3 q_in [T, C] with 1 x 128 scales sf_in [T, C/128] (UE8M0) ->
    column-block E4M3 q ([T, C] or [C, T]) and sf [T/gran_k, C]."""
    qi = q_in.view(torch.uint8) if q_in.dtype != torch.uint8 else q_in
    _need(qi, torch.uint8, "q_in", 2)
    _need(sf_in, torch.uint8, "sf_in", 2)
    T, C = qi.shape
    if tuple(sf_in.shape) != (T, C // 128):
        raise ValueError("sf_in must be [T, C / 128]")
    q8 = q.view(torch.uint8) if q.dtype != torch.uint8 else q
    _check_out(q8, sf, T, C, layout, gran_k)
    _check(lib().dg_requant_transpose_fp8(
        _dptr(qi), _dptr(sf_in), T, C, _dptr(q8), _dptr(sf), _layout(layout), gran_k,
        _stream(stream)))


def dg_quant_moe_layout_fp8(x, src_rows, q, sf, x_sf=None, layout: str = "token",
                            gran_k: int = 128, stream=None):
    """Column-block cast of the MoE-layout rows x[src_rows] (-1: a zero row).
    x: bf16 [T_src, C], or E4M3 codes [T_src, C] with x_sf uint8 [T_src, C/128];
    src_rows: int32 CUDA tensor [T]; q ([T, C] or [C, T]), sf [T/gran_k, C]."""
    if x_sf is None:
        _need(x, torch.bfloat16, "x", 2)
        xp = x
    else:
        xp = x.view(torch.uint8) if x.dtype != torch.uint8 else x
        _need(xp, torch.uint8, "x", 2)
        _need(x_sf, torch.uint8, "x_sf", 2)
        if tuple(x_sf.shape) != (xp.shape[0], xp.shape[1] // 128):
            raise ValueError("x_sf must be [T_src, C / 128]")
    _need(src_rows, torch.int32, "src_rows", 1)
    T_src, C = xp.shape
    T = src_rows.numel()
    q8 = q.view(torch.uint8) if q.dtype != torch.uint8 else q
    _check_out(q8, sf, T, C, layout, gran_k)
    _check(lib().dg_quant_moe_layout_fp8(
        _dptr(xp), _dptr(x_sf), T_src, C, _dptr(src_rows), T, _dptr(q8), _dptr(sf),
        _layout(layout), gran_k, _stream(stream)))


def dg_moe_layout_plan(topk_idx, G: int, align: int = 128, with_pairs: bool = False,
                       stream=None):
    """The MoE token layout from routing topk_idx (int32 CUDA [T_tok, topk],
    -1 = unused slot).  Returns device tensors (ks [G], src_rows [cap], and
    pair_rows [cap] if with_pairs), cap = T_tok * topk + G * (align - 1); rows
    past the layout's end are -1 (the layout has ks.sum() rows)."""
    _need(topk_idx, torch.int32, "topk_idx", 2)
    T_tok, topk = topk_idx.shape
    cap = T_tok * topk + G * (align - 1)
    dev = topk_idx.device
    ks = torch.empty(G, dtype=torch.int32, device=dev)
    src = torch.empty(cap, dtype=torch.int32, device=dev)
    pair = torch.empty(cap, dtype=torch.int32, device=dev) if with_pairs else None
    _check(lib().dg_moe_layout_plan(_dptr(topk_idx), T_tok, topk, G, align, _dptr(ks),
                                    _dptr(src), _dptr(pair), cap, _stream(stream)))
    return (ks, src, pair) if with_pairs else (ks, src)


def dg_swiglu_backward_quant_fp8(h, da, q_dh, sf_dh, q_a=None, sf_a=None, gran_k: int = 128,
                                 stream=None):
    """SwiGLU backward fused with the column-block cast: h bf16 [T, 2I] = [g | u],
    da bf16 [T, I] -> q_dh [T, 2I] / sf_dh [T/gran_k, 2I] (dh = [dg | du]) and,
    if given, q_a [T, I] / sf_a [T/gran_k, I] (a = silu(g) * u)."""
    _need(h, torch.bfloat16, "h", 2)
    _need(da, torch.bfloat16, "da", 2)
    T, I2 = h.shape
    I = I2 // 2
    if I2 % 2 or tuple(da.shape) != (T, I):
        raise ValueError("h must be [T, 2I] and da [T, I]")
    q8 = q_dh.view(torch.uint8) if q_dh.dtype != torch.uint8 else q_dh
    _check_out(q8, sf_dh, T, I2, "token", gran_k)
    qa8 = None
    if q_a is not None:
        qa8 = q_a.view(torch.uint8) if q_a.dtype != torch.uint8 else q_a
        _check_out(qa8, sf_a, T, I, "token", gran_k)
    _check(lib().dg_swiglu_backward_quant_fp8(
        _dptr(h), _dptr(da), T, I, _dptr(q8), _dptr(sf_dh), _dptr(qa8), _dptr(sf_a), gran_k,
        _stream(stream)))


def dg_last_error() -> str:
    return lib().dg_last_error().decode()


def dg_sync_check(stream=None):
    _check(lib().dg_sync_check(_stream(stream)))


def dg_version() -> int:
    return lib().dg_version()
