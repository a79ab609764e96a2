"""GB300 (sm_103a) K-grouped FP8/BF16 MoE weight-gradient kernels (and the
M-grouped FP8 data gradient that pairs with them).

The product is the C-ABI library ``libdg.so`` (declared in
``include/dg_wgrad.h``) built from ``csrc/``; ``binding`` is its thin Python
binding with the same function names.
"""
from .binding import (  # noqa: F401
    DGError, DG_OK, DG_ERR_INVALID_ARG, DG_ERR_UNSUPPORTED, DG_ERR_CUDA, DG_ERR_TIMEOUT,
    dg_k_grouped_fp8_wgrad, dg_k_grouped_fp8_wgrad_nt, dg_k_grouped_bf16_wgrad,
    dg_m_grouped_fp8_dgrad, dg_m_grouped_fp8_dgrad_nt,
    dg_quant_transpose_fp8,
    dg_requant_transpose_fp8, dg_quant_moe_layout_fp8, dg_moe_layout_plan,
    dg_swiglu_backward_quant_fp8,
    dg_last_error, dg_sync_check, dg_version, lib,
)
