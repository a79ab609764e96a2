"""CPU oracle for the K-grouped FP8/BF16 weight-gradient path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, double-precision
restatement of what the path computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg may
import it.  The product (the CUDA library and its Python binding) never calls
it, and it shares no code with the CUDA path.

Modules
-------
``e4m3``   the OCP FP8 E4M3 ("e4m3fn") encoding, round-to-nearest-even, and the
           UE8M0 power-of-two scale byte.
``quant``  the column-block quantiser: one UE8M0 scale per column per
           ``gran_k``-token block, values cast to E4M3 (the transpose + cast
           step a weight-gradient GEMM needs); the forward pass's 1 x 128
           row-tile cast and its exact dequantisation (re-quantising stored
           FP8 activations); the MoE token layout (its plan from top-k
           routing, and the row gather with zero padding rows).
``swiglu`` the SwiGLU backward of a MoE expert (dh = [dg | du] and the
           recomputed activation a), cast by columns.
``wgrad``  the K-grouped GEMM ``D[e] = C[e] + A_e^T B_e`` with per-block
           scales, in float64, plus the tolerance budget ``S = sum |a b s|``.
``dgrad``  the M-grouped data gradient ``dx_e = dy_e W_e`` (the other GEMM of
           an expert's backward) with per-block scales along K, in float64.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against something other than itself (a library cast, exact rational
arithmetic, closed forms, invariants).  No function is "parity unpinned".
"""
from .e4m3 import e4m3_decode, e4m3_encode, ue8m0_to_float, E4M3_MAX  # noqa: F401
from .quant import (  # noqa: F401
    scale_exponent, quant_colblock, quant_rowtile, dequant_rowtile, requant_colblock,
    gather_rows, moe_layout_cast, moe_layout_plan,
)
from .swiglu import sigmoid, swiglu_backward, swiglu_backward_cast  # noqa: F401
from .wgrad import (  # noqa: F401
    dequant_colblock, kgrouped_fp8_wgrad, kgrouped_bf16_wgrad,
    kgrouped_fp8_wgrad_rows, kgrouped_bf16_wgrad_rows, expert_offsets,
    fp32_bound, bf16_bound,
)
from .dgrad import mgrouped_fp8_dgrad, mgrouped_fp8_dgrad_rows  # noqa: F401
