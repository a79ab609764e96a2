"""Seeded synthetic inputs for the K-grouped weight-gradient workloads.

This module only draws random numbers: expert token counts and raw operand
values.  It holds none of the method's arithmetic (no quantisation, no GEMM),
so that the CPU oracle and the CUDA path can both take their inputs from it
without sharing any computation.

Every workload is a MoE weight-gradient problem ``D[e] (+)= A_e^T B_e`` in the
shapes of the MoE layers the weight-gradient pages discuss (up/gate-proj and
down-proj of a 7168-wide model, a fine-grained BF16 case, and the full
cast-then-GEMM pipeline).  Counts follow a Zipf-skewed expert popularity, the
routing skew a MoE backward pass sees.

Draw order per workload (one ``torch.Generator`` seeded with the workload's
seed): counts, A, B, outlier masks, C.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    G: int
    M: int
    N: int
    sum_k: int
    kind: str                 # "fp8" | "bf16" | "pipeline"
    out_dtype: str            # "f32" | "bf16"
    accumulate: bool          # D += (C == D, in place)
    c_std: float = 0.0
    zipf_s: float = 1.2
    count_unit: int = 128     # tokens per multinomial draw (1 = token level)
    empty_frac: float = 0.0   # fraction of experts forced empty (bf16 case)
    outlier_p: float = 0.0
    outlier_mul: float = 1.0
    fixed_ks: Optional[tuple] = None
    gran_k: int = 128
    notes: str = field(default="")

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.sum_k


WORKLOADS = {
    # Tiny FP8 case: four experts, one empty, accumulated onto C in place.
    "fp8_tiny_g4": Workload("fp8_tiny_g4", 0, 4, 128, 256, 512, "fp8", "f32", True,
                            c_std=1.0, fixed_ks=(128, 0, 256, 128)),
    # MoE up/gate-proj wgrad: M = 2 x 2048 (gate + up), N = 7168 hidden.
    "moe_upgate_fp8_g32": Workload("moe_upgate_fp8_g32", 1, 32, 4096, 7168, 32768,
                                   "fp8", "f32", False),
    # Profiling-size up/gate case: same M, N and count law, 8 experts, 8192
    # tokens (output 0.94 GB, operands 92 MB: still well above L2).
    "moe_upgate_fp8_g8": Workload("moe_upgate_fp8_g8", 5, 8, 4096, 7168, 8192,
                                  "fp8", "f32", False),
    # MoE down-proj wgrad with 1% outliers x100, BF16 output.
    "moe_down_fp8_g32": Workload("moe_down_fp8_g32", 2, 32, 7168, 2048, 32768,
                                 "fp8", "bf16", False, outlier_p=0.01, outlier_mul=100.0),
    # Fine-grained BF16-input variant, token-level (unaligned) counts, ~30% empty.
    "bf16_fine_g256": Workload("bf16_fine_g256", 3, 256, 1024, 1024, 65536, "bf16", "f32",
                               True, c_std=0.1, zipf_s=1.5, count_unit=1, empty_frac=0.3),
    # Full pipeline: bf16 dY [T, 4096] and X [T, 7168] -> cast -> K-grouped FP8 GEMM.
    "pipeline_fp8_g64": Workload("pipeline_fp8_g64", 4, 64, 4096, 7168, 131072,
                                 "pipeline", "f32", True, c_std=0.01),
    # M-grouped data gradient of the up/gate projection: dx [T, 7168] =
    # dh [T, 4096] W[e] with W [32, 4096, 7168]; here M is the contraction
    # (h_out = 4096), N = h_in, sum_k the tokens.  Operands are E4M3 codes.
    "moe_upgate_dgrad_fp8_g32": Workload("moe_upgate_dgrad_fp8_g32", 6, 32, 4096, 7168, 32768,
                                         "dgrad", "bf16", False),
}


def zipf_popularity(G: int, s: float) -> torch.Tensor:
    """p_e proportional to (e+1)^-s, in expert order."""
    w = torch.arange(1, G + 1, dtype=torch.float64) ** (-s)
    return w / w.sum()


def expert_counts(w: Workload, gen: torch.Generator) -> list:
    """Per-expert token counts K_e, summing to ``w.sum_k``.

    Counts are drawn in units of ``w.count_unit`` tokens from a multinomial over
    Zipf(s) popularity.  For 128-token units at least one expert is left empty
    (the least popular one donates its blocks to expert 0 if none came out
    empty), so every FP8 workload exercises the empty-group path.  For the
    token-level case a seeded ``empty_frac`` of the experts get popularity 0.
    """
    if w.fixed_ks is not None:
        return list(w.fixed_ks)
    p = zipf_popularity(w.G, w.zipf_s)
    if w.empty_frac > 0:
        n_empty = int(round(w.empty_frac * w.G))
        dead = torch.randperm(w.G, generator=gen)[:n_empty]
        p = p.clone()
        p[dead] = 0.0
        p = p / p.sum()
    units = w.sum_k // w.count_unit
    draws = torch.multinomial(p.float(), units, replacement=True, generator=gen)
    cnt = torch.bincount(draws, minlength=w.G)
    if w.count_unit > 1 and int((cnt == 0).sum()) == 0:
        cnt[0] += cnt[w.G - 1]
        cnt[w.G - 1] = 0
    ks = [int(c) * w.count_unit for c in cnt]
    assert sum(ks) == w.sum_k
    return ks


def counts_for(name: str) -> list:
    w = WORKLOADS[name]
    gen = torch.Generator().manual_seed(w.seed)
    return expert_counts(w, gen)


def draw_operands(name: str, device: str = "cpu", rows_limit: Optional[int] = None):
    """Draw (ks, A_raw, B_raw, C) for a workload.

    A_raw is [sum_k, M], B_raw is [sum_k, N]: fp32 for the FP8 workloads (they
    are quantised afterwards by whichever side consumes them), bf16 for the
    BF16 and pipeline workloads.  C is fp32 [G, M, N] or None.

    ``device="cuda"`` draws on the GPU with a CUDA generator (fast, for timing
    runs; values differ from the CPU draw).  ``rows_limit`` is not supported for
    full-size parity (kept None there).
    """
    w = WORKLOADS[name]
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    ks = expert_counts(w, gen)
    if device != "cpu":
        gen = torch.Generator(device=device).manual_seed(w.seed)
    dt = torch.float32 if w.kind == "fp8" else torch.bfloat16
    sk = w.sum_k if rows_limit is None else rows_limit
    A = torch.randn(sk, w.M, generator=gen, device=device, dtype=torch.float32)
    B = torch.randn(sk, w.N, generator=gen, device=device, dtype=torch.float32)
    if w.outlier_p > 0:
        ma = torch.rand(sk, w.M, generator=gen, device=device) < w.outlier_p
        mb = torch.rand(sk, w.N, generator=gen, device=device) < w.outlier_p
        A = torch.where(ma, A * w.outlier_mul, A)
        B = torch.where(mb, B * w.outlier_mul, B)
    A = A.to(dt)
    B = B.to(dt)
    C = None
    if w.accumulate:
        C = torch.randn(w.G, w.M, w.N, generator=gen, device=device,
                        dtype=torch.float32) * w.c_std
    return ks, A, B, C


def random_codes(shape, gen: torch.Generator, device: str = "cpu") -> torch.Tensor:
    """Uniform random E4M3 bytes, the two NaN encodings (0x7F, 0xFF) replaced
    by 0x3C and 0xBC."""
    c = torch.randint(0, 256, shape, generator=gen, device=device, dtype=torch.uint8)
    nan = (c & 0x7F) == 0x7F
    return torch.where(nan, c ^ 0x43, c)


def draw_dgrad_operands(name: str, device: str = "cpu"):
    """Draw (ms, a, sfa, w, sfw) for an M-grouped data-gradient workload:
    a E4M3 [sum_m, K] with UE8M0 sfa [sum_m, K / gran_k] in [120, 136), w E4M3
    [G, K, N] with sfw [G, K / gran_k, N] in [112, 128), all uint8.  Token
    counts as ``expert_counts``.  ``device="cuda"`` draws on the GPU (values
    differ from the CPU draw)."""
    w = WORKLOADS[name]
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    ms = expert_counts(w, gen)
    if device != "cpu":
        gen = torch.Generator(device=device).manual_seed(w.seed)
    K, N, g = w.M, w.N, w.gran_k
    a = random_codes((w.sum_k, K), gen, device)
    sfa = torch.randint(120, 136, (w.sum_k, K // g), generator=gen, device=device,
                        dtype=torch.uint8)
    wt = random_codes((w.G, K, N), gen, device)
    sfw = torch.randint(112, 128, (w.G, K // g, N), generator=gen, device=device,
                        dtype=torch.uint8)
    return ms, a, sfa, wt, sfw


def random_counts(G: int, sum_blocks: int, unit: int, seed: int, empty: int = 0) -> list:
    """Uniform-random counts for small parity cases: ``sum_blocks`` units of
    ``unit`` tokens over G experts, with ``empty`` experts forced to zero."""
    gen = torch.Generator().manual_seed(seed)
    p = torch.ones(G, dtype=torch.float64)
    if empty:
        dead = torch.randperm(G, generator=gen)[:empty]
        p[dead] = 0.0
    p = p / p.sum()
    if sum_blocks == 0:
        return [0] * G
    draws = torch.multinomial(p.float(), sum_blocks, replacement=True, generator=gen)
    cnt = torch.bincount(draws, minlength=G)
    return [int(c) * unit for c in cnt]


def randn(shape, seed: int, dtype=torch.float32, std: float = 1.0) -> torch.Tensor:
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=gen, dtype=torch.float32) * std).to(dtype)
