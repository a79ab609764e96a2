"""Throughput of the K-grouped FP8 weight-gradient hot path on GB300.

Default workload: the MoE up/gate-proj weight gradient (G=32 experts,
M=4096, N=7168, sum K=32768 routed tokens with Zipf(1.2) counts in 128-token
units, E4M3 operands with UE8M0 1x128 column-block scales, FP32 output).  One
step = one dg_k_grouped_fp8_wgrad call over inputs resident in HBM; the metric
is 2*M*N*sum(K) / step time in TFLOP/s.

The same JSON line also carries:
  roofline      the GEMM kernel's algorithmic bytes / CUDA-event launch time
                against the measured HBM copy bandwidth, plus its tensor
                fraction against the dense FP8 peak, measured in the same run
                (cuBLASLt e4m3 8192^3 through torch._scaled_mm, best of 10);
  configs       every workload of the path, each device-resident and timed
                on its own: the tiny in-place case (see `tiny`), the up/gate
                headline, the down-projection (BF16 output, 1 % outliers),
                the fine-grained BF16 case (D += in place) and the pipeline
                (the cast of dY [131072, 4096] and X [131072, 7168], the
                in-place GEMM onto C, and cast + GEMM), each with its roofline;
  pipeline      the cast-inclusive step (BF16 dY, X -> dg_quant_transpose_fp8
                x2 -> GEMM) on the headline's shapes, and the cast's roofline;
  nt            the same GEMM with K-major operands (dg_k_grouped_fp8_wgrad_nt)
                fed by the channel-major cast;
  casts         the re-quantisation of stored FP8 operands, the cast fused
                with the MoE layout and the cast fused with the SwiGLU
                backward, each against the HBM roofline;
  dgrad         the M-grouped FP8 data gradient of the up/gate projection
                (dg_m_grouped_fp8_dgrad, and _nt with K-major weights)
                against the FP8 peak;
  tiny          host and device time per call of the tiny in-place workload;
  e2e           the same metric through the C ABI with pinned host buffers:
                H2D of the step's operands and D2H of the result D in the
                timed region (each step's D2H overlapping the next step's
                H2D and call, two device results alternating);
  cpu_baseline  the float64 CPU oracle timed on a bounded sample;
  clocks        nvidia-smi samples taken during warm-up + timed region.

``--impl reference`` times the float64 oracle (the reference arm: the pages
hold no runnable code) on a bounded sample of the same workload.  Under torchrun each rank runs its own
replica of the workload (weak scaling, no data-path collective); rank 0
prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from grouped_fp8_weight_gb300 import workloads  # noqa: E402

METRIC = "K-grouped FP8 wgrad TFLOP/s (2·M·N·ΣK_i) and % of GB300 dense FP8 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CSRC = os.path.join(ROOT, "grouped_fp8_weight_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


GEMM_SOURCES = ("ptx.cuh", "wgrad_params.h", "wgrad_kernel.cuh", "wgrad_fp8.cu")


def kernel_source_sha() -> str:
    """Hash of the FP8 GEMM kernel's sources (traffic figures expire with it)."""
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def fp8_tiles(M: int, N: int) -> str:
    """Tile widths of the FP8 weight gradient for an M x N output:
    the kernel's N is N, or M when its tiles are transposed (N % 224 != 0 and
    M % 224 == 0); a kernel N that is a multiple of 1792 (of 256 and of 224)
    runs mixed 256 / 224-column tiles unless DG_MIXED_TILES=0."""
    nk = M if (N % 224 and M % 224 == 0) else N
    if nk % 1792 == 0 and os.environ.get("DG_MIXED_TILES", "") != "0":
        return "256 | 224 mixed"
    return "224" if nk % 224 == 0 else "128"


def recorded_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes for (kernel, workload) from the committed ncu
    summary, or None if absent or taken on a different kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    sha = kernel_source_sha()
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload and parts[2] == sha:
                return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 50 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": rows[0][1],
                "reasons": reasons, "samples": len(rows)}


def measure_fp8_peak(dev, sustained_s: float = 0.0):
    """Dense FP8 (E4M3 x E4M3 -> BF16, FP32 accumulation) throughput of
    cuBLASLt through torch._scaled_mm on 8192^3 with per-tensor scales: the
    best of 10 timed calls (burst) and, if sustained_s > 0, the mean rate of
    back-to-back calls over that many seconds (sustained).  This is the
    library's dense FP8 rate on this GPU, the denominator of every FP8
    tensor fraction."""
    n = 8192
    gen = torch.Generator(device=dev).manual_seed(7)
    a = torch.randn(n, n, generator=gen, device=dev).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, generator=gen, device=dev).to(torch.float8_e4m3fn).t()
    one = torch.ones((), dtype=torch.float32, device=dev)

    def mm():
        return torch._scaled_mm(a, b, one, one, out_dtype=torch.bfloat16)

    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        mm()
        e.record()
        e.synchronize()
        best = min(best, s.elapsed_time(e))
    flops = 2.0 * n ** 3
    out = {"burst_tflops": flops / (best * 1e-3) / 1e12, "shape": [n, n, n],
           "how": "torch._scaled_mm e4m3 x e4m3 -> bf16, per-tensor scales, best of 10"}
    if sustained_s > 0:
        calls, t_ms = 0, 0.0
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        s.record()
        while time.perf_counter() - t0 < sustained_s:
            for _ in range(20):
                mm()
            calls += 20
            torch.cuda.synchronize()
        e.record()
        e.synchronize()
        t_ms = s.elapsed_time(e)
        out["sustained_tflops"] = calls * flops / (t_ms * 1e-3) / 1e12
        out["sustained_seconds"] = t_ms / 1e3
    del a, b
    return out


def make_inputs(w, dev):
    """Operands for the workload, built on the device: BF16 N(0, 1) draws cast
    by the library's own column-block quantiser (dg_quant_transpose_fp8)."""
    import grouped_fp8_weight_gb300 as dg
    ks = workloads.counts_for(w.name)
    gen = torch.Generator(device=dev).manual_seed(w.seed)
    a_raw = torch.randn(w.sum_k, w.M, generator=gen, device=dev).to(torch.bfloat16)
    b_raw = torch.randn(w.sum_k, w.N, generator=gen, device=dev).to(torch.bfloat16)
    qa = torch.empty(w.sum_k, w.M, dtype=torch.uint8, device=dev)
    sa = torch.empty(w.sum_k // 128, w.M, dtype=torch.uint8, device=dev)
    qb = torch.empty(w.sum_k, w.N, dtype=torch.uint8, device=dev)
    sb = torch.empty(w.sum_k // 128, w.N, dtype=torch.uint8, device=dev)
    dg.dg_quant_transpose_fp8(a_raw, qa, sa)
    dg.dg_quant_transpose_fp8(b_raw, qb, sb)
    torch.cuda.synchronize()
    return ks, a_raw, b_raw, qa, sa, qb, sb


def algorithmic_bytes(w, ks):
    """Bytes the GEMM must move: operands and scales once, D written once
    (read too when accumulating in place)."""
    sk = sum(ks)
    ops = sk * (w.M + w.N) + (sk // 128) * (w.M + w.N)
    d_bytes = w.G * w.M * w.N * (4 if w.out_dtype == "f32" else 2)
    return ops + d_bytes * (2 if w.accumulate else 1)


def time_events(fn, steps, stream):
    """Mean ms of fn() over `steps` launches, CUDA events on `stream`."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / steps


def moe_layout_rows(ks, t_tok: int, seed: int) -> np.ndarray:
    """Source token of every row of the expert layout: expert e's K_e rows take
    K_e distinct tokens of t_tok, drawn at random and kept in token order."""
    rng = np.random.default_rng(seed)
    rows = [np.sort(rng.choice(t_tok, size=k, replace=False)) for k in ks if k > 0]
    return np.concatenate(rows).astype(np.int32)


def measure_casts(w, ks, dev, stream, pk, steps):
    """The other casts of the path on the workload's operand shapes, each
    against the HBM roofline: re-quantising stored FP8 (1 x 128 tiles, random
    codes and scale bytes) of dY [sum_k, M] and X [sum_k, N]; the BF16 cast of
    X fused with the MoE layout (each expert's rows gathered from sum_k / 2
    tokens), and the same from stored E4M3 rows; and the SwiGLU backward fused with the cast of dh [sum_k, M] and
    of the activation [sum_k, M / 2]."""
    import grouped_fp8_weight_gb300 as dg
    gen = torch.Generator(device=dev).manual_seed(w.seed + 100)
    out = {}
    bufs = []
    for C in (w.M, w.N):
        q_in = torch.randint(0, 256, (w.sum_k, C), generator=gen, device=dev, dtype=torch.uint8)
        q_in[(q_in & 0x7F) == 0x7F] = 0x7E
        sf_in = torch.randint(110, 140, (w.sum_k, C // 128), generator=gen, device=dev,
                              dtype=torch.uint8)
        bufs.append((q_in, sf_in, torch.empty_like(q_in),
                     torch.empty(w.sum_k // 128, C, dtype=torch.uint8, device=dev)))

    def requant():
        for q_in, sf_in, q, sf in bufs:
            dg.dg_requant_transpose_fp8(q_in, sf_in, q, sf)

    for _ in range(3):
        requant()
    ms = time_events(requant, steps, stream)
    nb = sum(w.sum_k * C * 2 + 2 * w.sum_k * C // 128 for C in (w.M, w.N))
    out["requant"] = {"ms": ms, "kernel": "requant_tm_kernel<128> (e4m3 1x128 source, token-major)",
                      "launches_per_step": 2, "bound": "hbm",
                      "achieved": nb / (ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                      "frac": nb / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], "algorithmic_bytes": nb}
    del bufs

    t_tok = w.sum_k // 2
    src_h = moe_layout_rows(ks, t_tok, w.seed + 101)
    uniq = int(np.unique(src_h).size)        # source rows read at least once
    src = torch.from_numpy(src_h).to(dev)
    x = torch.randn(t_tok, w.N, generator=gen, device=dev).to(torch.bfloat16)
    q = torch.empty(w.sum_k, w.N, dtype=torch.uint8, device=dev)
    sf = torch.empty(w.sum_k // 128, w.N, dtype=torch.uint8, device=dev)

    def layout_cast():
        dg.dg_quant_moe_layout_fp8(x, src, q, sf)

    for _ in range(3):
        layout_cast()
    ms = time_events(layout_cast, steps, stream)
    # each distinct source row read once (a row gathered into several experts'
    # slices is re-read from L2), each output row written once
    nb = uniq * w.N * 2 + w.sum_k * w.N + w.sum_k * 4 + (w.sum_k // 128) * w.N
    out["moe_layout"] = {"ms": ms, "kernel": "gather_cast_kernel<128> (rows by TMA gather4 and cp.async, token-major)",
                         "launches_per_step": 1, "source_tokens": t_tok, "rows": w.sum_k,
                         "distinct_source_rows": uniq,
                         "bound": "hbm", "achieved": nb / (ms * 1e-3) / 1e9,
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": nb / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], "algorithmic_bytes": nb}
    del x

    # the same layout from stored E4M3 rows with their 1 x 128 scales
    # (re-quantised while gathered)
    x8 = torch.randint(0, 256, (t_tok, w.N), generator=gen, device=dev, dtype=torch.uint8)
    x8[(x8 & 0x7F) == 0x7F] = 0x7E
    x8_sf = torch.randint(110, 140, (t_tok, w.N // 128), generator=gen, device=dev,
                          dtype=torch.uint8)

    def layout_requant():
        dg.dg_quant_moe_layout_fp8(x8, src, q, sf, x8_sf)

    for _ in range(3):
        layout_requant()
    ms = time_events(layout_requant, steps, stream)
    nb = (uniq * (w.N + w.N // 128) + w.sum_k * w.N + w.sum_k * 4 +
          (w.sum_k // 128) * w.N)
    out["moe_layout_fp8"] = {"ms": ms,
                             "kernel": "requant_tm_kernel<128, gather> (e4m3 1x128 source rows, token-major)",
                             "launches_per_step": 1, "source_tokens": t_tok, "rows": w.sum_k,
                             "distinct_source_rows": uniq,
                             "bound": "hbm", "achieved": nb / (ms * 1e-3) / 1e9,
                             "peak": pk["hbm_gbs"], "unit": "GB/s",
                             "frac": nb / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                             "algorithmic_bytes": nb}
    del x8, x8_sf, q, sf, src

    # SwiGLU backward fused with the cast: h = [g | u] [sum_k, M] and da
    # [sum_k, M/2] (BF16) -> dh = [dg | du] (the A operand, [sum_k, M]) and the
    # recomputed activation a [sum_k, M/2], both cast by columns.
    T, I = w.sum_k, w.M // 2
    h = torch.randn(T, 2 * I, generator=gen, device=dev).to(torch.bfloat16)
    da = torch.randn(T, I, generator=gen, device=dev).to(torch.bfloat16)
    q = torch.empty(T, 2 * I, dtype=torch.uint8, device=dev)
    sf = torch.empty(T // 128, 2 * I, dtype=torch.uint8, device=dev)
    qa = torch.empty(T, I, dtype=torch.uint8, device=dev)
    sfa = torch.empty(T // 128, I, dtype=torch.uint8, device=dev)

    def swiglu_cast():
        dg.dg_swiglu_backward_quant_fp8(h, da, q, sf, qa, sfa)

    for _ in range(3):
        swiglu_cast()
    ms = time_events(swiglu_cast, steps, stream)
    nb = T * I * (2 * 2 + 2) + T * I * (2 + 1) + (T // 128) * I * 3
    out["swiglu"] = {"ms": ms, "kernel": "swiglu_bwd_cast_kernel<128, with a>",
                     "launches_per_step": 1, "T": T, "I": I, "bound": "hbm",
                     "achieved": nb / (ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": nb / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], "algorithmic_bytes": nb}
    return out


def measure_tiny(dev, stream, steps):
    """Latency of the tiny in-place workload (G = 4, M = 128, N = 256,
    ks = [128, 0, 256, 128], D += A^T B): host time per call (validation,
    planning, tensor maps, two launches; calls issued back to back) and device
    time per call (CUDA events over the same back-to-back calls)."""
    import time
    import grouped_fp8_weight_gb300 as dg
    w = workloads.WORKLOADS["fp8_tiny_g4"]
    ks, _, _, qa, sa, qb, sb = make_inputs(w, dev)
    ks_dev = torch.tensor(ks, dtype=torch.int32, device=dev)
    d = torch.zeros(w.G, w.M, w.N, dtype=torch.float32, device=dev)

    def call():
        dg.dg_k_grouped_fp8_wgrad(qa, sa, qb, sb, d, d, ks, ks_dev, 128)

    for _ in range(10):
        call()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        call()
    host_us = (time.perf_counter() - t0) / steps * 1e6
    torch.cuda.synchronize()
    dev_ms = time_events(call, steps, stream)
    dg.dg_sync_check()
    return {"workload": w.name, "host_us_per_call": host_us, "device_us_per_call": dev_ms * 1e3,
            "launches_per_call": 2, "flops": w.flops,
            "note": "back-to-back calls; the device time includes the scale-pack launch"}


def measure_dgrad(dev, stream, pk, steps, fp8p):
    """The M-grouped FP8 data gradient of the up/gate projection (dx = dh W_e,
    K = 4096, N = 7168, the headline's token counts law), device-resident,
    CUDA events; one dg_m_grouped_fp8_dgrad call = two scale-packing passes +
    the GEMM."""
    import grouped_fp8_weight_gb300 as dg
    name = "moe_upgate_dgrad_fp8_g32"
    w = workloads.WORKLOADS[name]
    ms_, a, sfa, wt, sfw = workloads.draw_dgrad_operands(name, device=str(dev))
    ms_dev = torch.tensor(ms_, dtype=torch.int32, device=dev)
    d = torch.empty(w.sum_k, w.N, dtype=torch.bfloat16, device=dev)

    def call():
        dg.dg_m_grouped_fp8_dgrad(a, sfa, wt, sfw, d, ms_, ms_dev, 128)

    for _ in range(3):
        call()
    ms = time_events(call, steps, stream)
    dg.dg_sync_check()
    # the same with the weights stored K-major, [G, N, K]
    wt_k = wt.transpose(1, 2).contiguous()

    def call_nt():
        dg.dg_m_grouped_fp8_dgrad_nt(a, sfa, wt_k, sfw, d, ms_, ms_dev, 128)

    for _ in range(3):
        call_nt()
    ms_nt = time_events(call_nt, steps, stream)
    dg.dg_sync_check()
    del wt_k
    live = sum(1 for m in ms_ if m > 0)
    K, N, T = w.M, w.N, w.sum_k
    nbytes = T * K + T * (K // 128) + live * K * N + live * (K // 128) * N + T * N * 2
    flops = 2.0 * T * K * N
    fp8_peak = fp8p["tflops"]
    tflops = flops / (ms * 1e-3) / 1e12
    del a, sfa, wt, sfw, d
    return {"ms": ms, "value": tflops, "unit": "TFLOP/s", "workload": name,
            "kernel": "kgrouped_wgrad_kernel<fp8, 224, bf16, M-grouped>",
            "shape": {"G": w.G, "K": K, "N": N, "sum_m": T, "experts_with_tokens": live},
            "launches_per_step": 3, "bound": "tensor", "achieved": tflops, "peak": fp8_peak,
            "frac": tflops / fp8_peak, "peak_source": fp8p["source"], "algorithmic_bytes": nbytes,
            "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "kmajor_weights": {"ms": ms_nt, "value": flops / (ms_nt * 1e-3) / 1e12,
                               "frac": flops / (ms_nt * 1e-3) / 1e12 / fp8_peak,
                               "entry": "dg_m_grouped_fp8_dgrad_nt (W [G, N, K])"}}


def measure_inplace(w, dev, pk, fp8_peak, steps, warmup=5):
    """The in-place workloads, device-resident, CUDA events: the fine-grained
    BF16 GEMM (BF16 operands, D += A^T B) or the pipeline (BF16 dY and X cast
    by dg_quant_transpose_fp8, then the FP8 GEMM D += A^T B); for the pipeline
    also the cast pair alone and cast + GEMM."""
    import grouped_fp8_weight_gb300 as dg
    ks, A, B, C = workloads.draw_operands(w.name, device=str(dev))
    ks_dev = torch.tensor(ks, dtype=torch.int32, device=dev)
    d = C
    ne = sum(1 for k in ks if k > 0)
    stream = torch.cuda.current_stream()
    if w.kind == "bf16":
        ops = w.sum_k * (w.M + w.N) * 2

        def step():
            dg.dg_k_grouped_bf16_wgrad(A, B, d, d, ks, ks_dev)
        kname = "kgrouped_wgrad_kernel<bf16, 256, f32 reduce>"
        peak_t, peak_name = pk["bf16_tflops"], "bf16 (measured cuBLAS burst)"
    else:
        qa = torch.empty(w.sum_k, w.M, dtype=torch.uint8, device=dev)
        sa = torch.empty(w.sum_k // 128, w.M, dtype=torch.uint8, device=dev)
        qb = torch.empty(w.sum_k, w.N, dtype=torch.uint8, device=dev)
        sb = torch.empty(w.sum_k // 128, w.N, dtype=torch.uint8, device=dev)
        dg.dg_quant_transpose_fp8(A, qa, sa)
        dg.dg_quant_transpose_fp8(B, qb, sb)
        ops = w.sum_k * (w.M + w.N) + (w.sum_k // 128) * (w.M + w.N)

        def step():
            dg.dg_k_grouped_fp8_wgrad(qa, sa, qb, sb, d, d, ks, ks_dev, 128)
        kname = f"kgrouped_wgrad_kernel<fp8, {fp8_tiles(w.M, w.N)}, f32 reduce>"
        peak_t, peak_name = fp8_peak["tflops"], fp8_peak["source"]
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ms = time_events(step, steps, stream)
    dg.dg_sync_check()
    alg = ops + ne * w.M * w.N * 4 * 2          # D read and written for non-empty experts
    tf = w.flops / (ms * 1e-3) / 1e12
    gbs = alg / (ms * 1e-3) / 1e9
    out = {"workload": w.name, "ms": ms, "value": tf, "unit": "TFLOP/s", "kernel": kname,
           "launches_per_step": 1 if w.kind == "bf16" else 2,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / pk["hbm_gbs"], "algorithmic_bytes": alg},
           "tensor_frac": tf / peak_t, "tensor_peak": peak_name,
           "nonempty_experts": ne, "steps": steps,
           "shape": {"G": w.G, "M": w.M, "N": w.N, "sum_k": w.sum_k, "max_k": max(ks)}}
    if w.kind == "pipeline":
        # the pipeline's other steps: the cast of dY and X, and cast + GEMM
        def cast_pair():
            dg.dg_quant_transpose_fp8(A, qa, sa)
            dg.dg_quant_transpose_fp8(B, qb, sb)

        for _ in range(3):
            cast_pair()
        ms_cast = time_events(cast_pair, steps, stream)
        ms_pipe = time_events(lambda: (cast_pair(), step()), steps, stream)
        dg.dg_sync_check()
        cast_bytes = w.sum_k * (w.M + w.N) * 3 + (w.sum_k // 128) * (w.M + w.N)
        out["cast"] = {"ms": ms_cast, "kernel": "cast_colblock_kernel<128, token-major> x2",
                       "roofline": {"bound": "hbm", "achieved": cast_bytes / (ms_cast * 1e-3) / 1e9,
                                    "peak": pk["hbm_gbs"], "unit": "GB/s",
                                    "frac": cast_bytes / (ms_cast * 1e-3) / 1e9 / pk["hbm_gbs"],
                                    "algorithmic_bytes": cast_bytes},
                       "shapes": {"dY": [w.sum_k, w.M], "X": [w.sum_k, w.N]}}
        out["cast_plus_gemm"] = {"ms": ms_pipe, "value": w.flops / (ms_pipe * 1e-3) / 1e12,
                                 "unit": "TFLOP/s", "launches_per_step": 4}
        del qa, sa, qb, sb
    del A, B, C, d
    torch.cuda.empty_cache()
    return out


def measure_fp8_config(name, dev, pk, fp8_peak, steps):
    """A device-resident FP8 weight-gradient workload other than the headline
    (the down-projection: BF16 output, outliers): operands drawn on the device
    and cast by the library's own cast, CUDA events over `steps` calls."""
    import grouped_fp8_weight_gb300 as dg
    w = workloads.WORKLOADS[name]
    ks, a_raw, b_raw, qa, sa, qb, sb = make_inputs(w, dev)
    del a_raw, b_raw
    ks_dev = torch.tensor(ks, dtype=torch.int32, device=dev)
    out_dt = torch.float32 if w.out_dtype == "f32" else torch.bfloat16
    d = torch.empty(w.G, w.M, w.N, dtype=out_dt, device=dev)

    def step():
        dg.dg_k_grouped_fp8_wgrad(qa, sa, qb, sb, d, None, ks, ks_dev, 128)

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    ms = time_events(step, steps, torch.cuda.current_stream())
    dg.dg_sync_check()
    tf = w.flops / (ms * 1e-3) / 1e12
    alg = algorithmic_bytes(w, ks)
    del qa, sa, qb, sb, d
    torch.cuda.empty_cache()
    return {"workload": name, "ms": ms, "value": tf, "unit": "TFLOP/s", "steps": steps,
            "kernel": f"kgrouped_wgrad_kernel<fp8, {fp8_tiles(w.M, w.N)}, "
                      + ("bf16, transposed tiles>" if w.out_dtype == "bf16" else "f32>"),
            "launches_per_step": 2,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": fp8_peak["tflops"],
                         "unit": "TFLOP/s", "frac": tf / fp8_peak["tflops"],
                         "peak_source": fp8_peak["source"]},
            "hbm_frac": alg / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], "algorithmic_bytes": alg,
            "shape": {"G": w.G, "M": w.M, "N": w.N, "sum_k": w.sum_k, "max_k": max(ks),
                      "empty_experts": sum(1 for k in ks if k == 0), "out": w.out_dtype}}


def fp8_peak_for(dev, pk):
    """The dense FP8 denominator: cuBLASLt's e4m3 8192^3 rate measured now on
    this GPU (best of 10), or 2 x the measured BF16 burst if that fails."""
    try:
        r = measure_fp8_peak(dev)
        return {"tflops": r["burst_tflops"], "source": "measured: " + r["how"]}
    except Exception as exc:  # noqa: BLE001 - reported, not hidden
        return {"tflops": 2.0 * pk["bf16_tflops"],
                "source": f"assumed 2 x measured BF16 burst (FP8 measurement failed: {exc})"}


def cpu_oracle_sample(w, ks, qa, sa, qb, sb, n_rows=1024):
    """Time the float64 oracle on all experts x n_rows seeded rows of M x all N."""
    import oracle
    rows = np.sort(np.random.default_rng(w.seed).choice(w.M, n_rows, replace=False))
    qa_h = qa[:, torch.from_numpy(rows).to(qa.device)].cpu().numpy()
    sa_h = sa[:, torch.from_numpy(rows).to(sa.device)].cpu().numpy()
    qb_h, sb_h = qb.cpu().numpy(), sb.cpu().numpy()
    t0 = time.perf_counter()
    oracle.kgrouped_fp8_wgrad_rows(qa_h, sa_h, qb_h, sb_h, ks, np.arange(n_rows), 128)
    dt = time.perf_counter() - t0
    flops = 2.0 * n_rows * w.N * sum(ks)
    cores = len(os.sched_getaffinity(0))
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "seconds": dt,
            "sample": f"all {w.G} experts x {n_rows} seeded rows of M x all N "
                      f"({flops / 1e9:.1f} of {w.flops / 1e9:.0f} GFLOP), float64 numpy"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device) -> float:
    """Largest `value` over the ranks of the default process group (the
    slowest replica sets the job's time); `value` itself when ws == 1."""
    if ws <= 1:
        return value
    import torch.distributed as tdist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_replica: float, ws: int, ms_max: float) -> float:
    """Whole-job TFLOP/s: every rank runs one replica of the workload (weak
    scaling), all finishing within ms_max."""
    return ws * flops_per_replica / (ms_max * 1e-3) / 1e12


def run_reference(args):
    """Reference arm: the CPU oracle, timed on a bounded sample of the workload
    per step (all experts x 32 seeded rows of M x 256 seeded columns of N)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = workloads.WORKLOADS[args.workload]
    import oracle
    ks = workloads.counts_for(w.name)
    n_rows, n_cols = 32, 256
    gen = torch.Generator().manual_seed(w.seed)
    # Operands: N(0, 1) columns quantised by the oracle itself (columns are
    # independent, so the sampled columns are exactly the workload's columns).
    a_cols = torch.randn(w.sum_k, n_rows, generator=gen).numpy()
    b_cols = torch.randn(w.sum_k, n_cols, generator=gen).numpy()
    qa, sa = oracle.quant_colblock(a_cols, 128)
    qb, sb = oracle.quant_colblock(b_cols, 128)
    flops = 2.0 * n_rows * n_cols * w.sum_k
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.kgrouped_fp8_wgrad_rows(qa, sa, qb, sb, ks, np.arange(n_rows), 128)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    v = flops / t / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = (f"per step: all {w.G} experts x {n_rows} seeded rows of M x {n_cols} columns "
              f"of N ({flops / 1e6:.1f} MFLOP of {w.flops / 1e9:.0f} GFLOP), float64 numpy")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, ks),
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, ks):
    return {"workload": w.name, "G": w.G, "M": w.M, "N": w.N, "sum_k": w.sum_k,
            "empty_experts": sum(1 for k in ks if k == 0), "max_k": max(ks),
            "gran_k": 128, "operands": "e4m3 + ue8m0 1x128", "out": w.out_dtype,
            "accumulate": w.accumulate, "parallelism": "replicas (one workload per GPU)",
            "l2": (f"inputs and output larger than L2 (operands "
                   f"{w.sum_k * (w.M + w.N) / 1e9:.2f} GB, D "
                   f"{w.G * w.M * w.N * (4 if w.out_dtype == 'f32' else 2) / 1e9:.2f} GB); no flush")}


def run_ours(args):
    import grouped_fp8_weight_gb300 as dg
    from grouped_fp8_weight_gb300 import build as build_mod
    build_mod.build()
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=dev)
    w = workloads.WORKLOADS[args.workload]
    pk, pk_kind = peaks()
    if w.kind not in ("fp8",):
        if not args.profile:
            raise SystemExit("the full bench line runs with the headline FP8 workload and "
                             "times the others inside it; --workload X --profile times X alone")
        out = measure_inplace(w, dev, pk, fp8_peak_for(dev, pk), args.steps, args.warmup)
        if rank == 0:
            print(json.dumps({"profile_only": True, **out}), flush=True)
        return 0
    if args.profile_tiny:
        out = measure_tiny(dev, torch.cuda.current_stream(), max(args.steps, 50))
        if rank == 0:
            print(json.dumps({"profile_only": True, "tiny": out}), flush=True)
        return 0
    if args.profile_dgrad:
        # the data-gradient leg alone, for kernel captures
        out = measure_dgrad(dev, torch.cuda.current_stream(), pk, args.steps,
                            fp8_peak_for(dev, pk))
        if rank == 0:
            print(json.dumps({"profile_only": True, "dgrad": out}), flush=True)
        return 0
    if args.profile_casts:
        # the cast legs alone (no GEMM buffers), for kernel captures
        ks = workloads.counts_for(w.name)
        casts = measure_casts(w, ks, dev, torch.cuda.current_stream(), pk, args.steps)
        dg.dg_sync_check()
        if rank == 0:
            print(json.dumps({"profile_only": True, "config": workload_config(w, ks),
                              "casts": casts}), flush=True)
        return 0
    fp8p = fp8_peak_for(dev, pk)
    ks, a_raw, b_raw, qa, sa, qb, sb = make_inputs(w, dev)
    ks_dev = torch.tensor(ks, dtype=torch.int32, device=dev)
    out_dt = torch.float32 if w.out_dtype == "f32" else torch.bfloat16
    d = torch.empty(w.G, w.M, w.N, dtype=out_dt, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        dg.dg_k_grouped_fp8_wgrad(qa, sa, qb, sb, d, None, ks, ks_dev, 128)

    def barrier():
        if ws > 1:
            import torch.distributed as tdist
            tdist.barrier()

    # ---- device-resident timing (the headline value)
    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        ms = time_events(step, args.steps, stream)
        torch.cuda.synchronize()
        barrier()
    dg.dg_sync_check()
    ms_max = max_over_ranks(ms, ws, dev)
    flops = w.flops
    value = job_throughput(flops, ws, ms_max)

    # ---- roofline of the GEMM kernel (the only kernel of the step)
    alg = algorithmic_bytes(w, ks)
    gbs = alg / (ms * 1e-3) / 1e9
    fp8_peak = fp8p["tflops"]
    tflops = flops / (ms * 1e-3) / 1e12
    t_hbm = alg / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (fp8_peak * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    traffic = recorded_traffic("kgrouped_fp8", w.name)
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / pk["hbm_gbs"], "traffic": traffic}
    else:
        roof = {"bound": "tensor", "achieved": tflops, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": tflops / fp8_peak, "traffic": traffic}
    roof.update({"kernel": f"kgrouped_wgrad_kernel<fp8, {fp8_tiles(w.M, w.N)}, f32>",
                 "peak_source": pk_kind,
                 "algorithmic_bytes": alg, "tensor_tflops": tflops,
                 "tensor_peak_tflops": fp8_peak, "tensor_frac": tflops / fp8_peak,
                 "attainable_frac": max(t_hbm, t_tc) / (ms * 1e-3),
                 "timed": "one dg_k_grouped_fp8_wgrad call: scale-packing pass + GEMM kernel",
                 "tensor_peak_source": fp8p["source"]})

    if args.profile:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": "TFLOP/s",
                              "ms_per_step": ms_max, "config": workload_config(w, ks),
                              "roofline": roof, "profile_only": True}), flush=True)
        return 0

    # ---- the cast-inclusive step on the same shapes (all hot-path kernels)
    def cast_only():
        dg.dg_quant_transpose_fp8(a_raw, qa, sa)
        dg.dg_quant_transpose_fp8(b_raw, qb, sb)

    for _ in range(3):
        cast_only()
    ms_cast = time_events(cast_only, max(5, args.steps // 4), stream)
    for _ in range(2):
        cast_only()
        step()
    ms_pipe = time_events(lambda: (cast_only(), step()), max(5, args.steps // 4), stream)
    cast_bytes = w.sum_k * (w.M + w.N) * 3 + (w.sum_k // 128) * (w.M + w.N)
    pipeline = {"ms_per_step": ms_pipe, "value": flops / (ms_pipe * 1e-3) / 1e12,
                "unit": "TFLOP/s", "steps": "cast(dY) + cast(X) + GEMM",
                "cast_ms": ms_cast, "cast_roofline": {
                    "bound": "hbm", "achieved": cast_bytes / (ms_cast * 1e-3) / 1e9,
                    "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": cast_bytes / (ms_cast * 1e-3) / 1e9 / pk["hbm_gbs"],
                    "algorithmic_bytes": cast_bytes}}
    dg.dg_sync_check()

    # ---- the same GEMM with K-major (NT) operands from the channel-major cast
    qa_t = torch.empty(w.M, w.sum_k, dtype=torch.uint8, device=dev)
    qb_t = torch.empty(w.N, w.sum_k, dtype=torch.uint8, device=dev)
    dg.dg_quant_transpose_fp8(a_raw, qa_t, sa, "channel")
    dg.dg_quant_transpose_fp8(b_raw, qb_t, sb, "channel")

    def step_nt():
        dg.dg_k_grouped_fp8_wgrad_nt(qa_t, sa, qb_t, sb, d, None, ks, ks_dev, 128)

    for _ in range(3):
        step_nt()
    ms_nt = time_events(step_nt, max(5, args.steps // 4), stream)
    nt = {"ms_per_step": ms_nt, "value": flops / (ms_nt * 1e-3) / 1e12, "unit": "TFLOP/s",
          "kernel": f"kgrouped_wgrad_kernel<fp8, {fp8_tiles(w.M, w.N)}, f32, K-major>",
          "operands": "a [M, sum_k], b [N, sum_k] from the channel-major cast",
          "hbm_frac": alg / (ms_nt * 1e-3) / 1e9 / pk["hbm_gbs"],
          "tensor_frac": flops / (ms_nt * 1e-3) / 1e12 / fp8_peak}
    del qa_t, qb_t
    dg.dg_quant_transpose_fp8(a_raw, qa, sa)      # restore the token-major scales
    dg.dg_quant_transpose_fp8(b_raw, qb, sb)
    dg.dg_sync_check()

    casts = measure_casts(w, ks, dev, stream, pk, max(5, args.steps // 4))
    dg.dg_sync_check()
    dgrad = measure_dgrad(dev, stream, pk, max(5, args.steps // 4), fp8p)
    tiny = measure_tiny(dev, stream, 200)
    # ---- the other workloads, each device-resident and timed on its own
    configs = {
        "fp8_tiny_g4": {"see": "tiny"},
        "moe_upgate_fp8_g32": {"see": "value / roofline", "ms": ms, "value": tflops,
                               "tensor_frac": tflops / fp8_peak},
        "moe_down_fp8_g32": measure_fp8_config("moe_down_fp8_g32", dev, pk, fp8p,
                                               max(20, args.steps // 4)),
        "bf16_fine_g256": measure_inplace(workloads.WORKLOADS["bf16_fine_g256"], dev, pk, fp8p,
                                          max(20, args.steps // 4)),
        "pipeline_fp8_g64": measure_inplace(workloads.WORKLOADS["pipeline_fp8_g64"], dev, pk,
                                            fp8p, max(10, args.steps // 20)),
    }

    # ---- end to end through the C ABI with pinned host buffers.  Every step
    # copies its inputs in, calls the GEMM and copies the whole result out.
    # The result's copy runs on a stream of its own, so that it overlaps the
    # next step's input copies and call (two device results alternate; a call
    # waits until the copy of the result it overwrites has finished), as a
    # training loop would run them.  The timed region ends when the last
    # step's result is on the host.
    h_qa, h_sa = qa.cpu().pin_memory(), sa.cpu().pin_memory()
    h_qb, h_sb = qb.cpu().pin_memory(), sb.cpu().pin_memory()
    h_d = torch.empty(d.shape, dtype=d.dtype).pin_memory()
    outs = (d, torch.empty_like(d))
    out_stream = torch.cuda.Stream(device=dev)
    computed = [torch.cuda.Event(), torch.cuda.Event()]
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    n_e2e = [0]

    def e2e_step():
        i = n_e2e[0] % 2
        n_e2e[0] += 1
        qa.copy_(h_qa, non_blocking=True)
        sa.copy_(h_sa, non_blocking=True)
        qb.copy_(h_qb, non_blocking=True)
        sb.copy_(h_sb, non_blocking=True)
        stream.wait_event(copied[i])     # the previous copy out of outs[i] has finished
        dg.dg_k_grouped_fp8_wgrad(qa, sa, qb, sb, outs[i], None, ks, ks_dev, 128)
        computed[i].record(stream)
        out_stream.wait_event(computed[i])
        with torch.cuda.stream(out_stream):
            h_d.copy_(outs[i], non_blocking=True)
        copied[i].record(out_stream)

    e2e_steps = max(2, min(5, args.steps))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    stream.wait_event(copied[(n_e2e[0] - 1) % 2])
    e_end.record(stream)
    e_end.synchronize()
    ms_e2e = e_start.elapsed_time(e_end) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in (h_qa, h_sa, h_qb, h_sb))
    d2h = h_d.numel() * h_d.element_size()
    e2e = {"value": flops / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
           "steps": e2e_steps,
           "overlap": "each step's result copy overlaps the next step's input copies and call"}
    dg.dg_sync_check()
    del h_qa, h_sa, h_qb, h_sb, h_d, outs

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(w, ks, qa, sa, qb, sb)

    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 x e4m3 -> f32", "data": "synthetic",
            "config": workload_config(w, ks), "fp8_peak_frac": tflops / fp8_peak,
            "roofline": roof, "configs": configs, "pipeline": pipeline, "nt": nt,
            "casts": casts, "dgrad": dgrad, "tiny": tiny,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clk.summary(),
            # per step: the scale-packing pass and the GEMM kernel
            "gpu_launches": 2 * args.steps}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="moe_upgate_fp8_g32")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="device-timed leg only (for ncu captures)")
    ap.add_argument("--profile-tiny", action="store_true",
                    help="time the tiny in-place workload's call latency alone")
    ap.add_argument("--profile-dgrad", action="store_true",
                    help="time the M-grouped data-gradient leg alone (for kernel captures)")
    ap.add_argument("--profile-casts", action="store_true",
                    help="the cast legs only, `--steps` launches each (for ncu captures)")
    ap.add_argument("--fp8-peak", action="store_true",
                    help="measure the dense FP8 peak (burst and 4-s sustained) and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.fp8_peak:
        dev = torch.device("cuda", 0)
        with ClockSampler(0) as clk:
            r = measure_fp8_peak(dev, sustained_s=4.0)
        r["clocks"] = clk.summary()
        print(json.dumps(r), flush=True)
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
