/*
 * dg_wgrad.h -- C ABI of the GB300 (sm_103a) K-grouped weight-gradient library.
 *
 * Mixture-of-Experts weight gradient, one GEMM per expert, all experts in one
 * launch:  D[e] (+)= A_e^T B_e  (with the casts that produce its FP8 operands,
 * and the M-grouped data gradient dx_e = dy_e W_e that pairs with it).  The operands are concatenated along tokens:
 * A is [sum_k, M] (upstream gradients dy, M = h_out), B is [sum_k, N] (input
 * activations x, N = h_in), and expert e owns the contiguous rows
 * [off_e, off_e + K_e), off_e = K_0 + ... + K_{e-1}.  The GEMM's reduction
 * axis is the token axis.
 *   Sources: "How to Use DeepGEMM Weight Gradient Kernels for Training
 *   Backward Passes" (sections "API Entry Points", "FP8 Implementation
 *   Example", "BF16 Alternative", "Dispatch and Tensor-Map Handling");
 *   "Is DeepGEMM directly applicable to backward in training?" (qijiaxing,
 *   26 Mar 2025: dw = dy^T x, K = tokens, one scale per 128 tokens along K).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument named a, b, w, sfa, sfb, sfw, d, c, x, x_sf, q_in,
 *    sf_in, src_rows, pair_rows, topk_idx, ks, h, da, q_dh, sf_dh, q_a, sf_a,
 *    q, sf, ks_dev, ms_dev is a DEVICE pointer on the current CUDA device;
 *    ks_host and ms_host are HOST pointers.
 *  - All matrices are dense row-major with the last index contiguous (no
 *    padding between rows).  Device pointers must be 16-byte aligned.
 *  - The caller owns every buffer.  The first call on a device allocates one
 *    small status word for that device, kept until process exit.  Each FP8
 *    GEMM call also takes scratch for its packed scale factors (below) from a
 *    memory pool the library creates per device: allocated and freed in
 *    stream order on `stream` (cudaMallocFromPoolAsync / cudaFreeAsync), so
 *    calls on different streams never share it; the pool keeps freed blocks
 *    for reuse.  The data-gradient calls and dg_moe_layout_plan take their
 *    scratch from the same pool.
 *    The BF16 GEMM and the casts allocate nothing per call.
 *  - Work is enqueued on `stream` (NULL = legacy default stream) and runs
 *    asynchronously.  ks_host / ms_host are read during the call only;
 *    device buffers must stay valid until the enqueued work completes.
 *  - Argument errors are returned before anything is enqueued; the output is
 *    then untouched.  dg_last_error() gives a message for the calling thread.
 *  - DG_LOG=1 in the environment makes each GEMM call print its plan (tile
 *    orientation and width, tiles, entries split along K, output mode) to
 *    stderr.
 *  - Device-side waits are bounded (default 4 s; environment variable
 *    DG_WAIT_LIMIT_US, else DG_WAIT_LIMIT_MS, read at each call).  A wait that
 *    runs out makes the kernel stop early and record DG_ERR_TIMEOUT in the
 *    device status word, which dg_sync_check() reports; the output is then
 *    unspecified.  Waits for copies already in flight, on the way out, keep a
 *    limit of at least 2 s so that no copy outlives the kernel.
 *  - DG_DETERMINISTIC=1 in the environment (read at each call) keeps every
 *    expert of an in-place FP8 or BF16 GEMM in one piece (no split along K;
 *    see c under dg_k_grouped_fp8_wgrad), making in-place results bitwise
 *    reproducible at some cost in balance.
 */
#ifndef DG_WGRAD_H
#define DG_WGRAD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dg_stream_t; /* identical to cudaStream_t */

typedef enum {
    DG_OK = 0,
    DG_ERR_INVALID_ARG = 1,  /* bad shape, size, alignment, pointer or option */
    DG_ERR_UNSUPPORTED = 2,  /* device is not sm_103, or a size above a stated limit */
    DG_ERR_CUDA = 3,         /* a CUDA runtime / driver call failed */
    DG_ERR_TIMEOUT = 4       /* a bounded device-side wait ran out (see above) */
} dg_status;

typedef enum { DG_F32 = 0, DG_BF16 = 1 } dg_dtype;

typedef enum {
    DG_TOKEN_MAJOR = 0,   /* q is [T, C]: same layout as x (what the TN GEMM reads) */
    DG_CHANNEL_MAJOR = 1  /* q is [C, T]: the physical transpose of x */
} dg_layout;

/* Largest number of experts per call (one schedule entry per expert). */
#define DG_MAX_GROUPS 1024

/*
 * dg_k_grouped_fp8_wgrad -- K-grouped FP8 weight gradient with 1x1xgran_k
 * block scales.
 *
 *   D[e, m, n] = Cterm[e, m, n] + sum_{k in expert e}
 *                fp8(a[k, m]) * 2^(sfa[k / gran_k, m] - 127)
 *              * fp8(b[k, n]) * 2^(sfb[k / gran_k, n] - 127)
 *
 * Source: "How to Use DeepGEMM Weight Gradient Kernels for Training Backward
 * Passes", sections "API Entry Points" (k_grouped_fp8_gemm_tn_contiguous: the
 * TN form that reads [sum_k, M] / [sum_k, N] operands directly) and "FP8
 * Implementation Example" ((tensor, scale) operand pairs, ks on host and as a
 * device tensor, optional accumulator, recipe (1, 1, 128) with gran_k 32 or
 * 128); the DeepGEMM knowledge-base article "UE8M0 Format in DeepGEMM" (scales
 * are power-of-two UE8M0 bytes consumed by the SM100 tensor core).
 *
 *   a       E4M3 codes [sum_k, M]           sfa  UE8M0 bytes [sum_k / gran_k, M]
 *   b       E4M3 codes [sum_k, N]           sfb  UE8M0 bytes [sum_k / gran_k, N]
 *   d       output [G, M, N], FP32 or BF16 (d_dtype); BF16 is rounded to
 *           nearest-even from the FP32 accumulator.
 *   c       NULL: Cterm = 0.  c == d: accumulate in place (D += ...).  Any other
 *           pointer: a separate FP32 [G, M, N] accumulator (not modified).
 *           Only with d_dtype == DG_F32.  In place, an expert much longer than
 *           the others is split along K into parts that each add into D, so
 *           the order of the FP32 additions (and the last bits of D) may vary
 *           from run to run (unless DG_DETERMINISTIC is set); every other mode
 *           writes each element once and is bitwise reproducible.
 *   G       number of experts, 0 <= G <= DG_MAX_GROUPS.
 *   M, N    positive multiples of 16.
 *   sum_k   total tokens; must equal ks_host[0] + ... + ks_host[G-1].
 *   ks_host, ks_dev  per-expert token counts (host / device copies, same
 *           values).  Each K_e >= 0 and a multiple of 128 (an expert's slice is
 *           whole 128-token blocks).  K_e == 0 experts are skipped: with c == d
 *           their D[e] is untouched, with c == NULL it is zeroed, with a
 *           separate c it is a copy of C[e] ("Dispatch and Tensor-Map
 *           Handling": zero-size groups are skipped).  ks_dev is read by the
 *           kernel to confirm the host copy; a mismatch is recorded as
 *           DG_ERR_INVALID_ARG in the status word (see dg_sync_check).
 *   gran_k  32 or 128: tokens per scale block ("FP8 Implementation Example").
 * Work enqueued: a scale-packing pass, then the GEMM.  The pass rewrites every
 * group of four scale rows (four 128-token blocks at gran_k 128, the four
 * 32-token blocks of one 128-token block at gran_k 32) of each expert into
 * 512-byte records laid out as the tensor core reads scales, so the GEMM loads
 * them with TMA.  Scratch: (scale groups) x (2 * ceil(M' / 256) +
 * ceil(N' / BN) * ceil(BN / 128)) x 512 bytes, where (M', N') = (N, M) when
 * N % 224 != 0 and M % 224 == 0 (the kernel then computes tiles of D^T) and
 * (M, N) otherwise, BN = 224 if N' % 224 == 0 else 128, and the scale groups
 * are ceil(K_e / 512) per expert at gran_k 128 and K_e / 128 at gran_k 32
 * (about four times as many; an in-place expert split along K counts each
 * part's groups) -- about 3.9 MB for G = 32, M = 4096, N = 7168,
 * sum_k = 32768 at gran_k 128.
 * Errors: DG_ERR_INVALID_ARG for any violated condition above (including
 * NULL pointers where data is needed and misaligned pointers),
 * DG_ERR_UNSUPPORTED off sm_103, DG_ERR_CUDA on a failed launch or scratch
 * allocation.
 */
dg_status dg_k_grouped_fp8_wgrad(const void *a, const uint8_t *sfa,
                                 const void *b, const uint8_t *sfb,
                                 void *d, dg_dtype d_dtype, const float *c,
                                 int G, int M, int N, int64_t sum_k,
                                 const int *ks_host, const int *ks_dev,
                                 int gran_k, dg_stream_t stream);

/*
 * dg_k_grouped_fp8_wgrad_nt -- dg_k_grouped_fp8_wgrad with K-major (NT)
 * operands: a is E4M3 [M, sum_k] and b is E4M3 [N, sum_k] (the token axis
 * contiguous: the channel-major output of the casts, q [C, T]).  Everything
 * else -- scales sfa [sum_k / gran_k, M] and sfb [sum_k / gran_k, N], d, c,
 * ks, gran_k, errors, scratch -- is as for dg_k_grouped_fp8_wgrad, and the
 * result is the same sum.
 *
 * Source: "How to Use DeepGEMM Weight Gradient Kernels for Training Backward
 * Passes", section "API Entry Points" (k_grouped_fp8_gemm_nt_contiguous: A
 * non-transposed [M, K], B transposed [N, K]); "Is DeepGEMM directly applicable
 * to backward in training?" (qijiaxing, 26 Mar 2025: dy^T as A [h_out,
 * tokens], x^T as B [h_in, tokens]; 3 Apr 2025: a contiguous K axis is the
 * layout the NT form is built for).
 */
dg_status dg_k_grouped_fp8_wgrad_nt(const void *a, const uint8_t *sfa,
                                    const void *b, const uint8_t *sfb,
                                    void *d, dg_dtype d_dtype, const float *c,
                                    int G, int M, int N, int64_t sum_k,
                                    const int *ks_host, const int *ks_dev,
                                    int gran_k, dg_stream_t stream);

/*
 * dg_k_grouped_bf16_wgrad -- K-grouped weight gradient with BF16 operands and
 * FP32 accumulation, no scales:  D[e] = Cterm[e] + A_e^T B_e.
 *
 * Source: "How to Use DeepGEMM Weight Gradient Kernels for Training Backward
 * Passes", section "BF16 Alternative" (k_grouped_bf16_gemm_tn_contiguous,
 * same call shape as the FP8 form without scales).
 *
 *   a  BF16 [sum_k, M], b  BF16 [sum_k, N]; d, d_dtype, c as for the FP8 call.
 *   M, N positive multiples of 8.  K_e >= 0 arbitrary (no block alignment).
 * Errors as for the FP8 call.
 */
dg_status dg_k_grouped_bf16_wgrad(const void *a, const void *b,
                                  void *d, dg_dtype d_dtype, const float *c,
                                  int G, int M, int N, int64_t sum_k,
                                  const int *ks_host, const int *ks_dev,
                                  dg_stream_t stream);

/*
 * dg_m_grouped_fp8_dgrad -- the other GEMM of a MoE expert's backward, the
 * data (input) gradient, M-grouped over a contiguous token layout:
 *
 *   D[t, n] = sum_{k < K} fp8(A[t, k]) 2^(sfa[t, k / gran_k] - 127)
 *                         * fp8(W[e, k, n]) 2^(sfw[e, k / gran_k, n] - 127)
 *
 * for every token row t of expert e (rows [off_e, off_e + M_e), off_e =
 * M_0 + ... + M_{e-1}): dx_e = dy_e W_e with W_e the expert's [h_out, h_in]
 * weight as a linear layer stores it.
 *
 * Source: "Is DeepGEMM directly applicable to backward in training?"
 * (YouJiacheng, 26 Feb 2025: a GEMM's backward is two GEMMs; LyricZhao, same
 * day: the library ships the data-gradient GEMM, the weight gradient needs
 * the K-grouped kernel and the fused casts).  The pages give no layout or
 * scale recipe for it; this entry point takes the plainest one consistent
 * with the rest of the path: dy as the forward pass stores activations (E4M3,
 * one UE8M0 scale per token per gran_k channels, the 1 x 128 tile) and the
 * weight with one UE8M0 scale per column per gran_k rows of K (a 128 x 128
 * block scale is this with each block's byte repeated over its columns), both
 * scales along the contraction axis as the tensor core's block-scaled MMA
 * consumes them ("UE8M0 Format in DeepGEMM", packed scales on SM100).
 *
 *   a      E4M3 [sum_m, K], row-major (K contiguous): dy, experts' rows contiguous.
 *   sfa    UE8M0 [sum_m, K / gran_k].
 *   w      E4M3 [G, K, N], row-major (N contiguous).
 *   sfw    UE8M0 [G, K / gran_k, N].
 *   d      [sum_m, N] FP32 (d_dtype DG_F32) or BF16 (DG_BF16, round to
 *          nearest even), written (no accumulator).
 *   G      0 <= G <= DG_MAX_GROUPS; K a positive multiple of 128; N a
 *          positive multiple of 16; G * K < 2^31.
 *   ms_host, ms_dev  per-expert token counts (host / device copies, same
 *          values), each >= 0 and a multiple of 128 (the padded MoE layout,
 *          dg_moe_layout_plan); they sum to sum_m.  Experts with no tokens
 *          own no rows.  ms_dev is checked by the kernel as ks_dev is.
 *   gran_k 32 or 128.
 * Work enqueued: two scale-packing passes (dy's scales per 128-token chunk,
 * the weights' per N tile), then the GEMM.  Scratch from the device pool:
 * (ceil(K / 128 / g) x (sum_m / 128 + 1) + E x ceil(K / 128 / g) x
 * ceil(N / BN) x ceil(BN / 128)) x 512 bytes, g = 4 at gran_k 128 and 1 at
 * 32, E the experts with tokens, BN as above.  Errors as for the weight
 * gradient calls; DG_ERR_UNSUPPORTED also for an output of 2^40 bytes or more.
 */
dg_status dg_m_grouped_fp8_dgrad(const void *a, const uint8_t *sfa,
                                 const void *w, const uint8_t *sfw,
                                 void *d, dg_dtype d_dtype,
                                 int G, int K, int N, int64_t sum_m,
                                 const int *ms_host, const int *ms_dev,
                                 int gran_k, dg_stream_t stream);

/*
 * dg_m_grouped_fp8_dgrad_nt -- dg_m_grouped_fp8_dgrad with the weights stored
 * K-major: w is E4M3 [G, N, K] (row n of expert e holds W_e[:, n], K
 * contiguous), the layout of a transposed weight copy.  The scales keep the
 * layout sfw [G, K / gran_k, N] (one per column n per gran_k rows of K), and
 * a, sfa, d, ms, gran_k, the result, errors and scratch are as for
 * dg_m_grouped_fp8_dgrad.  G * N < 2^31.
 *
 * Source: as dg_m_grouped_fp8_dgrad; "How to Use DeepGEMM Weight Gradient
 * Kernels for Training Backward Passes", section "API Entry Points" (the NT
 * operand form: the second operand transposed, K contiguous).
 */
dg_status dg_m_grouped_fp8_dgrad_nt(const void *a, const uint8_t *sfa,
                                    const void *w, const uint8_t *sfw,
                                    void *d, dg_dtype d_dtype,
                                    int G, int K, int N, int64_t sum_m,
                                    const int *ms_host, const int *ms_dev,
                                    int gran_k, dg_stream_t stream);

/*
 * dg_quant_transpose_fp8 -- the cast a weight-gradient GEMM needs: per column,
 * per gran_k-token block, one power-of-two scale, values to E4M3.
 *
 *   amax    = max_{k in block} |x[k, col]|
 *   e       = clamp(ceil(log2(amax / 448)), -127, 127)   (amax == 0 -> -127)
 *   sf      = e + 127                                     (UE8M0 byte)
 *   q[k, col] = E4M3 round-to-nearest-even of x[k, col] * 2^-e
 *
 * Source: "Is DeepGEMM directly applicable to backward in training?"
 * (LyricZhao, 26 Feb 2025: weight gradients need fused transpose + cast
 * kernels; hxdtest quoting the DeepSeek-V3 workflow, 4 May 2025: activations
 * are transposed and re-quantised into 128x1 tiles; qijiaxing, 26 Mar 2025:
 * every 128 elements along the token axis share one scale).  448 is the
 * largest E4M3 magnitude, so the cast never saturates.
 *
 *   x         BF16 [T, C] (tokens x channels).
 *   T         non-negative multiple of gran_k.
 *   C         positive multiple of 16.
 *   q         E4M3 out: [T, C] (DG_TOKEN_MAJOR) or [C, T] (DG_CHANNEL_MAJOR).
 *   sf        UE8M0 out [T / gran_k, C].
 *   gran_k    32 or 128.
 * Inputs must be finite.  Errors: DG_ERR_INVALID_ARG / DG_ERR_UNSUPPORTED /
 * DG_ERR_CUDA as above.
 */
dg_status dg_quant_transpose_fp8(const void *x, int64_t T, int C,
                                 void *q, uint8_t *sf,
                                 dg_layout q_layout, int gran_k,
                                 dg_stream_t stream);

/*
 * dg_requant_transpose_fp8 -- re-quantise stored FP8 activations for the
 * weight gradient: from the forward pass's 1 x 128 tiles (one scale per token
 * per 128 channels) to column blocks (one scale per channel per gran_k
 * tokens), with the same cast as dg_quant_transpose_fp8 applied to the
 * exactly dequantised values:
 *
 *   x[t, c] = E4M3(q_in[t, c]) * 2^(sf_in[t, c / 128] - 127)
 *   (q, sf) = dg_quant_transpose_fp8 of x
 *
 * Source: "Is DeepGEMM directly applicable to backward in training?" (hxdtest,
 * 4 May 2025, quoting the DeepSeek-V3 workflow: forward activations are
 * stored as 1x128 FP8 tiles; the backward pass reads them out, dequantises,
 * transposes and re-quantises them into 128x1 tiles; TheTinyTeddy, 12 Mar
 * 2025: the FP8 weight-gradient GEMM lets activations be stored in FP8).  The
 * pages do not give the stored scales' format; here they are UE8M0 bytes (the
 * SM100 format of "UE8M0 Format in DeepGEMM").
 *
 *   q_in      E4M3 codes [T, C] (token-major, as the forward pass stored them).
 *   sf_in     UE8M0 bytes [T, C / 128]; bytes 0..254 (255 is NaN: unsupported).
 *   T         non-negative multiple of gran_k.
 *   C         positive multiple of 128.
 *   q, sf, q_layout, gran_k   as for dg_quant_transpose_fp8.
 * Every dequantised value is exact in the kernel (it works on x * 2^-8, which
 * is finite and exact in FP32 for every code and scale byte), so the result is
 * bit-identical to the definition above.  Errors as for dg_quant_transpose_fp8.
 */
dg_status dg_requant_transpose_fp8(const void *q_in, const uint8_t *sf_in,
                                   int64_t T, int C,
                                   void *q, uint8_t *sf,
                                   dg_layout q_layout, int gran_k,
                                   dg_stream_t stream);

/*
 * dg_quant_moe_layout_fp8 -- the column-block cast fused with the MoE token
 * layout: output row t is source row src_rows[t], or a row of zeros where
 * src_rows[t] == -1 (padding an expert's slice up to whole 128-token blocks),
 * then cast as by dg_quant_transpose_fp8 (BF16 source) or
 * dg_requant_transpose_fp8 (stored FP8 source).
 *
 * Source: "Is DeepGEMM directly applicable to backward in training?"
 * (LyricZhao, 26 Feb 2025: weight-gradient support needs utility kernels with
 * the cast fused with the MoE layout; NiuMa, 18 Mar 2025: the FP8 weight
 * gradient needs each expert's token count to be a multiple of 128).
 *
 *   x         x_sf == NULL: BF16 [T_src, C].  Otherwise E4M3 codes [T_src, C]
 *             with x_sf UE8M0 [T_src, C / 128] (1 x 128 tiles, as for
 *             dg_requant_transpose_fp8; C then a multiple of 128).
 *   T_src     source rows (>= 0, < 2^31).
 *   src_rows  device int32 [T]: source row of each output row, or -1.  An
 *             entry outside [-1, T_src) gives a zero row and is recorded as
 *             DG_ERR_INVALID_ARG in the device status word (dg_sync_check).
 *   T         output rows: a non-negative multiple of gran_k (each expert's
 *             slice is a whole number of blocks).
 *   q, sf, q_layout, gran_k   as for dg_quant_transpose_fp8, over the T output
 *             rows.
 * Errors as for dg_quant_transpose_fp8.
 */
dg_status dg_quant_moe_layout_fp8(const void *x, const uint8_t *x_sf,
                                  int64_t T_src, int C,
                                  const int *src_rows, int64_t T,
                                  void *q, uint8_t *sf,
                                  dg_layout q_layout, int gran_k,
                                  dg_stream_t stream);

/*
 * dg_moe_layout_plan -- the MoE token layout that dg_quant_moe_layout_fp8 and
 * the K-grouped GEMMs consume, built on the device from top-k routing.
 *
 * Expert e's slice holds its routing pairs (t, j) (topk_idx[t, j] == e) in the
 * order of the pair index t * topk + j, then -1 padding rows up to a multiple
 * of `align`; the slices follow in expert order.  ks[e] is the slice's padded
 * length, so ks feeds the GEMM's ks_dev directly (and, copied to the host, its
 * ks_host).  Deterministic: the same routing always gives the same layout.
 *
 * Source: "Is DeepGEMM directly applicable to backward in training?"
 * (LyricZhao, 26 Feb 2025: casts fused with the MoE layout; NiuMa, 18 Mar
 * 2025: the FP8 weight gradient needs each expert's token count to be a
 * multiple of 128, which padding provides).
 *
 *   topk_idx   device int32 [T_tok, topk]: the expert of each (token, slot),
 *              or -1 for an unused slot.  An entry outside [-1, G) is skipped
 *              and recorded as DG_ERR_INVALID_ARG in the device status word
 *              (dg_sync_check).
 *   T_tok      tokens (>= 0);  topk >= 1;  T_tok * topk + G * (align - 1) < 2^31.
 *   G          experts, 1 <= G <= DG_MAX_GROUPS.
 *   align      slice length multiple, 1..65536 (128 for the FP8 GEMM).
 *   ks         device int32 [G] out.
 *   src_rows   device int32 [cap] out: the source token t of each row, -1 on
 *              padding and on every row past the layout's end.
 *   pair_rows  device int32 [cap] out, or NULL: the pair index t * topk + j of
 *              each row (for operands stored per routed pair), -1 likewise.
 *   cap        rows of src_rows / pair_rows; at least T_tok * topk +
 *              G * (align - 1), the largest layout any routing can give.
 * Scratch: (ceil(T_tok * topk / 4096) + 1) * G int32 counters from the
 * library's stream-ordered pool.  Errors: DG_ERR_INVALID_ARG (arguments,
 * cap too small, NULL or misaligned pointers), DG_ERR_UNSUPPORTED (G above
 * DG_MAX_GROUPS, sizes above the limit), DG_ERR_CUDA.
 */
dg_status dg_moe_layout_plan(const int *topk_idx, int64_t T_tok, int topk,
                             int G, int align,
                             int *ks, int *src_rows, int *pair_rows,
                             int64_t cap, dg_stream_t stream);

/*
 * dg_swiglu_backward_quant_fp8 -- the SwiGLU backward of a MoE expert fused
 * with the column-block cast of its outputs, token-major:
 *
 *   h = [g | u] (gate half first), s = 1 / (1 + e^-g), silu(g) = g * s
 *   dg = da * u * s * (1 + g * (1 - s)),  du = da * silu(g),  a = silu(g) * u
 *   (q_dh, sf_dh) = cast of dh = [dg | du]   (the up/gate weight gradient's A)
 *   (q_a, sf_a)   = cast of a                 (the down-projection's B)
 * with the cast of dg_quant_transpose_fp8 (one UE8M0 scale per column per
 * gran_k tokens).
 *
 * Source: "Is DeepGEMM directly applicable to backward in training?"
 * (LyricZhao, 26 Feb 2025: weight-gradient support needs utility kernels,
 * among them casting fused with SwiGLU).  The pages give no formula; this is
 * the standard SwiGLU.
 *
 *   h       BF16 [T, 2I];  da  BF16 [T, I].
 *   T       non-negative multiple of gran_k.   I  positive multiple of 16.
 *   q_dh    E4M3 [T, 2I];  sf_dh  UE8M0 [T / gran_k, 2I].
 *   q_a     E4M3 [T, I] and sf_a UE8M0 [T / gran_k, I], or both NULL.
 *   gran_k  32 or 128.
 * Arithmetic: FP32 with explicitly rounded operations, e^-|g| from expf and
 * 1 / (1 + e^-|g|) from the hardware reciprocal (within 1 ulp); dg, du and a must stay finite in FP32
 * (non-finite values are unsupported).  Each quantised code and scale is the
 * one of a value within a few FP32 ulp of the exact result (the tests bound
 * it).  Errors as for dg_quant_transpose_fp8.
 */
dg_status dg_swiglu_backward_quant_fp8(const void *h, const void *da,
                                       int64_t T, int I,
                                       void *q_dh, uint8_t *sf_dh,
                                       void *q_a, uint8_t *sf_a,
                                       int gran_k, dg_stream_t stream);

/*
 * dg_k_grouped_fp8_wgrad_noalloc -- dg_k_grouped_fp8_wgrad for callers that
 * cannot allocate device memory.  The pages have no counterpart: this is an
 * addition of this library.
 *
 * The ordinary call allocates a 16-byte status record per device (cudaMalloc)
 * on its first use and takes stream-ordered scratch for the packed scale
 * factors on every call.  A caller whose device memory is owned by its own
 * caching allocator, or that must not take the device synchronisation
 * cudaMalloc can cause, cannot accept that.  This entry point computes exactly
 * what dg_k_grouped_fp8_wgrad computes, with the same arguments and errors,
 * by the same host steps (validation, schedule with its tile orientation and
 * split along K, tensor maps, scale packing, launch), and allocates nothing:
 * the status record and the packed scale records live in one file-scope
 * device array of the library, 256 bytes + 32 MiB (every GPU that loads this
 * part of the library holds it until the process exits).
 *  - The first call on a device does the set-up (device queries, the
 *    array's device address via cudaGetSymbolAddress); make that first call
 *    before any stream capture.
 *  - Each call clears the record and rewrites the scale records on `stream`
 *    before its GEMM; calls that overlap on the GPU (on different streams)
 *    share the array and race on it.
 *  - It never synchronises.  dg_sync_check() reads and clears this entry
 *    point's record as well as the ordinary one, so device-side timeouts and
 *    ks_dev mismatches are reported there.
 *  - Limits: the packed scale records must fit 32 MiB (their size is given
 *    under dg_k_grouped_fp8_wgrad; G = 64, M = 4096, N = 7168,
 *    sum_k = 131072 needs 14 MB at gran_k 128 and about four times that,
 *    above the limit, at gran_k 32); larger problems, and sizes above the kernel's own limits
 *    (G > DG_MAX_GROUPS, sum_k > 2^31 - 256), are rejected with
 *    DG_ERR_UNSUPPORTED and a message before any CUDA call.
 */
dg_status dg_k_grouped_fp8_wgrad_noalloc(const void *a, const uint8_t *sfa,
                                         const void *b, const uint8_t *sfb,
                                         void *d, dg_dtype d_dtype, const float *c,
                                         int G, int M, int N, int64_t sum_k,
                                         const int *ks_host, const int *ks_dev,
                                         int gran_k, dg_stream_t stream);

/* Message describing the calling thread's last non-OK status ("" if none). */
const char *dg_last_error(void);

/*
 * Synchronise `stream`, then read and clear the current device's status words
 * (the ordinary entry points' record and dg_k_grouped_fp8_wgrad_noalloc's).
 * Allocates nothing.  Returns DG_ERR_TIMEOUT if a kernel gave up on a bounded
 * wait,
 * DG_ERR_INVALID_ARG if a kernel found ks_dev different from ks_host, a
 * src_rows entry or a topk_idx entry out of range,
 * DG_ERR_CUDA if the synchronisation failed, else DG_OK.
 */
dg_status dg_sync_check(dg_stream_t stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int dg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DG_WGRAD_H */
