// Host <-> device contract of the K-grouped weight-gradient kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace dg {

constexpr int kMaxGroups = 1024;   // must equal DG_MAX_GROUPS

// One schedule entry: an expert and a token slice of it (the whole slice, or
// for in-place accumulation one part of a long expert's).  Entries with
// k_len > 0 come first, longest first; after them come experts whose output
// must be written without a GEMM (K_e == 0 with no accumulator or a separate one).
//
// M-grouped data gradient (mgroup = 1): one entry per expert with tokens, in
// expert order; k_off = e * K (the expert's first row of W), k_len = K,
// k_exp = the expert's token count, row_off its first token row, tile_off its
// first tile (tiles: 256-token chunks x N tiles), g_off its first packed scale
// group of W.
struct SchedEntry {
  int expert;
  int k_off;
  int k_len;
  int g_off;   // FP8: first packed scale group of this entry
  int k_exp;   // the expert's whole token count (an entry may be one part of it)
  int row_off;    // M-grouped only
  int tile_off;   // M-grouped only
};

// Division by an invariant divisor d >= 1 for numerators x < 2^31
// (Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994): with l = ceil(log2 d) and p = 31 + l,
// mul = ceil(2^p / d) fits 32 bits and x / d = umulhi(x, mul) >> (p - 32);
// d == 1 is the identity (mul = 0).
struct FastDiv {
  uint32_t mul;
  uint32_t shift;
};
inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f{0, 0};
  if (d <= 1) return f;
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  const uint32_t p = 31 + l;
  f.mul = static_cast<uint32_t>(((1ull << p) + d - 1) / d);
  f.shift = p - 32;
  return f;
}
__device__ __forceinline__ int fast_div(int x, FastDiv f) {
  return f.mul == 0 ? x : static_cast<int>(__umulhi(static_cast<uint32_t>(x), f.mul) >> f.shift);
}

enum OutMode : int {
  OUT_F32 = 0,         // D = acc
  OUT_F32_REDUCE = 1,  // D += acc (C aliases D), done by TMA reduce-add
  OUT_F32_C = 2,       // D = C + acc, C separate
  OUT_BF16 = 3,        // D = bf16(acc)
};

struct WgradParams {
  CUtensorMap tmA;     // operand A [sum_k, M], 128-byte swizzled tiles
  CUtensorMap tmB;     // operand B [sum_k, N], 128-byte swizzled tiles
  CUtensorMap tmBn;    // mixed widths: B boxes of the narrow tiles (kNarrowBN / 2 columns)
  CUtensorMap tmSFA;   // FP8: packed scale records of A, 512 bytes each (see PackParams)
  CUtensorMap tmSFB;   // FP8: packed scale records of B, CB x 512 bytes per box
  CUtensorMap tmD;     // output [G, M, N] as 3-D {N, M, G}
  CUtensorMap tmC;     // separate accumulator, same shape (OUT_F32_C only)
  int M, N, G;
  int m_tiles, n_tiles, tiles_per_group;
  int num_mma_tiles;   // tiles that run a GEMM
  int num_tiles;       // all tiles, fill tiles last
  int gran_k;          // 32 or 128 (FP8)
  int out_mode;
  int m_fastest;       // tile order inside an expert: 1 = M tiles vary fastest
  int sf_mc;           // FP8: packed A records per scale group (2 * m_tiles)
  int chunk;           // stages of a lane-0 tile per turn (FP8: a multiple of 4)
  int mgroup;          // 1: M-grouped data gradient (see SchedEntry)
  int n_entries;       // M-grouped: schedule entries
  int n_sched;         // valid entries of sched (copied to shared memory when they fit)
  FastDiv div_tpg, div_mt, div_nt;   // by tiles_per_group, m_tiles, n_tiles
  // Mixed tile widths (FP8, kernel N a multiple of 256 and of 224): the first
  // n_wide schedule entries are cut into 256-column tiles (wide_tiles of them,
  // first in the tile list; n_tiles_w per row), every later entry into
  // 224-column tiles (n_tiles per row).  Their packed B records come first
  // (sf_gw scale groups of n_tiles_w tiles each).  Zero otherwise.
  int n_wide, wide_tiles, n_tiles_w, tpg_w, sf_gw;
  FastDiv div_tpg_w, div_nt_w;
  // FP8: the GEMM is launched as a programmatic dependent of the scale-pack
  // pass just before it (host only: selects the launch attribute).
  int pdl;
  uint64_t wait_limit_ns;
  DevStatus *status;
  const int *ks_dev;
#ifdef DG_KERNEL_TIMERS
  unsigned long long *timers;   // profiling builds: 32 counters per CTA
#endif
  SchedEntry sched[kMaxGroups];
};
static_assert(sizeof(WgradParams) <= 32764, "kernel parameters are limited to 32764 bytes");

// Host: the fields derived from the tile counts, and the schedule length.
inline void set_derived(WgradParams &p, int n_sched) {
  p.n_sched = n_sched;
  p.div_tpg = make_fastdiv(static_cast<uint32_t>(p.tiles_per_group > 0 ? p.tiles_per_group : 1));
  p.div_mt = make_fastdiv(static_cast<uint32_t>(p.m_tiles > 0 ? p.m_tiles : 1));
  p.div_nt = make_fastdiv(static_cast<uint32_t>(p.n_tiles > 0 ? p.n_tiles : 1));
  p.div_tpg_w = make_fastdiv(static_cast<uint32_t>(p.tpg_w > 0 ? p.tpg_w : 1));
  p.div_nt_w = make_fastdiv(static_cast<uint32_t>(p.n_tiles_w > 0 ? p.n_tiles_w : 1));
}

// FP8 scale packing (scale_pack.cu): every scale group the GEMM uses, laid
// out as the 32-row x 16-byte records tcgen05.cp copies into tensor memory.
// Group j of schedule entry s (K_e > 0) is record group g_off[s] + j; it covers
// scale rows row_off[s] + 4j .. + 3, and rows at or past row_end[s] read as 0.
struct PackParams {
  const uint8_t *sfa, *sfb;   // [sum_k / gran_k, M] and [sum_k / gran_k, N]
  uint32_t *sfa_p;            // [n_groups][MC][128 words]
  uint32_t *sfb_p;            // [GW][NTW][CB] then [n_groups - GW][NT][CB], 128 words each
  int M, N, MC, NT, CB, BN;
  int GW, NTW, BNW;           // mixed widths: the first GW groups use NTW tiles of BNW columns
  int n_entries, n_groups;
  int g_off[kMaxGroups];
  int row_off[kMaxGroups];
  int row_end[kMaxGroups];
};

// Fills pk's plan (and p.sched[i].g_off, p.sf_mc, p.sf_gw) from the first
// n_mma schedule entries of p for block width bn (the narrow width when
// p.n_wide > 0: the first p.n_wide entries then use p.n_tiles_w tiles of
// kWideBN columns); returns the scratch bytes the packed records need (0 when
// there is no GEMM work).
size_t plan_scale_pack(WgradParams &p, PackParams &pk, int n_mma, int gran_k, int bn);
// Points pk at `scratch` (16-byte aligned, plan_scale_pack's size).
void bind_scale_pack(PackParams &pk, void *scratch, const uint8_t *sfa, const uint8_t *sfb);
cudaError_t launch_pack_scales(const PackParams &p, cudaStream_t stream);

// M-grouped data gradient: A's scales are per token row ([sum_m, KB] with
// KB = K / gran_k scale columns); their records are [NGK][TC][128 words]
// (group j of K's scale columns 4j..4j+3, 128-token chunk tc: word 4l + q
// holds the scales of token 128 tc + 32 q + l), zero past sum_m or KB.
struct TokenPackParams {
  const uint8_t *sfa;
  uint32_t *sfa_p;
  int64_t sum_m;
  int KB, NGK, TC;
};
cudaError_t launch_pack_token_scales(const TokenPackParams &p, cudaStream_t stream);

// Launchers (one translation unit each): `pairs` clusters of two CTAs (capped
// at the number that fit the GPU at once).  Return the launch error, if any.
cudaError_t launch_kgrouped_fp8(const WgradParams &p, int block_n, int pairs,
                                cudaStream_t stream);
cudaError_t launch_kgrouped_bf16(const WgradParams &p, int block_n, int pairs,
                                 cudaStream_t stream);
// FP8 with K-major operands (tmA / tmB map [M, sum_k] / [N, sum_k]).
cudaError_t launch_kgrouped_fp8_nt(const WgradParams &p, int block_n, int pairs,
                                   cudaStream_t stream);
// Transposed output tiles (the kernel's A is the caller's B, its M the
// caller's N; D and C maps keep the caller's [G, M, N]); block_n 224, or 256
// (mixed widths).
cudaError_t launch_kgrouped_fp8_t(const WgradParams &p, int block_n, int pairs,
                                  cudaStream_t stream);
cudaError_t launch_kgrouped_fp8_nt_t(const WgradParams &p, int block_n, int pairs,
                                     cudaStream_t stream);
// M-grouped FP8 data gradient (tmA maps dy as {K, sum_m}, tmB the weights as
// {N, G * K}, tmD the output as {N, sum_m, 1}).
cudaError_t launch_mgrouped_fp8(const WgradParams &p, int block_n, int pairs,
                                cudaStream_t stream);
// The same with the weights stored K-major, W [G, N, K]: tmB maps them as
// {K, G * N} and each entry's k_off is e * N (its first row of W).
cudaError_t launch_mgrouped_fp8_nt(const WgradParams &p, int block_n, int pairs,
                                   cudaStream_t stream);
// Column-block casts (quant.cu).  x is BF16 [T_src, C], or, with x_sf set,
// E4M3 codes [T_src, C] with one UE8M0 scale per token per 128 channels
// (x_sf [T_src, C / 128]).  With src_rows set, output row t takes source row
// src_rows[t] (-1: a row of zeros); otherwise row t (T_src == T).
struct CastArgs {
  CUtensorMap tmx;     // BF16 gather, token-major: x as {C, T_src}, boxes of 256 x 1
  const void *x;
  const uint8_t *x_sf;
  const int *src_rows;
  int64_t T_src, T;
  int C;
  uint8_t *q, *sf;
  DevStatus *status;   // records DEV_BAD_ROW for a src_rows entry outside [-1, T_src)
  int use_tmx;         // 1: tmx is valid and the row gather runs through TMA
  uint64_t wait_limit_ns;
};
cudaError_t launch_cast_colblock(const CastArgs &a, int channel_major, int gran_k,
                                 cudaStream_t stream);

// MoE layout plan (moe_layout.cu) from routing idx[n] (n = tokens x topk).
struct MoePlanArgs {
  const int *idx;
  int64_t n;
  int topk, G, align;
  int *ks, *src_rows, *pair_rows;   // pair_rows may be null
  int64_t cap;                      // rows of src_rows / pair_rows
  void *scratch;                    // moe_plan_scratch_bytes(n, G), 16-byte aligned
  DevStatus *status;                // records DEV_BAD_ROUTE for an entry outside [-1, G)
};
size_t moe_plan_scratch_bytes(int64_t n, int G);

// SwiGLU backward fused with the column-block cast (swiglu.cu).
struct SwigluArgs {
  CUtensorMap tm_h;     // h as {2I, T} BF16, boxes of 32 channels x 128 tokens
  CUtensorMap tm_da;    // da as {I, T} BF16, same boxes
  int64_t T;
  int I;
  int n_tt, n_tc;       // tiles along tokens (128) and along channels of I (32)
  uint8_t *q_dh, *sf_dh;   // E4M3 [T, 2I], UE8M0 [T / gran_k, 2I]
  uint8_t *q_a, *sf_a;     // E4M3 [T, I], UE8M0 [T / gran_k, I], or null
  DevStatus *status;       // bounded waits record DEV_TIMEOUT here
  uint64_t wait_limit_ns;
};
// `ctas`: persistent CTAs (two per SM fit).
cudaError_t launch_swiglu_bwd_cast(const SwigluArgs &p, int gran_k, int ctas, cudaStream_t stream);
cudaError_t launch_moe_layout_plan(const MoePlanArgs &a, int sms, cudaStream_t stream);

// Tile shape: a CTA pair covers 256 rows of M (128 per CTA) and block_n
// columns of N.
constexpr int kPairM = 256;
// Stages of a long tile issued per turn before the MMA stream switches to the
// other accumulator's tile (FP8 stages are 128 tokens, BF16 64).  FP32 output
// (4 bytes per element to store) drains a tile in about as long as 48 MMA
// stages take; BF16 output in half that, and its tiles interleave best in
// short turns; in-place accumulation (reduce-add) was measured best at 16.
constexpr int kFp8Chunk = 48;
constexpr int kFp8ChunkBf16Out = 8;
constexpr int kFp8ChunkBf16OutMixed = 12;   // BF16 output with mixed tile widths
constexpr int kFp8ChunkInPlace = 16;
static_assert(kFp8Chunk % 4 == 0 && kFp8ChunkBf16Out % 4 == 0 && kFp8ChunkInPlace % 4 == 0 &&
                  kFp8ChunkBf16OutMixed % 4 == 0,
              "lane chunks must start on a scale group (four k-blocks)");
// Mixed tile widths: the lane-0 turns of the wide tiles may reach this
// percentage of the narrow tiles' count (FP32 output / the other modes).
constexpr int kMixPercentF32 = 50;
constexpr int kMixPercent = 100;
// Epilogue chunk: output columns per staged TMA store box (32 rows high).
constexpr int kEpiCols = 32;
// Staging row of kEpiCols elements of `bytes` each is stored with the TMA
// swizzle of its width (32, 64 or 128 bytes).
inline CUtensorMapSwizzle epi_swizzle(int elem_bytes) {
  const int row = kEpiCols * elem_bytes;
  return row >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                    : row == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
}
constexpr int kBf16Chunk = 80;
// Mixed tile widths: block_n kWideBN selects the FP8 variant whose first
// accumulator is 256 columns wide and second kNarrowBN (256 + 224 + two
// 12-column scale slots fit the 512 tensor-memory columns).
constexpr int kWideBN = 256;
constexpr int kNarrowBN = 224;
int fp8_pick_block_n(int N);
int bf16_pick_block_n(int N);

}  // namespace dg
