// Host <-> device contract of the K-grouped weight-gradient kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace dg {

constexpr int kMaxGroups = 1024;   // must equal DG_MAX_GROUPS

// One schedule entry: an expert and its token slice.  Entries with k_len > 0
// come first, longest first; after them come experts whose output must be
// written without a GEMM (K_e == 0 with no accumulator or a separate one).
struct SchedEntry {
  int expert;
  int k_off;
  int k_len;
  int pad;
};

enum OutMode : int {
  OUT_F32 = 0,         // D = acc
  OUT_F32_REDUCE = 1,  // D += acc (C aliases D), done by TMA reduce-add
  OUT_F32_C = 2,       // D = C + acc, C separate
  OUT_BF16 = 3,        // D = bf16(acc)
};

struct WgradParams {
  CUtensorMap tmA;     // operand A [sum_k, M], 128-byte swizzled tiles
  CUtensorMap tmB;     // operand B [sum_k, N], 128-byte swizzled tiles
  CUtensorMap tmSFA;   // UE8M0 [sum_k / gran_k, M]   (FP8 only)
  CUtensorMap tmSFB;   // UE8M0 [sum_k / gran_k, N]   (FP8 only)
  CUtensorMap tmD;     // output [G, M, N] as 3-D {N, M, G}
  CUtensorMap tmC;     // separate accumulator, same shape (OUT_F32_C only)
  int M, N, G;
  int m_tiles, n_tiles, tiles_per_group;
  int num_mma_tiles;   // tiles that run a GEMM
  int num_tiles;       // all tiles, fill tiles last
  int gran_k;          // 32 or 128 (FP8)
  int out_mode;
  int m_fastest;       // tile order inside an expert: 1 = M tiles vary fastest
  uint64_t wait_limit_ns;
  DevStatus *status;
  const int *ks_dev;
#ifdef DG_KERNEL_TIMERS
  unsigned long long *timers;   // profiling builds: 32 counters per CTA
#endif
  SchedEntry sched[kMaxGroups];
};

// Launchers (one translation unit each): `pairs` clusters of two CTAs (capped
// at the number that fit the GPU at once).  Return the launch error, if any.
cudaError_t launch_kgrouped_fp8(const WgradParams &p, int block_n, int pairs,
                                cudaStream_t stream);
cudaError_t launch_kgrouped_bf16(const WgradParams &p, int block_n, int pairs,
                                 cudaStream_t stream);
cudaError_t launch_quant_colblock(const void *x, int64_t T, int C, void *q, uint8_t *sf,
                                  int channel_major, int gran_k, cudaStream_t stream);

// Tile shape: a CTA pair covers 256 rows of M (128 per CTA) and block_n
// columns of N.
constexpr int kPairM = 256;
int fp8_pick_block_n(int N);
int bf16_pick_block_n(int N);

}  // namespace dg
