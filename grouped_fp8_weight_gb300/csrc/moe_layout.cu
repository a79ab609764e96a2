// MoE token layout from top-k routing, for the cast fused with the layout.
//
// Expert e's slice holds its (token, slot) routing pairs in pair order
// t * topk + j, then -1 padding rows up to a multiple of `align`; the slices
// follow in expert order.  Deterministic (no ordering by atomics):
//   fill     every row of the output map -> -1
//   count    one warp per chunk of kPlanChunk routing entries counts its
//            entries per expert (shared-memory counters) -> counts[chunk][e]
//   scan     one CTA: per expert, the exclusive prefix of its counts over the
//            chunks (in place) and its padded total; an exclusive scan of the
//            padded totals gives each slice's first row
//   scatter  one warp per chunk walks its entries 32 at a time in order; lanes
//            routed to the same expert find each other with __match_any_sync
//            and take consecutive rows by their rank among those lanes
#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "wgrad_params.h"

namespace dg {

namespace {

constexpr int kPlanChunk = 4096;   // routing entries per warp
constexpr int kPlanWarps = 8;      // warps (chunks) per CTA

__global__ void plan_fill_kernel(int *src_rows, int *pair_rows, int64_t cap) {
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < cap;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    src_rows[r] = -1;
    if (pair_rows != nullptr) pair_rows[r] = -1;
  }
}

__global__ void __launch_bounds__(kPlanWarps * 32)
    plan_count_kernel(const int *__restrict__ idx, int64_t n, int G, int n_chunks,
                      int *__restrict__ counts, DevStatus *status) {
  extern __shared__ int cnt[];   // [kPlanWarps][G]
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int chunk = blockIdx.x * kPlanWarps + w;
  int *c = cnt + w * G;
  for (int e = l; e < G; e += 32) c[e] = 0;
  __syncwarp();
  if (chunk < n_chunks) {
    const int64_t i0 = static_cast<int64_t>(chunk) * kPlanChunk;
    const int64_t i1 = min(n, i0 + kPlanChunk);
    for (int64_t i = i0 + l; i < i1; i += 32) {
      const int e = __ldg(idx + i);
      if (e >= 0 && e < G)
        atomicAdd(c + e, 1);
      else if (e != -1)
        atomicCAS(&status->code, DEV_OK, DEV_BAD_ROUTE);
    }
    __syncwarp();
    for (int e = l; e < G; e += 32) counts[static_cast<int64_t>(chunk) * G + e] = c[e];
  }
}

// One CTA of kScanThreads threads (G <= kScanThreads).
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
    plan_scan_kernel(int *__restrict__ counts, int n_chunks, int G, int align,
                     int *__restrict__ ks, int *__restrict__ offs) {
  __shared__ int warp_sum[kScanThreads / 32];
  const int e = threadIdx.x;
  const int w = e >> 5, l = e & 31;
  int padded = 0;
  if (e < G) {
    int run = 0;
    for (int c = 0; c < n_chunks; ++c) {
      int *p = counts + static_cast<int64_t>(c) * G + e;
      const int v = *p;
      *p = run;
      run += v;
    }
    padded = (run + align - 1) / align * align;
    ks[e] = padded;
  }
  // exclusive scan of `padded` over the experts
  int x = padded;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, d);
    if (l >= d) x += y;
  }
  if (l == 31) warp_sum[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = warp_sum[l];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, d);
      if (l >= d) s += y;
    }
    warp_sum[l] = s;   // inclusive sums of the warps
  }
  __syncthreads();
  const int before = (w > 0 ? warp_sum[w - 1] : 0) + x - padded;
  if (e < G) offs[e] = before;
}

__global__ void __launch_bounds__(kPlanWarps * 32)
    plan_scatter_kernel(const int *__restrict__ idx, int64_t n, int topk, int G, int n_chunks,
                        const int *__restrict__ counts, const int *__restrict__ offs,
                        int *__restrict__ src_rows, int *__restrict__ pair_rows) {
  extern __shared__ int base[];   // [kPlanWarps][G]: next row of each expert
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int chunk = blockIdx.x * kPlanWarps + w;
  if (chunk >= n_chunks) return;   // whole warps leave together
  int *b = base + w * G;
  for (int e = l; e < G; e += 32) b[e] = offs[e] + counts[static_cast<int64_t>(chunk) * G + e];
  __syncwarp();
  const uint32_t lt = (1u << l) - 1u;
  const int64_t i0 = static_cast<int64_t>(chunk) * kPlanChunk;
  const int64_t i1 = min(n, i0 + kPlanChunk);
  for (int64_t s = i0; s < i1; s += 32) {
    const int64_t i = s + l;
    int e = (i < i1) ? __ldg(idx + i) : -1;
    const bool valid = e >= 0 && e < G;
    if (!valid) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (valid) {
      const int pos = b[e] + __popc(peers & lt);
      src_rows[pos] = static_cast<int>(i / topk);
      if (pair_rows != nullptr) pair_rows[pos] = static_cast<int>(i);
    }
    __syncwarp();
    if (valid && (peers & lt) == 0) b[e] += __popc(peers);
    __syncwarp();
  }
}

}  // namespace

size_t moe_plan_scratch_bytes(int64_t n, int G) {
  const int64_t n_chunks = (n + kPlanChunk - 1) / kPlanChunk;
  return static_cast<size_t>((n_chunks + 1) * G) * sizeof(int);
}

cudaError_t launch_moe_layout_plan(const MoePlanArgs &a, int sms, cudaStream_t stream) {
  const int n_chunks = static_cast<int>((a.n + kPlanChunk - 1) / kPlanChunk);
  int *counts = static_cast<int *>(a.scratch);
  int *offs = counts + static_cast<int64_t>(n_chunks) * a.G;
  const size_t smem = static_cast<size_t>(kPlanWarps) * a.G * sizeof(int);   // <= 32 KB
  const int64_t fill_blocks = std::min<int64_t>((a.cap + 255) / 256, 8ll * sms);
  if (fill_blocks > 0)
    plan_fill_kernel<<<static_cast<unsigned>(fill_blocks), 256, 0, stream>>>(a.src_rows,
                                                                            a.pair_rows, a.cap);
  const unsigned blocks = static_cast<unsigned>((n_chunks + kPlanWarps - 1) / kPlanWarps);
  if (blocks > 0)
    plan_count_kernel<<<blocks, kPlanWarps * 32, smem, stream>>>(a.idx, a.n, a.G, n_chunks,
                                                                 counts, a.status);
  plan_scan_kernel<<<1, kScanThreads, 0, stream>>>(counts, n_chunks, a.G, a.align, a.ks, offs);
  if (blocks > 0)
    plan_scatter_kernel<<<blocks, kPlanWarps * 32, smem, stream>>>(
        a.idx, a.n, a.topk, a.G, n_chunks, counts, offs, a.src_rows, a.pair_rows);
  return cudaGetLastError();
}

}  // namespace dg
