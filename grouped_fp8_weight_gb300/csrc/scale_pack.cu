// Scale-factor packing pass run before the FP8 K-grouped GEMM.
//
// The block-scaled MMA reads UE8M0 scales from tensor memory, where a group
// of four scale rows for a 128-row chunk of a matrix is laid out as 32 rows of
// 16 bytes: row l, byte 4q + i holds scale row i of matrix row 32q + l.  This
// pass writes every scale group the GEMM will use in exactly that layout, one
// 512-byte record per (group, 128-row chunk), so that the GEMM fetches them
// with TMA straight into the buffers tcgen05.cp copies from -- no repacking
// (and no proxy fence) inside the GEMM.
//
// Records:
//   SFA_p[gp][mc]      : rows m = 128 mc + 32 q + l of A's scales, mc < MC
//   SFB_p[gp][nt][c]   : columns n = nt * BN + 128 c + 32 q + l of B's scales,
//                        c < CB; columns outside the tile or past N are 0.
//                        With mixed tile widths the first GW groups (those of
//                        the wide entries) have NTW tiles of BNW columns and
//                        come first; the others follow with NT tiles of BN.
// where gp runs over the scale groups of all experts with K_e > 0 in schedule
// order: group j of schedule entry s is gp = g_off[s] + j and covers scale
// rows k_off[s] / gran_k + 4j .. + 3 (rows past the expert's end are 0).
// The M-grouped data gradient uses the B records alone (MC = 0) for its
// weights' scales [G * K / gran_k, N], and its own A records (per token row,
// pack_token_scales_kernel).
#include "wgrad_params.h"

namespace dg {

namespace {

__global__ void __launch_bounds__(128) pack_scales_kernel(const __grid_constant__ PackParams p) {
  griddep_launch_dependents();   // the GEMM may start its prologue and operand loads now
  const int gp = blockIdx.x;
  // schedule entry owning this group (g_off is increasing over entries)
  int lo = 0, hi = p.n_entries - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.g_off[mid] <= gp) lo = mid; else hi = mid - 1;
  }
  const int j = gp - p.g_off[lo];
  const int64_t row0 = p.row_off[lo] + 4ll * j;
  const int rows = min(4, p.row_end[lo] - static_cast<int>(4ll * j + p.row_off[lo]));
  const int t = threadIdx.x;
  const int l = t >> 2, q = t & 3;
  const int col_in = 32 * q + l;       // column within a 128-column chunk
  const int r = blockIdx.y;            // record of this group: A chunks, then B (tile, chunk)
  const bool wide = gp < p.GW;
  const int NT = wide ? p.NTW : p.NT, BN = wide ? p.BNW : p.BN;
  if (r >= p.MC + NT * p.CB) return;   // the grid covers the larger tile count
  uint32_t w = 0;
  if (r < p.MC) {
    const int m = 128 * r + col_in;
    if (m < p.M)
      for (int i = 0; i < rows; ++i)
        w |= static_cast<uint32_t>(p.sfa[(row0 + i) * p.M + m]) << (8 * i);
    p.sfa_p[(static_cast<int64_t>(gp) * p.MC + r) * 128 + t] = w;
  } else {
    const int rb = r - p.MC;           // nt * CB + c
    const int nt = rb / p.CB, c = rb - nt * p.CB;
    const int nn = 128 * c + col_in;
    const int n = nt * BN + nn;
    if (nn < BN && n < p.N)
      for (int i = 0; i < rows; ++i)
        w |= static_cast<uint32_t>(p.sfb[(row0 + i) * p.N + n]) << (8 * i);
    const int64_t rec = wide ? static_cast<int64_t>(gp) * p.NTW * p.CB + rb
                             : static_cast<int64_t>(p.GW) * p.NTW * p.CB +
                                   static_cast<int64_t>(gp - p.GW) * p.NT * p.CB + rb;
    p.sfb_p[rec * 128 + t] = w;
  }
}

// A's records for the M-grouped data gradient: one CTA per (group, token
// chunk); thread 4l + q packs the four scale columns of token 128 tc + 32 q + l.
__global__ void __launch_bounds__(128) pack_token_scales_kernel(const __grid_constant__ TokenPackParams p) {
  griddep_launch_dependents();
  const int j = blockIdx.x, tc = blockIdx.y;
  const int t = threadIdx.x;
  const int l = t >> 2, q = t & 3;
  const int64_t row = 128ll * tc + 32 * q + l;
  uint32_t w = 0;
  if (row < p.sum_m)
    for (int i = 0; i < 4; ++i) {
      const int col = 4 * j + i;
      if (col < p.KB) w |= static_cast<uint32_t>(p.sfa[row * p.KB + col]) << (8 * i);
    }
  p.sfa_p[(static_cast<int64_t>(j) * p.TC + tc) * 128 + t] = w;
}

}  // namespace

cudaError_t launch_pack_token_scales(const TokenPackParams &p, cudaStream_t stream) {
  if (p.NGK <= 0 || p.TC <= 0) return cudaSuccess;
  pack_token_scales_kernel<<<dim3(p.NGK, p.TC), 128, 0, stream>>>(p);
  return cudaGetLastError();
}

size_t plan_scale_pack(WgradParams &p, PackParams &pk, int n_mma, int gran_k, int bn) {
  const int gs = (gran_k == 128) ? 4 : 1;   // k-blocks per scale group
  int gp = 0, gw = 0;
  for (int i = 0; i < n_mma; ++i) {
    if (i == p.n_wide) gw = gp;   // the wide entries' groups end here
    const int kb = p.sched[i].k_len / 128;
    const int rows_per_kb = 128 / gran_k;
    p.sched[i].g_off = gp;
    pk.g_off[i] = gp;
    pk.row_off[i] = p.sched[i].k_off / gran_k;
    pk.row_end[i] = pk.row_off[i] + kb * rows_per_kb;
    gp += (kb + gs - 1) / gs;
  }
  if (p.n_wide >= n_mma) gw = gp;
  pk.M = p.M;
  pk.N = p.N;
  pk.MC = 2 * p.m_tiles;
  pk.NT = p.n_tiles;
  pk.CB = (bn + 127) / 128;
  pk.BN = bn;
  pk.GW = p.n_wide > 0 ? gw : 0;
  pk.NTW = p.n_wide > 0 ? p.n_tiles_w : 0;
  pk.BNW = p.n_wide > 0 ? kWideBN : 0;
  pk.n_entries = n_mma;
  pk.n_groups = gp;
  p.sf_mc = pk.MC;
  p.sf_gw = pk.GW;
  return (static_cast<size_t>(gp) * pk.MC + static_cast<size_t>(pk.GW) * pk.NTW * pk.CB +
          static_cast<size_t>(gp - pk.GW) * pk.NT * pk.CB) * 512;
}

void bind_scale_pack(PackParams &pk, void *scratch, const uint8_t *sfa, const uint8_t *sfb) {
  pk.sfa = sfa;
  pk.sfb = sfb;
  pk.sfa_p = static_cast<uint32_t *>(scratch);
  pk.sfb_p = pk.sfa_p + static_cast<size_t>(pk.n_groups) * pk.MC * 128;
}

cudaError_t launch_pack_scales(const PackParams &p, cudaStream_t stream) {
  if (p.n_groups <= 0) return cudaSuccess;
  const dim3 grid(p.n_groups, p.MC + (p.NTW > p.NT ? p.NTW : p.NT) * p.CB);
  pack_scales_kernel<<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dg
