// Persistent, warp-specialised K-grouped weight-gradient kernel for sm_103a.
//
//   D[e] (+)= A_e^T B_e,   A_e = A[off_e : off_e + K_e, :],  B_e likewise.
//
// One CTA per SM walks the tile list (expert, m-tile, n-tile) with a stride of
// gridDim.x; experts are ordered longest-first so that the heavy tiles start
// first and the tail of the launch is made of short tiles.  Roles:
//   warp 0      TMA producer: A/B tiles (and, for FP8, the raw UE8M0 scale rows)
//               of each token block into an S-stage shared-memory ring.
//   warp 1      tensor-memory owner and MMA issuer: repacks the stage's scale
//               bytes for tcgen05.cp, copies them into tensor memory, issues
//               four tcgen05.mma per stage (block-scaled E4M3, or BF16), and
//               commits stage release / accumulator-ready to mbarriers.
//   warps 2..5  epilogue: tensor memory -> registers -> swizzled shared-memory
//               staging -> TMA store (or TMA reduce-add for in-place D += acc).
// Two accumulators live in tensor memory, so the epilogue of one tile overlaps
// the MMAs of the next.
//
// Operands are MN-major (the token axis is K and is the slow axis in memory):
// an operand tile for one stage is BK token rows x 128-byte swizzle atoms.
#pragma once

#include <cuda_bf16.h>

#include "wgrad_params.h"

namespace dg {

template <bool kFP8, int kBN>
struct WgradCfg {
  static constexpr int BM = 128;
  static constexpr int ELEM = kFP8 ? 1 : 2;
  static constexpr int BK = kFP8 ? 128 : 64;            // tokens per stage
  static constexpr int ATOM = 128 / ELEM;               // elements per swizzle row
  static constexpr int MMA_K = kFP8 ? 32 : 16;          // K of one tcgen05.mma
  static constexpr int KSTEPS = BK / MMA_K;             // 4
  static constexpr int BN_LOAD = (kBN + ATOM - 1) / ATOM * ATOM;
  static constexpr int A_ATOMS = BM / ATOM;
  static constexpr int B_ATOMS = BN_LOAD / ATOM;
  static constexpr int ATOM_BYTES = BK * 128;           // BK rows x 128 bytes
  static constexpr int A_BYTES = A_ATOMS * ATOM_BYTES;
  static constexpr int B_BYTES = B_ATOMS * ATOM_BYTES;
  static constexpr int KSTEP_BYTES = MMA_K * 128;
  // Descriptor strides: SBO = 1024 (8 token rows x 128 B) between K groups,
  // LBO = ATOM_BYTES between 128-byte atoms along M/N.  A single-atom operand
  // never steps along M/N, so its LBO is set to the K-group stride as well.
  static constexpr int A_LBO = A_ATOMS > 1 ? ATOM_BYTES : 1024;
  static constexpr int STAGES = kBN > 128 ? 3 : 5;
  static constexpr int NUM_ACC = 2;
  static constexpr int SF_CHUNKS_B = kFP8 ? (kBN + 127) / 128 : 0;
  static constexpr int SFA_RAW = kFP8 ? 512 : 0;        // up to 4 rows x 128
  static constexpr int SFB_RAW = kFP8 ? ((kBN * 4 + 127) / 128) * 128 : 0;
  static constexpr int UT_A = kFP8 ? 512 : 0;           // 32 rows x 16 bytes
  static constexpr int UT_B = 512 * SF_CHUNKS_B;
  static constexpr int STG_BYTES = 16384;               // 128 rows x 128 bytes
  static constexpr int SF_BUFS = 4;                     // tensor-memory scale buffers
  static constexpr int SFA_COL = NUM_ACC * kBN;
  static constexpr int SFB_COL = SFA_COL + 4 * SF_BUFS;
  static constexpr int TMEM_COLS = 512;
  static_assert(!kFP8 || SFB_COL + 4 * SF_CHUNKS_B * SF_BUFS <= TMEM_COLS, "tmem budget");
  static_assert(NUM_ACC * kBN <= TMEM_COLS, "tmem budget");
  static_assert(kBN % 32 == 0 && kBN <= 256, "block N");

  static constexpr int OFF_B = 0;
  static constexpr int OFF_A = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_STG = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_STG + 2 * STG_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_RAW;
  static constexpr int OFF_UTA = OFF_SFB + STAGES * SFB_RAW;
  static constexpr int OFF_UTB = OFF_UTA + STAGES * UT_A;
  static constexpr int OFF_BAR = (OFF_UTB + STAGES * UT_B + 7) / 8 * 8;
  // barriers: full[S], empty[S], accf[2], acce[2], cbar[2], drain
  static constexpr int NUM_BARS = 2 * STAGES + 2 * NUM_ACC + 2 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Roles' wait sites, reported in DevStatus::where.
enum : int { W_PROD_EMPTY = 0x01, W_PROD_DRAIN = 0x02, W_MMA_ACCE = 0x11, W_MMA_FULL = 0x12,
             W_MMA_DRAIN = 0x13, W_EPI_ACCF = 0x21, W_EPI_C = 0x22 };

// AND-reduce a predicate over the 128 epilogue threads (named barrier 1), so
// that all four epilogue warps take the same branch.
__device__ __forceinline__ bool epi_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(ok))
      : "memory");
  return r != 0;
}

template <bool kFP8, int kBN, int kOut>
__global__ void __launch_bounds__(192, 1)
    kgrouped_wgrad_kernel(const __grid_constant__ WgradParams p) {
  using Cfg = WgradCfg<kFP8, kBN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
  uint64_t *full = bars;
  uint64_t *empty = bars + S;
  uint64_t *accf = bars + 2 * S;
  uint64_t *acce = accf + 2;
  uint64_t *cbar = acce + 2;
  uint64_t *drain = cbar + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], 4);
      mbar_init(&cbar[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tmA);
      prefetch_tmap(&p.tmB);
      if constexpr (kFP8) {
        prefetch_tmap(&p.tmSFA);
        prefetch_tmap(&p.tmSFB);
      }
      const int sf_rows = kFP8 ? Cfg::BK / p.gran_k : 0;
      const uint32_t tx = Cfg::A_BYTES + Cfg::B_BYTES + (kFP8 ? (128 + kBN) * sf_rows : 0);
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_mma_tiles; t += gridDim.x) {
        const int gi = t / p.tiles_per_group;
        const int lt = t - gi * p.tiles_per_group;
        const SchedEntry se = p.sched[gi];
        const int mt = lt / p.n_tiles;
        const int m0 = mt * Cfg::BM;
        const int n0 = (lt - mt * p.n_tiles) * kBN;
        if (p.ks_dev != nullptr && lt == 0 && p.ks_dev[se.expert] != se.k_len)
          atomicCAS(&p.status->code, DEV_OK, DEV_KS_MISMATCH);
        const int nk = (se.k_len + Cfg::BK - 1) / Cfg::BK;
        for (int j = 0; j < nk; ++j, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, lim, p.status, W_PROD_EMPTY, t)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], tx);
          const int k = se.k_off + j * Cfg::BK;
          uint8_t *sa = smem + Cfg::OFF_A + s * Cfg::A_BYTES;
          uint8_t *sb = smem + Cfg::OFF_B + s * Cfg::B_BYTES;
#pragma unroll
          for (int a = 0; a < Cfg::A_ATOMS; ++a)
            tma_load_2d(sa + a * Cfg::ATOM_BYTES, &p.tmA, &full[s], m0 + a * Cfg::ATOM, k);
#pragma unroll
          for (int b = 0; b < Cfg::B_ATOMS; ++b)
            tma_load_2d(sb + b * Cfg::ATOM_BYTES, &p.tmB, &full[s], n0 + b * Cfg::ATOM, k);
          if constexpr (kFP8) {
            tma_load_2d(smem + Cfg::OFF_SFA + s * Cfg::SFA_RAW, &p.tmSFA, &full[s], m0,
                        k / p.gran_k);
            tma_load_2d(smem + Cfg::OFF_SFB + s * Cfg::SFB_RAW, &p.tmSFB, &full[s], n0,
                        k / p.gran_k);
          }
        }
      }
      // Let every load this CTA started land before the CTA can exit.
      const uint32_t armed = it;
      for (uint32_t i = (armed > static_cast<uint32_t>(S) ? armed - S : 0); i < armed; ++i)
        mbar_wait(&full[i % S], (i / S) & 1, abort_flag, lim, p.status, W_PROD_DRAIN,
                  static_cast<int>(i), false);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t it = 0, tl = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.num_mma_tiles; t += gridDim.x, ++tl) {
      const int gi = t / p.tiles_per_group;
      const SchedEntry se = p.sched[gi];
      const int nk = (se.k_len + Cfg::BK - 1) / Cfg::BK;
      const int tail = se.k_len - (nk - 1) * Cfg::BK;  // rows valid in the last stage
      const int b = tl & 1;
      ok = mbar_wait(&acce[b], ((tl >> 1) & 1) ^ 1, abort_flag, lim, p.status, W_MMA_ACCE, t);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + b * kBN;
      for (int j = 0; j < nk; ++j, ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1;
        ok = mbar_wait(&full[s], ph, abort_flag, lim, p.status, W_MMA_FULL, t);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint8_t *sa = smem + Cfg::OFF_A + s * Cfg::A_BYTES;
        uint8_t *sb = smem + Cfg::OFF_B + s * Cfg::B_BYTES;
        if constexpr (kFP8) {
          // Repack the stage's scale bytes into the tensor-memory scale layout:
          // for each 128-row chunk, 32 rows of 16 bytes where row r, word w holds
          // the scales of matrix row 32w + r, one byte per 32-token sub-block.
          const int rows = Cfg::BK / p.gran_k;  // 1 or 4 scale rows per stage
          const uint8_t *ra = smem + Cfg::OFF_SFA + s * Cfg::SFA_RAW;
          const uint8_t *rb = smem + Cfg::OFF_SFB + s * Cfg::SFB_RAW;
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int m = 32 * q + lane;
            if (rows == 1) {
              w[q] = static_cast<uint32_t>(ra[m]) * 0x01010101u;
            } else {
              w[q] = static_cast<uint32_t>(ra[m]) | (static_cast<uint32_t>(ra[128 + m]) << 8) |
                     (static_cast<uint32_t>(ra[256 + m]) << 16) |
                     (static_cast<uint32_t>(ra[384 + m]) << 24);
            }
          }
          *reinterpret_cast<uint4 *>(smem + Cfg::OFF_UTA + s * Cfg::UT_A + 16 * lane) =
              make_uint4(w[0], w[1], w[2], w[3]);
#pragma unroll
          for (int c = 0; c < Cfg::SF_CHUNKS_B; ++c) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int n = 128 * c + 32 * q + lane;
              uint32_t v = 0;
              if (n < kBN) {
                if (rows == 1) {
                  v = static_cast<uint32_t>(rb[n]) * 0x01010101u;
                } else {
                  v = static_cast<uint32_t>(rb[n]) | (static_cast<uint32_t>(rb[kBN + n]) << 8) |
                      (static_cast<uint32_t>(rb[2 * kBN + n]) << 16) |
                      (static_cast<uint32_t>(rb[3 * kBN + n]) << 24);
                }
              }
              w[q] = v;
            }
            *reinterpret_cast<uint4 *>(smem + Cfg::OFF_UTB + s * Cfg::UT_B + 512 * c +
                                       16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
        } else {
          // BF16: an expert's last stage may run past its slice; zero those
          // token rows of both operands so they add nothing.
          if (j == nk - 1 && tail < Cfg::BK) {
            // Row k of an atom occupies bytes [k*128, k*128 + 128) of that atom.
            const int per_atom = (Cfg::BK - tail) * 8;   // 16-byte chunks per atom
            for (int i = lane; i < per_atom * (Cfg::A_ATOMS + Cfg::B_ATOMS); i += 32) {
              const int atom = i / per_atom;
              const int r = i - atom * per_atom;
              uint8_t *base = atom < Cfg::A_ATOMS
                                  ? sa + atom * Cfg::ATOM_BYTES
                                  : sb + (atom - Cfg::A_ATOMS) * Cfg::ATOM_BYTES;
              *reinterpret_cast<uint4 *>(base + tail * 128 + r * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
        }
        __syncwarp();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
          if constexpr (kFP8) {
            const uint32_t sfb = it % Cfg::SF_BUFS;
            const uint32_t sfa_t = tmem_base + Cfg::SFA_COL + 4 * sfb;
            const uint32_t sfb_t = tmem_base + Cfg::SFB_COL + 4 * Cfg::SF_CHUNKS_B * sfb;
            tmem_cp_32x128b_warpx4(sfa_t,
                                   smem_desc(smem_u32(smem + Cfg::OFF_UTA + s * Cfg::UT_A), 0,
                                             128, 0));
#pragma unroll
            for (int c = 0; c < Cfg::SF_CHUNKS_B; ++c)
              tmem_cp_32x128b_warpx4(
                  sfb_t + 4 * c,
                  smem_desc(smem_u32(smem + Cfg::OFF_UTB + s * Cfg::UT_B + 512 * c), 0, 128, 0));
#pragma unroll
            for (int ks = 0; ks < Cfg::KSTEPS; ++ks) {
              const uint64_t ad =
                  smem_desc(a0 + ks * Cfg::KSTEP_BYTES, Cfg::A_LBO, 1024, 2);
              const uint64_t bd =
                  smem_desc(b0 + ks * Cfg::KSTEP_BYTES, Cfg::ATOM_BYTES, 1024, 2);
              mma_mxf8(d_tmem, ad, bd, idesc_mxf8(Cfg::BM, kBN, ks, ks), sfa_t, sfb_t,
                       (j | ks) != 0);
            }
          } else {
#pragma unroll
            for (int ks = 0; ks < Cfg::KSTEPS; ++ks) {
              const uint64_t ad =
                  smem_desc(a0 + ks * Cfg::KSTEP_BYTES, Cfg::A_LBO, 1024, 2);
              const uint64_t bd =
                  smem_desc(b0 + ks * Cfg::KSTEP_BYTES, Cfg::ATOM_BYTES, 1024, 2);
              mma_bf16(d_tmem, ad, bd, idesc_bf16(Cfg::BM, kBN), (j | ks) != 0);
            }
          }
          mma_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&accf[b]);
      __syncwarp();
    }
    // Drain: every tcgen05 op this thread issued completes before tensor
    // memory is released.
    if (lane == 0) mma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, abort_flag, lim, p.status, W_MMA_DRAIN, 0, false);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;               // tensor-memory lane quadrant of this warp
    const int row = 32 * q + lane;        // tile row owned by this thread
    const int etid = threadIdx.x - 64;    // 0..127
    uint32_t tl = 0, nchunk_done = 0;
    uint32_t cuse[2] = {0, 0};
    constexpr bool kHasC = (kOut == OUT_F32_C);
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      const int gi = t / p.tiles_per_group;
      const int lt = t - gi * p.tiles_per_group;
      const int e = p.sched[gi].expert;
      const int mt = lt / p.n_tiles;
      const int m0 = mt * Cfg::BM;
      const int n0 = (lt - mt * p.n_tiles) * kBN;
      const bool mma_tile = t < p.num_mma_tiles;
      const int b = tl & 1;
      if (mma_tile) {
        const bool got =
            mbar_wait(&accf[b], (tl >> 1) & 1, abort_flag, lim, p.status, W_EPI_ACCF, t);
        if (!epi_all(got)) break;
        tc_fence_after();
      }
      const int ncols = min(kBN, p.N - n0);
      const int nch = (ncols + 31) / 32;
      bool ok = true;
      for (int c = 0; c < nch; ++c, ++nchunk_done) {
        const int sbuf = nchunk_done & 1;
        uint8_t *stg = smem + Cfg::OFF_STG + sbuf * Cfg::STG_BYTES;
        if (etid == 0) bulk_wait_read<1>();    // the store that last used stg is done reading
        named_bar_sync(1, 128);
        if (kHasC && etid == 0) {
          mbar_arrive_expect_tx(&cbar[sbuf], 128 * 128);
          tma_load_3d(stg, &p.tmC, &cbar[sbuf], n0 + 32 * c, m0, e);
        }
        float v[32];
        if (mma_tile) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * kBN + 32 * c,
                             r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          if (c == nch - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        if constexpr (kHasC) {
          ok = mbar_wait(&cbar[sbuf], cuse[sbuf] & 1, abort_flag, lim, p.status, W_EPI_C, t);
          cuse[sbuf]++;
          ok = epi_all(ok);
          if (!ok) break;
          const uint8_t *rowp = stg + row * 128;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 cv =
                *reinterpret_cast<const float4 *>(rowp + ((i ^ (row & 7)) << 4));
            v[4 * i + 0] += cv.x;
            v[4 * i + 1] += cv.y;
            v[4 * i + 2] += cv.z;
            v[4 * i + 3] += cv.w;
          }
        }
        if constexpr (kOut == OUT_BF16) {
          uint8_t *rowp = stg + row * 64;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const __nv_bfloat162 pr =
                  __floats2bfloat162_rn(v[8 * i + 2 * h], v[8 * i + 2 * h + 1]);
              w[h] = *reinterpret_cast<const uint32_t *>(&pr);
            }
            *reinterpret_cast<uint4 *>(rowp + ((i ^ ((row >> 1) & 3)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          uint8_t *rowp = stg + row * 128;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4 *>(rowp + ((i ^ (row & 7)) << 4)) =
                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (etid == 0) {
          if constexpr (kOut == OUT_F32_REDUCE)
            tma_reduce_add_3d(&p.tmD, stg, n0 + 32 * c, m0, e);
          else
            tma_store_3d(&p.tmD, stg, n0 + 32 * c, m0, e);
          bulk_commit();
        }
      }
      if (!ok) break;
      if (mma_tile) ++tl;
    }
    if (etid == 0) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

template <bool kFP8, int kBN, int kOut>
cudaError_t launch_wgrad_variant(const WgradParams &p, int grid, cudaStream_t stream) {
  using Cfg = WgradCfg<kFP8, kBN>;
  auto kern = kgrouped_wgrad_kernel<kFP8, kBN, kOut>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  kern<<<grid, 192, Cfg::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

template <bool kFP8, int kBN>
cudaError_t launch_wgrad_bn(const WgradParams &p, int grid, cudaStream_t stream) {
  switch (p.out_mode) {
    case OUT_F32: return launch_wgrad_variant<kFP8, kBN, OUT_F32>(p, grid, stream);
    case OUT_F32_REDUCE: return launch_wgrad_variant<kFP8, kBN, OUT_F32_REDUCE>(p, grid, stream);
    case OUT_F32_C: return launch_wgrad_variant<kFP8, kBN, OUT_F32_C>(p, grid, stream);
    case OUT_BF16: return launch_wgrad_variant<kFP8, kBN, OUT_BF16>(p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg
