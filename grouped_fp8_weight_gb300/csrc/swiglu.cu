// SwiGLU backward fused with the column-block FP8 cast, for sm_103a.
//
// A MoE expert's up/gate projection h = [g | u] (gate half first) feeds
// a = silu(g) * u.  For the upstream gradient da:
//   du = da * silu(g),  dg = da * u * silu'(g),
//   silu(g) = g * s,  silu'(g) = s * (1 + g * (1 - s)),  s = 1 / (1 + e^-g).
// The kernel casts dh = [dg | du] (the up/gate weight gradient's A operand)
// and, optionally, the recomputed a (the down-projection's B operand) with one
// UE8M0 scale per column per gran_k tokens, token-major.
//
// Persistent CTAs (two per SM) walk tiles of 128 tokens x 32 channels of I.
// Thread 0 brings each tile's g, u and da in by TMA (24 KB) into a ring of
// four buffers, so the next three tiles land while this one is processed.  Each thread
// takes 2 rows x 8 channels:
//   pass 1: evaluates them once in FP32, keeps the 48 values in registers and
//           column maxima of |dg|, |du|, |a|; the CTA combines the maxima per
//           token block;
//   pass 2: scales the values by 2^-e and converts with the hardware's
//           saturating RNE E4M3 conversion.
// The evaluation uses explicitly rounded operations (no contraction):
// t = e^-|g| from expf (no overflow), r = 1 / (1 + t) from the hardware
// reciprocal (within 1 ulp), and s = sigma(g), 1 - s taken as r and t * r by
// the sign of g (neither form cancels).
#include <cstdint>
#include <cuda_runtime.h>

#include "wgrad_params.h"

namespace dg {

namespace {

constexpr int kSgT = 128;                    // tokens per tile
constexpr int kSgC = 32;                     // channels of I per tile
constexpr int kSgCg = kSgC / 8;              // channel groups of 8 per tile
constexpr int kSgCols = 24;                  // output columns per thread: 8 dg, 8 du, 8 a
constexpr int kSgRows = 2;                   // rows per thread
static_assert(kSgCols == 24 && kSgCg == 4 && kSgRows == 2, "lane layout and maxima exchange: 24 columns over the 8 lanes of a channel group");
constexpr int kSgIn = kSgT * kSgC * 2;       // one BF16 input tile (8 KB)
constexpr int kSgBuf = 3 * kSgIn;            // g, u, da of one tile
constexpr int kSgRed = 8 * kSgCg * kSgCols * 4;   // per-warp partial maxima
constexpr int kSgStages = 4;                 // input buffers per CTA
constexpr int kSgFac = 4 * kSgCg * kSgCols * 4;   // quantisation factors of up to four token blocks
constexpr int kSgBytes = 4 * kSgCg * kSgCols;      // scale bytes of up to four token blocks
constexpr int kSgSmem =
    kSgStages * kSgBuf + kSgRed + kSgFac + kSgBytes + 8 * kSgStages + 16;   // + barriers, abort flag

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void swiglu_bwd(float g, float u, float da, float &dg, float &du,
                                           float &a) {
  // t = e^-|g| never overflows; r = 1 / (1 + t) (within 1 ulp; 1 + t is in
  // [1, 2], never subnormal).  s = sigma(g) and sn = 1 - s are r and t * r in
  // the order the sign of g gives.
  const float t = expf(-fabsf(g));
  const float r = rcp_approx(__fadd_rn(1.f, t));
  const float tr = __fmul_rn(t, r);
  const float s = g >= 0.f ? r : tr;
  const float sn = g >= 0.f ? tr : r;
  const float silu = __fmul_rn(g, s);
  const float dsilu = __fmul_rn(s, __fadd_rn(1.f, __fmul_rn(g, sn)));
  a = __fmul_rn(silu, u);
  du = __fmul_rn(da, silu);
  dg = __fmul_rn(__fmul_rn(da, u), dsilu);
}

// Exact ceil(log2(amax / 448)) from the float32 bit pattern of amax >= 0:
// amax = f * 2^q, 448 = 1.75 * 2^8: q - 8 + (f > 1.75).  Subnormal amax
// (below 2^-126) gives at most -134 and clamps to -127.
__device__ __forceinline__ int scale_exp_f32(uint32_t bits) {
  const int ef = static_cast<int>((bits >> 23) & 0xFF);
  const int e = (ef == 0) ? -127 : (ef - 127 - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0));
  return max(-127, min(127, e));
}

// 2^-e as a float for e in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2_neg(int e) {
  return e < 127 ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23)
                 : __uint_as_float(1u << 22);
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return static_cast<uint32_t>(r);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t quant4(float4 v, const float *m) {
  return cvt_e4m3x2(v.x * m[0], v.y * m[1]) | (cvt_e4m3x2(v.z * m[2], v.w * m[3]) << 16);
}

template <int kGran, bool kWithA>
__global__ void __launch_bounds__(256, 2) swiglu_bwd_cast_kernel(const __grid_constant__ SwigluArgs p) {
  extern __shared__ __align__(128) uint8_t sg_smem[];
  float *red = reinterpret_cast<float *>(sg_smem + kSgStages * kSgBuf);     // [8 warps][4][24]
  float *fac = reinterpret_cast<float *>(sg_smem + kSgStages * kSgBuf + kSgRed);   // [blocks][4][24]
  uint8_t *sbytes = sg_smem + kSgStages * kSgBuf + kSgRed + kSgFac;        // [blocks][4][24]
  uint64_t *full =
      reinterpret_cast<uint64_t *>(sg_smem + kSgStages * kSgBuf + kSgRed + kSgFac + kSgBytes);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(full + kSgStages);
  const int tid = threadIdx.x;
  const int w = tid >> 5, l = tid & 31;
  const int I = p.I;
  // thread: channel group cg (8 channels), rows 16w + 8i + rs (i = 0, 1)
  const int cg = l & 3, rs = l >> 2;
  const int n_tiles = p.n_tt * p.n_tc;

  if (tid == 0) {
    for (int k = 0; k < kSgStages; ++k) mbar_init(&full[k], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // g at channel c0, u at I + c0 (columns past 2I read as 0; those past I
  // in g's box are u's and are never used), da at c0; rows past T read as 0
  auto issue = [&](int u, int b) {
    const int tt = u / p.n_tc, tc = u - tt * p.n_tc;
    uint8_t *dst = sg_smem + b * kSgBuf;
    mbar_arrive_expect_tx(&full[b], kSgBuf);
    tma_load_2d(dst, &p.tm_h, &full[b], tc * kSgC, tt * kSgT);
    tma_load_2d(dst + kSgIn, &p.tm_h, &full[b], I + tc * kSgC, tt * kSgT);
    tma_load_2d(dst + 2 * kSgIn, &p.tm_da, &full[b], tc * kSgC, tt * kSgT);
  };
  int issued = 0;
  if (tid == 0) {
    for (int k = 0; k < kSgStages; ++k) {
      const int u = blockIdx.x + k * gridDim.x;
      if (u < n_tiles) {
        issue(u, k);
        ++issued;
      }
    }
  }

  // Column-wise evaluation of this thread's row i of the tile in buffer b.
  auto eval_row = [&](const uint8_t *buf, int i, float (&vg)[8], float (&vu)[8], float (&va)[8]) {
    const int r = 16 * w + 8 * i + rs;
    const uint4 gv = *reinterpret_cast<const uint4 *>(buf + r * (kSgC * 2) + 16 * cg);
    const uint4 uv = *reinterpret_cast<const uint4 *>(buf + kSgIn + r * (kSgC * 2) + 16 * cg);
    const uint4 dv = *reinterpret_cast<const uint4 *>(buf + 2 * kSgIn + r * (kSgC * 2) + 16 * cg);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
    const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const bool hi = k & 1;
      const float g = hi ? bf16_hi(gw[k >> 1]) : bf16_lo(gw[k >> 1]);
      const float u = hi ? bf16_hi(uw[k >> 1]) : bf16_lo(uw[k >> 1]);
      const float d = hi ? bf16_hi(dw[k >> 1]) : bf16_lo(dw[k >> 1]);
      swiglu_bwd(g, u, d, vg[k], vu[k], va[k]);
    }
  };

  int it = 0;
  for (int u = blockIdx.x; u < n_tiles; u += gridDim.x, ++it) {
    const int b = it % kSgStages;
    const uint32_t par = static_cast<uint32_t>(it / kSgStages) & 1u;
    const bool got = mbar_wait(&full[b], par, abort_flag, p.wait_limit_ns, p.status, 0x51, u);
    if (__syncthreads_or(!got)) break;   // the whole CTA leaves together
    const uint8_t *buf = sg_smem + b * kSgBuf;
    const int tt = u / p.n_tc, tc = u - tt * p.n_tc;
    const int64_t t0 = static_cast<int64_t>(tt) * kSgT;
    const int col = tc * kSgC + 8 * cg;
    const bool col_ok = col < I;

    // ---- pass 1: evaluate once (values kept in registers), column maxima
    // (inputs are finite: a float maximum of magnitudes)
    float vg[kSgRows][8], vu[kSgRows][8], va[kSgRows][8];
    float mx[kSgCols];
#pragma unroll
    for (int k = 0; k < kSgCols; ++k) mx[k] = 0.f;
#pragma unroll
    for (int i = 0; i < kSgRows; ++i) {
      eval_row(buf, i, vg[i], vu[i], va[i]);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        mx[k] = fmaxf(mx[k], fabsf(vg[i][k]));
        mx[8 + k] = fmaxf(mx[8 + k], fabsf(vu[i][k]));
        if constexpr (kWithA) mx[16 + k] = fmaxf(mx[16 + k], fabsf(va[i][k]));
      }
    }
    // every read of buffer b is done: it takes the tile kSgStages steps
    // ahead (issued after the barrier below)
    // The eight lanes of a channel group (rs = 0..7, lane bits 2-4) hold the
    // rows of one warp's 16.  Each exchange sends half of the columns still
    // held and keeps the other half (the half the lane's rs bit names), so
    // after three the lane holds the maxima of columns 3 rs .. 3 rs + 2 over
    // all 16 rows: 21 shuffles instead of 72.
    float m12[12], m6[6], m3[3];
    {
      const bool hb = (rs >> 2) & 1;
#pragma unroll
      for (int k = 0; k < 12; ++k) {
        const float send = hb ? mx[k] : mx[k + 12];
        const float keep = hb ? mx[k + 12] : mx[k];
        m12[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
      }
      const bool hm = (rs >> 1) & 1;
#pragma unroll
      for (int k = 0; k < 6; ++k) {
        const float send = hm ? m12[k] : m12[k + 6];
        const float keep = hm ? m12[k + 6] : m12[k];
        m6[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 8));
      }
      const bool hl = rs & 1;
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const float send = hl ? m6[k] : m6[k + 3];
        const float keep = hl ? m6[k + 3] : m6[k];
        m3[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 4));
      }
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) red[(w * kSgCg + cg) * kSgCols + 3 * rs + k] = m3[k];
    __syncthreads();
    if (tid == 0) {
      const int un = u + kSgStages * gridDim.x;
      if (un < n_tiles) {
        issue(un, b);
        ++issued;
      }
    }
    // block maxima (gran 128 over all eight warps, gran 32 over warps 2b,
    // 2b + 1), one scale per (block, column): its factor 2^-e and its byte
    // e + 127, written apart from the maxima so that one barrier covers both
    // (the next tile's maxima are written after its first barrier, this
    // tile's factors read before it)
    constexpr int kBlocks = kSgT / kGran;
    constexpr int kWpb = 8 / kBlocks;          // warps per block
    constexpr int kItems = kBlocks * kSgCg * kSgCols;
#pragma unroll
    for (int idx = tid; idx < kItems; idx += 256) {
      const int bb = idx / (kSgCg * kSgCols), rest = idx % (kSgCg * kSgCols);
      uint32_t fin = 0;
#pragma unroll
      for (int ww = 0; ww < kWpb; ++ww)
        fin = max(fin, __float_as_uint(red[(bb * kWpb + ww) * kSgCg * kSgCols + rest]));
      const int e = scale_exp_f32(fin);
      fac[idx] = pow2_neg(e);
      sbytes[idx] = static_cast<uint8_t>(e + 127);
    }
    __syncthreads();
    const int blk = (16 * w) / kGran;          // this thread's token block in the tile
    const int sidx = (blk * kSgCg + cg) * kSgCols;
    float mul[kSgCols];
#pragma unroll
    for (int k = 0; k < kSgCols; k += 4) {
      const float4 m4 = *reinterpret_cast<const float4 *>(fac + sidx + k);
      mul[k] = m4.x;
      mul[k + 1] = m4.y;
      mul[k + 2] = m4.z;
      mul[k + 3] = m4.w;
    }
    // scale bytes: the lanes holding the block's first row write them
    const int64_t tb = t0 + 16 * w;
    if (col_ok && rs == 0 && (16 * w) % kGran == 0 && tb < p.T) {
      const int64_t srow = tb / kGran;
      const uint2 *sb = reinterpret_cast<const uint2 *>(sbytes + sidx);
      *reinterpret_cast<uint2 *>(p.sf_dh + srow * 2 * I + col) = sb[0];
      *reinterpret_cast<uint2 *>(p.sf_dh + srow * 2 * I + I + col) = sb[1];
      if constexpr (kWithA) *reinterpret_cast<uint2 *>(p.sf_a + srow * I + col) = sb[2];
    }

    // ---- pass 2: quantise the kept values, store
#pragma unroll
    for (int i = 0; i < kSgRows; ++i) {
      const int64_t t = t0 + 16 * w + 8 * i + rs;
      if (col_ok && t < p.T) {
        const uint32_t og0 = quant4(make_float4(vg[i][0], vg[i][1], vg[i][2], vg[i][3]), mul);
        const uint32_t og1 = quant4(make_float4(vg[i][4], vg[i][5], vg[i][6], vg[i][7]), mul + 4);
        const uint32_t ou0 = quant4(make_float4(vu[i][0], vu[i][1], vu[i][2], vu[i][3]), mul + 8);
        const uint32_t ou1 = quant4(make_float4(vu[i][4], vu[i][5], vu[i][6], vu[i][7]), mul + 12);
        __stcs(reinterpret_cast<uint2 *>(p.q_dh + t * 2 * I + col), make_uint2(og0, og1));
        __stcs(reinterpret_cast<uint2 *>(p.q_dh + t * 2 * I + I + col), make_uint2(ou0, ou1));
        if constexpr (kWithA) {
          const uint32_t oa0 = quant4(make_float4(va[i][0], va[i][1], va[i][2], va[i][3]), mul + 16);
          const uint32_t oa1 = quant4(make_float4(va[i][4], va[i][5], va[i][6], va[i][7]), mul + 20);
          __stcs(reinterpret_cast<uint2 *>(p.q_a + t * I + col), make_uint2(oa0, oa1));
        }
      }
    }
  }
  // Leaving early (a wait ran out): let the copies in flight land (bounded).
  if (tid == 0)
    for (int k = it; k < issued; ++k)
      if (!mbar_wait(&full[k % kSgStages], static_cast<uint32_t>(k / kSgStages) & 1u, abort_flag,
                     drain_limit_ns(p.wait_limit_ns), p.status, 0x52, k, false))
        break;
}

template <int kGran, bool kWithA>
cudaError_t launch_sg(const SwigluArgs &p, int ctas, cudaStream_t stream) {
  // attribute set once per process (thread-safe static initialisation)
  static const cudaError_t setup = cudaFuncSetAttribute(
      swiglu_bwd_cast_kernel<kGran, kWithA>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSgSmem);
  if (setup != cudaSuccess) return setup;
  const int64_t tiles = static_cast<int64_t>(p.n_tt) * p.n_tc;
  const int grid = static_cast<int>(tiles < ctas ? tiles : ctas);
  swiglu_bwd_cast_kernel<kGran, kWithA><<<grid, 256, kSgSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_swiglu_bwd_cast(const SwigluArgs &p, int gran_k, int ctas, cudaStream_t stream) {
  const bool with_a = (p.q_a != nullptr);
  if (gran_k == 128)
    return with_a ? launch_sg<128, true>(p, ctas, stream) : launch_sg<128, false>(p, ctas, stream);
  return with_a ? launch_sg<32, true>(p, ctas, stream) : launch_sg<32, false>(p, ctas, stream);
}

}  // namespace dg
