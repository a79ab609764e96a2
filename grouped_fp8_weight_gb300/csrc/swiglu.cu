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
// One CTA covers 128 tokens x 64 channels of I; each thread loads 4 rows x
// 8 channels of g, u and da (16-byte loads), then
//   pass 1: evaluates them once in FP32, parks the values in shared memory
//           (96 KB) and keeps column maxima of |dg|, |du|, |a|; the CTA
//           combines the maxima per token block;
//   pass 2: scales the parked values by 2^-e and converts with the hardware's
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

constexpr int kSgT = 128;                    // tokens per CTA
constexpr int kSgC = 64;                     // channels of I per CTA
constexpr int kSgCols = 24;                  // output columns per thread: 8 dg, 8 du, 8 a
constexpr int kSgRows = 4;                   // rows per thread
// Evaluated values parked between the passes: per thread 4 rows x 24 floats,
// as float4 slot j of thread t at [j][t] (consecutive threads, consecutive
// 16 bytes: conflict-free).
constexpr int kSgVals = kSgRows * kSgCols / 4 * 256 * 16;      // 96 KB
constexpr int kSgRed = 8 * 8 * kSgCols * 4;                    // per-warp partial maxima
constexpr int kSgSmem = kSgVals + kSgRed;

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
__global__ void __launch_bounds__(256, 2) swiglu_bwd_cast_kernel(const SwigluArgs p) {
  extern __shared__ __align__(16) uint8_t sg_smem[];
  float4 *vals = reinterpret_cast<float4 *>(sg_smem);                       // [24][256]
  float *red = reinterpret_cast<float *>(sg_smem + kSgVals);                // [8 warps][8][24]
  const int tid = threadIdx.x;
  const int w = tid >> 5, l = tid & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kSgT;
  const int I = p.I;
  // thread: channel group cg (8 channels), rows 16w + 4i + rs (i = 0..3)
  const int cg = l & 7, rs = l >> 3;
  const int col = blockIdx.y * kSgC + 8 * cg;
  const bool col_ok = col < I;
  const uint16_t *h = static_cast<const uint16_t *>(p.h);
  const uint16_t *dap = static_cast<const uint16_t *>(p.da);

  // ---- loads: 4 rows x (g, u, da), 16 bytes each (rows past T read as 0)
  uint4 gv[kSgRows], uv[kSgRows], dv[kSgRows];
#pragma unroll
  for (int i = 0; i < kSgRows; ++i) {
    const int64_t t = t0 + 16 * w + 4 * i + rs;
    const bool ok = col_ok && t < p.T;
    gv[i] = ok ? __ldcs(reinterpret_cast<const uint4 *>(h + t * 2 * I + col)) : make_uint4(0, 0, 0, 0);
    uv[i] = ok ? __ldcs(reinterpret_cast<const uint4 *>(h + t * 2 * I + I + col)) : make_uint4(0, 0, 0, 0);
    dv[i] = ok ? __ldcs(reinterpret_cast<const uint4 *>(dap + t * I + col)) : make_uint4(0, 0, 0, 0);
  }

  // ---- pass 1: evaluate once, park the values, keep column maxima
  // (non-negative float bit patterns order like the floats: integer maxima)
  uint32_t mx[kSgCols];
#pragma unroll
  for (int k = 0; k < kSgCols; ++k) mx[k] = 0;
#pragma unroll
  for (int i = 0; i < kSgRows; ++i) {
    const uint32_t gw[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
    const uint32_t uw[4] = {uv[i].x, uv[i].y, uv[i].z, uv[i].w};
    const uint32_t dw[4] = {dv[i].x, dv[i].y, dv[i].z, dv[i].w};
    float vg[8], vu[8], va[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const bool hi = k & 1;
      const float g = hi ? bf16_hi(gw[k >> 1]) : bf16_lo(gw[k >> 1]);
      const float u = hi ? bf16_hi(uw[k >> 1]) : bf16_lo(uw[k >> 1]);
      const float d = hi ? bf16_hi(dw[k >> 1]) : bf16_lo(dw[k >> 1]);
      swiglu_bwd(g, u, d, vg[k], vu[k], va[k]);
      mx[k] = max(mx[k], __float_as_uint(fabsf(vg[k])));
      mx[8 + k] = max(mx[8 + k], __float_as_uint(fabsf(vu[k])));
      if constexpr (kWithA) mx[16 + k] = max(mx[16 + k], __float_as_uint(fabsf(va[k])));
    }
    const int j = 6 * i;
    vals[(j + 0) * 256 + tid] = make_float4(vg[0], vg[1], vg[2], vg[3]);
    vals[(j + 1) * 256 + tid] = make_float4(vg[4], vg[5], vg[6], vg[7]);
    vals[(j + 2) * 256 + tid] = make_float4(vu[0], vu[1], vu[2], vu[3]);
    vals[(j + 3) * 256 + tid] = make_float4(vu[4], vu[5], vu[6], vu[7]);
    if constexpr (kWithA) {
      vals[(j + 4) * 256 + tid] = make_float4(va[0], va[1], va[2], va[3]);
      vals[(j + 5) * 256 + tid] = make_float4(va[4], va[5], va[6], va[7]);
    }
  }
  // lanes with the same channel group (rs = 0..3) hold rows of one warp's 16
#pragma unroll
  for (int k = 0; k < kSgCols; ++k) {
    mx[k] = max(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], 8));
    mx[k] = max(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], 16));
  }
  if (l < 8) {
#pragma unroll
    for (int k = 0; k < kSgCols; ++k) red[(w * 8 + cg) * kSgCols + k] = __uint_as_float(mx[k]);
  }
  __syncthreads();
  // block maxima: gran 128 over all eight warps, gran 32 over warps 2b, 2b + 1
  constexpr int kBlocks = kSgT / kGran;
  constexpr int kWpb = 8 / kBlocks;          // warps per block
  constexpr int kItems = kBlocks * 8 * kSgCols;
  constexpr int kPer = (kItems + 255) / 256;
  uint32_t fin[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int idx = tid + 256 * i;
    fin[i] = 0;
    if (idx < kItems) {
      const int b = idx / (8 * kSgCols), rest = idx % (8 * kSgCols);
#pragma unroll
      for (int ww = 0; ww < kWpb; ++ww)
        fin[i] = max(fin[i], __float_as_uint(red[(b * kWpb + ww) * 8 * kSgCols + rest]));
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int idx = tid + 256 * i;
    if (idx < kItems) red[idx] = __uint_as_float(fin[i]);
  }
  __syncthreads();
  const int blk = (16 * w) / kGran;          // this thread's token block in the tile
  float mul[kSgCols];
  uint32_t sfw[6] = {0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int k = 0; k < kSgCols; ++k) {
    const int e = scale_exp_f32(__float_as_uint(red[(blk * 8 + cg) * kSgCols + k]));
    mul[k] = pow2_neg(e);
    sfw[k >> 2] |= static_cast<uint32_t>(e + 127) << (8 * (k & 3));
  }
  // scale bytes: the lanes holding the block's first row write them
  const int64_t tb = t0 + 16 * w;
  if (col_ok && rs == 0 && (16 * w) % kGran == 0 && tb < p.T) {
    const int64_t srow = tb / kGran;
    *reinterpret_cast<uint2 *>(p.sf_dh + srow * 2 * I + col) = make_uint2(sfw[0], sfw[1]);
    *reinterpret_cast<uint2 *>(p.sf_dh + srow * 2 * I + I + col) = make_uint2(sfw[2], sfw[3]);
    if constexpr (kWithA)
      *reinterpret_cast<uint2 *>(p.sf_a + srow * I + col) = make_uint2(sfw[4], sfw[5]);
  }

  // ---- pass 2: quantise the parked values, store
#pragma unroll
  for (int i = 0; i < kSgRows; ++i) {
    const int64_t t = t0 + 16 * w + 4 * i + rs;
    const int j = 6 * i;
    const uint32_t og0 = quant4(vals[(j + 0) * 256 + tid], mul);
    const uint32_t og1 = quant4(vals[(j + 1) * 256 + tid], mul + 4);
    const uint32_t ou0 = quant4(vals[(j + 2) * 256 + tid], mul + 8);
    const uint32_t ou1 = quant4(vals[(j + 3) * 256 + tid], mul + 12);
    if (col_ok && t < p.T) {
      __stcs(reinterpret_cast<uint2 *>(p.q_dh + t * 2 * I + col), make_uint2(og0, og1));
      __stcs(reinterpret_cast<uint2 *>(p.q_dh + t * 2 * I + I + col), make_uint2(ou0, ou1));
    }
    if constexpr (kWithA) {
      const uint32_t oa0 = quant4(vals[(j + 4) * 256 + tid], mul + 16);
      const uint32_t oa1 = quant4(vals[(j + 5) * 256 + tid], mul + 20);
      if (col_ok && t < p.T)
        __stcs(reinterpret_cast<uint2 *>(p.q_a + t * I + col), make_uint2(oa0, oa1));
    }
  }
}

template <int kGran, bool kWithA>
cudaError_t launch_sg(const SwigluArgs &p, cudaStream_t stream) {
  // attribute set once per process (thread-safe static initialisation)
  static const cudaError_t setup = cudaFuncSetAttribute(
      swiglu_bwd_cast_kernel<kGran, kWithA>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSgSmem);
  if (setup != cudaSuccess) return setup;
  const dim3 grid(static_cast<unsigned>((p.T + kSgT - 1) / kSgT),
                  static_cast<unsigned>((p.I + kSgC - 1) / kSgC));
  swiglu_bwd_cast_kernel<kGran, kWithA><<<grid, 256, kSgSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_swiglu_bwd_cast(const SwigluArgs &p, int gran_k, cudaStream_t stream) {
  const bool with_a = (p.q_a != nullptr);
  if (gran_k == 128)
    return with_a ? launch_sg<128, true>(p, stream) : launch_sg<128, false>(p, stream);
  return with_a ? launch_sg<32, true>(p, stream) : launch_sg<32, false>(p, stream);
}

}  // namespace dg
