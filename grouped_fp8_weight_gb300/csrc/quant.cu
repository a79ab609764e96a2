// Column-block FP8 casts (with optional physical transpose and MoE-layout row
// gather) for sm_103a.
//
// For every gran_k-token block and column of a matrix x[T, C]:
//   amax = max |x|, e = clamp(ceil(log2(amax / 448)), -127, 127),
//   sf = e + 127 (UE8M0), q = E4M3 round-to-nearest-even of x * 2^-e.
//
// Sources:
//   BF16       x[T, C] as stored.
//   E4M3 tiles the forward pass's stored activations: codes [T, C] with one
//              UE8M0 scale per token per 128 channels (x = e4m3 * 2^(b - 127));
//              dequantised exactly in registers, then cast by columns.
// Optional row gather (the MoE layout): output row t takes source row
// src_rows[t], or zeros where src_rows[t] == -1 (an expert's padding).
//
// HBM-bound: BF16 source 2 bytes read and 1 (+1/gran_k) written per element,
// E4M3 source 1 (+1/128) read.  One CTA covers 128 tokens x 256 channels.
// Each thread loads 16 rows x 8 channels with independent vector loads,
// reduces |x| (BF16: packed 16-bit maxima on the bit patterns, exact because
// non-negative floats order like their bit patterns; E4M3: float maxima of
// the dequantised values), combines the eight warps' partial maxima in shared
// memory, and converts with the hardware's saturating RNE E4M3 conversion.
// The channel-major variant transposes 4x4 byte blocks in registers and
// stages the tile in a swizzled shared-memory buffer so that both the shared
// stores and the 128-byte global row stores are conflict-free and coalesced.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "wgrad_params.h"

namespace dg {

namespace {

constexpr int kTileT = 128;
constexpr int kTileC = 256;

// Exact ceil(log2(amax / 448)) from the BF16 bit pattern of amax >= 0:
// amax = f * 2^q with f in [1, 2) and 448 = 1.75 * 2^8, so the result is
// q - 8 when f <= 1.75 and q - 7 otherwise.  Zero and subnormal amax (below
// 2^-126) clamp to -127.
__device__ __forceinline__ int scale_exp_from_bf16(uint32_t h) {
  const int ef = static_cast<int>((h >> 7) & 0xFF);
  const int mant = static_cast<int>(h & 0x7F);
  const int e = (ef == 0) ? -127 : (ef - 127 - 8 + (mant > 0x60 ? 1 : 0));
  return max(-127, min(127, e));
}

// Exact ceil(log2(amax / 448)) from the float32 bit pattern of a = amax * 2^-8
// (the E4M3 source keeps its dequantised values scaled by 2^-8 so that every
// one is finite and exact in float32).  amax / 448 = a / 1.75, so with
// a = f * 2^q (f in [1, 2)) the result is q + (f > 1.75).  Subnormal a (its
// mantissa m, a = m * 2^-149) takes q from m's top bit.
__device__ __forceinline__ int scale_exp_from_f32_shifted(uint32_t bits) {
  const int ef = static_cast<int>((bits >> 23) & 0xFF);
  const uint32_t mant = bits & 0x7FFFFFu;
  int e;
  if (ef != 0) {
    e = ef - 127 + (mant > 0x600000u ? 1 : 0);
  } else if (mant == 0) {
    e = -127;
  } else {
    const int p = 31 - __clz(static_cast<int>(mant));
    e = p - 149 + (4u * mant > (7u << p) ? 1 : 0);
  }
  return max(-127, min(127, e));
}

// 2^(b - 135) as a float (normal for b >= 9, subnormal below): the factor
// that takes an E4M3 value to its dequantised value times 2^-8.
__device__ __forceinline__ float pow2_b_minus_135(uint32_t b) {
  return b >= 9 ? __uint_as_float((b - 8) << 23) : __uint_as_float(1u << (b + 14));
}

// Two floats -> two E4M3 bytes (lo in the low byte), RNE, saturating.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return static_cast<uint32_t>(r);
}

// Two E4M3 bytes (lo in the low byte) -> two exact floats.  kFresh: decode
// again instead of reusing an earlier decode of the same bytes (which would
// keep every decoded value of the tile live in registers).
template <bool kFresh = false>
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t two) {
  uint32_t h;
  if constexpr (kFresh)
    asm volatile("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(two & 0xFFFFu)));
  else
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(two & 0xFFFFu)));
  return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

__device__ __forceinline__ uint32_t quant_word(uint32_t w, float m_lo, float m_hi) {
  const float lo = __uint_as_float(w << 16) * m_lo;
  const float hi = __uint_as_float(w & 0xFFFF0000u) * m_hi;
  return cvt_e4m3x2(lo, hi);
}

// Eight E4M3 source codes of one row (dequantised, times 2^-8 = the factor
// p) quantised with per-column factors 2^sh, sh = 135 - b (b = the column's
// new scale byte): ma = 2^min(sh, 127), and, only where sh > 127 (kBig),
// a second factor 2^(sh - 127) so that every factor stays representable.
// Every product is exact.
template <bool kBig>
__device__ __forceinline__ uint2 requant8(uint2 c, float p, const float *ma, const uint32_t *sfw) {
  uint32_t out[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t w = h ? c.y : c.x;
    const float2 a = e4m3x2_to_f32<true>(w);
    const float2 b = e4m3x2_to_f32<true>(w >> 16);
    const int k = 4 * h;
    float y[4] = {a.x * p * ma[k], a.y * p * ma[k + 1], b.x * p * ma[k + 2], b.y * p * ma[k + 3]};
    if constexpr (kBig) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int bo = static_cast<int>((sfw[h] >> (8 * j)) & 0xFFu);
        y[j] *= __uint_as_float(static_cast<uint32_t>(max(8 - bo, 0) + 127) << 23);
      }
    }
    out[h] = cvt_e4m3x2(y[0], y[1]) | (cvt_e4m3x2(y[2], y[3]) << 16);
  }
  return make_uint2(out[0], out[1]);
}

// Gather: the source rows of a tile's 128 output rows t0.., read once into
// shared memory by the first 128 threads (past T: -1; an entry outside
// [-1, T_src) is recorded in the status word and read as -1), so that every
// thread's row loads can then be issued together.  Ends with a barrier.
template <bool kGather>
__device__ __forceinline__ void stage_rows(const CastArgs &a, int64_t t0, int *rows_s) {
  if constexpr (kGather) {
    if (threadIdx.x < kTileT) {
      const int64_t t = t0 + threadIdx.x;
      int s = t < a.T ? __ldg(a.src_rows + t) : -1;
      if (s < -1 || s >= a.T_src) {
        atomicCAS(&a.status->code, DEV_OK, DEV_BAD_ROW);
        s = -1;
      }
      rows_s[threadIdx.x] = s;
    }
    __syncthreads();
  }
}

// Source row of the tile's row i (-1: not read): the staged entry, or t0 + i
// itself without the gather.
template <bool kGather>
__device__ __forceinline__ int64_t tile_source_row(const CastArgs &a, const int *rows_s,
                                                   int64_t t0, int i, bool col_ok) {
  if constexpr (kGather) {
    return col_ok ? rows_s[i] : -1;
  } else {
    const int64_t t = t0 + i;
    return (col_ok && t < a.T) ? t : -1;
  }
}

// The factor taking row i's E4M3 values to their dequantised values x 2^-8.
__device__ __forceinline__ float row_factor(const uint32_t (&sbw)[4], int i) {
  return pow2_b_minus_135((sbw[i >> 2] >> (8 * (i & 3))) & 0xFFu);
}

template <bool kBig>
__device__ __forceinline__ void requant_rows(uint2 (&o)[16], const uint2 (&v8)[16],
                                             const uint32_t (&sbw)[4], const float (&ma)[8],
                                             const uint32_t (&sfw)[2]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i] = requant8<kBig>(v8[i], row_factor(sbw, i), ma, sfw);
}

template <int kGran, bool kChannel, bool kFp8Src, bool kGather>
__global__ void __launch_bounds__(256, 2) cast_colblock_kernel(const CastArgs a) {
  __shared__ uint4 red[8][32][kFp8Src ? 2 : 1];
  __shared__ __align__(16) uint8_t tq[kChannel ? kTileC * kTileT : 16];
  __shared__ int rows_s[kGather ? kTileT : 1];
  __shared__ __align__(16) float fac_s[4 * kTileC];     // per (token block, column): factor
  __shared__ __align__(8) uint8_t sb_s[4 * kTileC];     // and scale byte
  const int w = threadIdx.x >> 5;
  const int l = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTileT;
  const int C = a.C;
  const int c0 = blockIdx.y * kTileC;
  const int col = c0 + 8 * l;
  const bool col_ok = col < C;
  stage_rows<kGather>(a, t0, rows_s);

  // ---- loads and column maxima
  uint4 v[kFp8Src ? 1 : 16];
  uint2 v8[kFp8Src ? 16 : 1];
  uint32_t sbw[4] = {0, 0, 0, 0};   // E4M3 source: scale byte of row i in byte i % 4 of word i / 4
  uint32_t m[4] = {0, 0, 0, 0};
  float fm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if constexpr (!kFp8Src) {
    const uint16_t *x = static_cast<const uint16_t *>(a.x);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t r = tile_source_row<kGather>(a, rows_s, t0, 16 * w + i, col_ok);
      v[i] = r >= 0 ? __ldcs(reinterpret_cast<const uint4 *>(x + r * C + col))
                    : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      m[0] = __vmaxu2(m[0], v[i].x & 0x7FFF7FFFu);
      m[1] = __vmaxu2(m[1], v[i].y & 0x7FFF7FFFu);
      m[2] = __vmaxu2(m[2], v[i].z & 0x7FFF7FFFu);
      m[3] = __vmaxu2(m[3], v[i].w & 0x7FFF7FFFu);
    }
    red[w][l][0] = make_uint4(m[0], m[1], m[2], m[3]);
  } else {
    // Rows not read hold code 0 (value 0 at any scale).
    const uint8_t *x = static_cast<const uint8_t *>(a.x);
    const int tiles = C / 128;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t r = tile_source_row<kGather>(a, rows_s, t0, 16 * w + i, col_ok);
      v8[i] = r >= 0 ? __ldcs(reinterpret_cast<const uint2 *>(x + r * C + col)) : make_uint2(0, 0);
      const uint32_t b = r >= 0 ? __ldg(a.x_sf + r * tiles + col / 128) : 0u;
      sbw[i >> 2] |= b << (8 * (i & 3));
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float p = pow2_b_minus_135((sbw[i >> 2] >> (8 * (i & 3))) & 0xFFu);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float2 f = e4m3x2_to_f32((h & 2 ? v8[i].y : v8[i].x) >> (16 * (h & 1)));
        fm[2 * h] = fmaxf(fm[2 * h], fabsf(f.x * p));
        fm[2 * h + 1] = fmaxf(fm[2 * h + 1], fabsf(f.y * p));
      }
    }
    red[w][l][0] = make_uint4(__float_as_uint(fm[0]), __float_as_uint(fm[1]),
                              __float_as_uint(fm[2]), __float_as_uint(fm[3]));
    red[w][l][kFp8Src ? 1 : 0] = make_uint4(__float_as_uint(fm[4]), __float_as_uint(fm[5]),
                                            __float_as_uint(fm[6]), __float_as_uint(fm[7]));
  }
  __syncthreads();

  // ---- block maxima -> scale exponents and quantisation factors, one per
  // (token block, column), computed once (red as [warp][column] maxima:
  // BF16 bit patterns, or float bit patterns of non-negative values, both
  // ordered like the values they encode)
  constexpr int kWarps = (kGran == 128) ? 8 : 2;
  constexpr int kItems = (kTileT / kGran) * kTileC;
#pragma unroll
  for (int it = threadIdx.x; it < kItems; it += 256) {
    const int bb = it / kTileC, c = it % kTileC;
    uint32_t mx = 0;
    int e;
    if constexpr (!kFp8Src) {
      const uint16_t *red16 = reinterpret_cast<const uint16_t *>(&red[0][0][0]);
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww)
        mx = max(mx, static_cast<uint32_t>(red16[(bb * kWarps + ww) * kTileC + c]));
      e = scale_exp_from_bf16(mx);
      fac_s[it] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    } else {
      const uint32_t *red32 = reinterpret_cast<const uint32_t *>(&red[0][0][0]);
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) mx = max(mx, red32[(bb * kWarps + ww) * kTileC + c]);
      e = scale_exp_from_f32_shifted(mx);
      // y = (x * 2^-8) * 2^sh with sh = 8 - e in [-119, 135]: the first factor
      // 2^min(sh, 127), the rest applied where a column needs it
      fac_s[it] = __uint_as_float(static_cast<uint32_t>(min(8 - e, 127) + 127) << 23);
    }
    sb_s[it] = static_cast<uint8_t>(e + 127);
  }
  __syncthreads();
  const int blk = (16 * w) / kGran;
  float mul[8], ma[8];
  {
    const float4 f0 = *reinterpret_cast<const float4 *>(fac_s + blk * kTileC + 8 * l);
    const float4 f1 = *reinterpret_cast<const float4 *>(fac_s + blk * kTileC + 8 * l + 4);
    const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      mul[k] = f[k];
      ma[k] = f[k];
    }
  }
  const uint2 sb2 = *reinterpret_cast<const uint2 *>(sb_s + blk * kTileC + 8 * l);
  const uint32_t sfw[2] = {sb2.x, sb2.y};
  // E4M3 source: a column needs the second factor (sh > 127: scale byte below 8)
  const bool big = kFp8Src && ((((sfw[0] - 0x08080808u) & ~sfw[0] & 0x80808080u) |
                                ((sfw[1] - 0x08080808u) & ~sfw[1] & 0x80808080u)) != 0);
  if (col_ok) {
    if constexpr (kGran == 128) {
      if (w == 0)
        *reinterpret_cast<uint2 *>(a.sf + (t0 / 128) * C + col) = make_uint2(sfw[0], sfw[1]);
    } else {
      const int64_t tb = t0 + 16 * w;
      if ((w & 1) == 0 && tb < a.T)
        *reinterpret_cast<uint2 *>(a.sf + (tb / 32) * C + col) = make_uint2(sfw[0], sfw[1]);
    }
  }

  // ---- quantise and store (rows past T are not written; gathered padding
  // rows are zeros)
  uint8_t *q = a.q;
  const int64_t T = a.T;
  uint2 o[16];
  if constexpr (!kFp8Src) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      o[i] = make_uint2(
          quant_word(v[i].x, mul[0], mul[1]) | (quant_word(v[i].y, mul[2], mul[3]) << 16),
          quant_word(v[i].z, mul[4], mul[5]) | (quant_word(v[i].w, mul[6], mul[7]) << 16));
  } else {
    if (big)
      requant_rows<true>(o, v8, sbw, ma, sfw);
    else
      requant_rows<false>(o, v8, sbw, ma, sfw);
  }
  if constexpr (!kChannel) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t t = t0 + 16 * w + i;
      if (col_ok && t < T) __stcs(reinterpret_cast<uint2 *>(q + t * C + col), o[i]);
    }
  } else {
    // 4x4 byte transposes: cw[cc][rg] = column cc, rows 4rg..4rg+3 of this thread.
    uint32_t cw[8][4];
#pragma unroll
    for (int rg = 0; rg < 4; ++rg) {
#pragma unroll
      for (int cg = 0; cg < 2; ++cg) {
        const uint32_t r0 = cg ? o[4 * rg].y : o[4 * rg].x;
        const uint32_t r1 = cg ? o[4 * rg + 1].y : o[4 * rg + 1].x;
        const uint32_t r2 = cg ? o[4 * rg + 2].y : o[4 * rg + 2].x;
        const uint32_t r3 = cg ? o[4 * rg + 3].y : o[4 * rg + 3].x;
        const uint32_t u0 = __byte_perm(r0, r1, 0x5140);
        const uint32_t u1 = __byte_perm(r0, r1, 0x7362);
        const uint32_t u2 = __byte_perm(r2, r3, 0x5140);
        const uint32_t u3 = __byte_perm(r2, r3, 0x7362);
        cw[4 * cg + 0][rg] = __byte_perm(u0, u2, 0x5410);
        cw[4 * cg + 1][rg] = __byte_perm(u0, u2, 0x7632);
        cw[4 * cg + 2][rg] = __byte_perm(u1, u3, 0x5410);
        cw[4 * cg + 3][rg] = __byte_perm(u1, u3, 0x7632);
      }
    }
    // Tile row = channel (128 token bytes); 16-byte chunk k holds tokens 16k..16k+15
    // and sits at chunk position k ^ ((channel / 8) % 8).
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const int c = 8 * l + cc;
      *reinterpret_cast<uint4 *>(tq + c * kTileT + ((w ^ (l & 7)) << 4)) =
          make_uint4(cw[cc][0], cw[cc][1], cw[cc][2], cw[cc][3]);
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int id = threadIdx.x + 256 * it;
      const int c = id >> 3;
      const int k = id & 7;
      const int gc = c0 + c;
      const int64_t t = t0 + 16 * k;
      if (gc < C && t < T) {
        const uint4 val =
            *reinterpret_cast<const uint4 *>(tq + c * kTileT + ((k ^ ((c >> 3) & 7)) << 4));
        __stcs(reinterpret_cast<uint4 *>(q + static_cast<int64_t>(gc) * T + t), val);
      }
    }
  }
}

// Re-quantisation into the token-major layout (the TN GEMM's operand): one
// CTA covers 128 tokens x 512 channels, each thread 16 rows x 16 channels
// with 16-byte loads, so that two CTAs per SM keep as many bytes in flight as
// the BF16 cast does.  A thread's 16 channels lie in one 128-channel tile of
// the source scales.  After the maxima the codes wait in shared memory (64 KB)
// instead of registers, and the quantise pass streams them row by row.  Each
// block scale is computed once per column (not by every thread of its
// column group) into shared memory.
constexpr int kRqTileC = 512;
constexpr int kRqRed = 8 * kRqTileC * 4;                   // per-warp column maxima
constexpr int kRqScales = 4 * kRqTileC * 5;                // factors and bytes, up to 4 blocks
constexpr int kRqSmem = kTileT * kRqTileC + kRqRed + kRqScales + kTileT * 4;   // + source rows

template <int kGran, bool kGather>
__global__ void __launch_bounds__(256, 2) requant_tm_kernel(const CastArgs a) {
  extern __shared__ __align__(16) uint8_t rq_smem[];
  uint4 *tile = reinterpret_cast<uint4 *>(rq_smem);                         // [128][32] x 16 B
  uint4 (*red)[32][4] = reinterpret_cast<uint4 (*)[32][4]>(rq_smem + kTileT * kRqTileC);
  const float *red_f = reinterpret_cast<const float *>(rq_smem + kTileT * kRqTileC);   // [8][512]
  float *maS = reinterpret_cast<float *>(rq_smem + kTileT * kRqTileC + kRqRed);         // [blocks][512]
  uint8_t *sbS = rq_smem + kTileT * kRqTileC + kRqRed + 4 * kRqTileC * 4;               // [blocks][512]
  int *rows_s = reinterpret_cast<int *>(rq_smem + kTileT * kRqTileC + kRqRed + kRqScales);   // [128]
  const int w = threadIdx.x >> 5;
  const int l = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTileT;
  const int C = a.C;
  const int col = blockIdx.y * kRqTileC + 16 * l;
  const bool col_ok = col < C;
  const uint8_t *x = static_cast<const uint8_t *>(a.x);
  const int tiles = C / 128;
  stage_rows<kGather>(a, t0, rows_s);

  uint32_t sbw[4] = {0, 0, 0, 0};   // scale byte of row i in byte i % 4 of word i / 4
  float fm[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) fm[k] = 0.f;
  {
    uint4 v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t r = tile_source_row<kGather>(a, rows_s, t0, 16 * w + i, col_ok);
      v[i] = r >= 0 ? __ldcs(reinterpret_cast<const uint4 *>(x + r * C + col))
                    : make_uint4(0, 0, 0, 0);
      const uint32_t b = r >= 0 ? __ldg(a.x_sf + r * tiles + col / 128) : 0u;
      sbw[i >> 2] |= b << (8 * (i & 3));
    }
    // column maxima of |x| * 2^-8 (exact floats; rows not read hold code 0)
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float p = row_factor(sbw, i);
      const uint32_t wd[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float2 f = e4m3x2_to_f32(wd[h >> 1] >> (16 * (h & 1)));
        fm[2 * h] = fmaxf(fm[2 * h], fabsf(f.x * p));
        fm[2 * h + 1] = fmaxf(fm[2 * h + 1], fabsf(f.y * p));
      }
      tile[(16 * w + i) * 32 + l] = v[i];
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    red[w][l][j] = make_uint4(__float_as_uint(fm[4 * j]), __float_as_uint(fm[4 * j + 1]),
                              __float_as_uint(fm[4 * j + 2]), __float_as_uint(fm[4 * j + 3]));
  __syncthreads();

  // Block maxima (float bit patterns of non-negative values: integer maxima),
  // one (token block, column) per item: its factor 2^min(8 - e, 127) and its
  // scale byte e + 127.
  constexpr int kWarps = (kGran == 128) ? 8 : 2;
  constexpr int kBlocks = kTileT / kGran;
  constexpr int kItems = kBlocks * kRqTileC;
#pragma unroll
  for (int it = threadIdx.x; it < kItems; it += 256) {
    const int bb = it / kRqTileC, c = it % kRqTileC;
    uint32_t m = 0;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww)
      m = max(m, __float_as_uint(red_f[(bb * kWarps + ww) * kRqTileC + c]));
    const int e = scale_exp_from_f32_shifted(m);
    maS[it] = __uint_as_float(static_cast<uint32_t>(min(8 - e, 127) + 127) << 23);
    sbS[it] = static_cast<uint8_t>(e + 127);
  }
  __syncthreads();
  const int blk = (16 * w) / kGran;
  float ma[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 f = *reinterpret_cast<const float4 *>(maS + blk * kRqTileC + 16 * l + 4 * j);
    ma[4 * j] = f.x;
    ma[4 * j + 1] = f.y;
    ma[4 * j + 2] = f.z;
    ma[4 * j + 3] = f.w;
  }
  const uint4 sb4 = *reinterpret_cast<const uint4 *>(sbS + blk * kRqTileC + 16 * l);
  const uint32_t sfw[4] = {sb4.x, sb4.y, sb4.z, sb4.w};
  // a column whose factor 2^(8 - e) needs more than 2^127 (scale byte below 8)
  bool big = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) big |= ((sfw[j] - 0x08080808u) & ~sfw[j] & 0x80808080u) != 0;
  if (col_ok) {
    if constexpr (kGran == 128) {
      if (w == 0)
        *reinterpret_cast<uint4 *>(a.sf + (t0 / 128) * C + col) =
            make_uint4(sfw[0], sfw[1], sfw[2], sfw[3]);
    } else {
      const int64_t tb = t0 + 16 * w;
      if ((w & 1) == 0 && tb < a.T)
        *reinterpret_cast<uint4 *>(a.sf + (tb / 32) * C + col) =
            make_uint4(sfw[0], sfw[1], sfw[2], sfw[3]);
    }
  }

  // quantise and store, one row at a time from shared memory
  const float ma_lo[8] = {ma[0], ma[1], ma[2], ma[3], ma[4], ma[5], ma[6], ma[7]};
  const float ma_hi[8] = {ma[8], ma[9], ma[10], ma[11], ma[12], ma[13], ma[14], ma[15]};
  const uint32_t sf_lo[2] = {sfw[0], sfw[1]}, sf_hi[2] = {sfw[2], sfw[3]};
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const uint4 c = tile[(16 * w + i) * 32 + l];
    const float p = pow2_b_minus_135((sbw[i >> 2] >> (8 * (i & 3))) & 0xFFu);
    uint2 lo, hi;
    if (big) {
      lo = requant8<true>(make_uint2(c.x, c.y), p, ma_lo, sf_lo);
      hi = requant8<true>(make_uint2(c.z, c.w), p, ma_hi, sf_hi);
    } else {
      lo = requant8<false>(make_uint2(c.x, c.y), p, ma_lo, sf_lo);
      hi = requant8<false>(make_uint2(c.z, c.w), p, ma_hi, sf_hi);
    }
    const int64_t t = t0 + 16 * w + i;
    if (col_ok && t < a.T)
      __stcs(reinterpret_cast<uint4 *>(a.q + t * C + col), make_uint4(lo.x, lo.y, hi.x, hi.y));
  }
}

// BF16 rows gathered into the token-major MoE layout: one CTA covers 128
// output rows x 256 channels, staged whole in a 64 KB shared tile so that it
// is in flight at once without holding registers (three CTAs per SM: 220.5
// KB).  The rows of the first kGtTmaWarps warps come by TMA (lanes of warp 0
// issue gather4 loads of four indexed rows of 512 bytes each); every other
// warp copies its own rows with 16-byte cp.async through the load path, so
// that both of the SM's copy engines work on the tile (two warps of eight
// by TMA measured within 1 % of the fastest split).  Padding rows (-1) load
// row 0, which the passes below replace by zeros, so every gathered row is in
// bounds.
// Then the column-block cast as above, reading the tile twice (maxima, then
// quantise and store), one 16-byte row chunk at a time.
constexpr int kGtScales = 4 * kTileC * 5;   // factors and scale bytes of up to four token blocks
constexpr int kGtTmaWarps = 2;              // warps whose rows come by TMA (the rest by cp.async)

// 16-byte asynchronous copy global -> shared through the load path
// (src_bytes 0: 16 zero bytes), its commit, and the wait for all of them.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
constexpr int kGtSmem = kTileT * kTileC * 2 + kTileT * 4 + 8 * 32 * 16 + kGtScales + 16;

template <int kGran>
__global__ void __launch_bounds__(256, 3) gather_cast_kernel(const __grid_constant__ CastArgs a) {
  extern __shared__ __align__(1024) uint8_t gt_smem[];
  uint8_t *tile = gt_smem;                                                 // [128][512 B]
  int *idx = reinterpret_cast<int *>(gt_smem + kTileT * kTileC * 2);       // [128]
  uint4 *red = reinterpret_cast<uint4 *>(gt_smem + kTileT * kTileC * 2 + kTileT * 4);   // [8][32]
  float *mulS = reinterpret_cast<float *>(gt_smem + kTileT * kTileC * 2 + kTileT * 4 + 8 * 32 * 16);
  uint8_t *sbS = reinterpret_cast<uint8_t *>(mulS + 4 * kTileC);
  uint64_t *bar = reinterpret_cast<uint64_t *>(gt_smem + kTileT * kTileC * 2 + kTileT * 4 + 8 * 32 * 16 +
                                               kGtScales);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar + 1);
  const int tid = threadIdx.x;
  const int w = tid >> 5, l = tid & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTileT;
  const int C = a.C;
  const int c0 = blockIdx.y * kTileC;
  const int col = c0 + 8 * l;
  const bool col_ok = col < C;

  if (tid < kTileT) {
    const int64_t t = t0 + tid;
    int s = t < a.T ? __ldg(a.src_rows + t) : -1;
    if (s < -1 || s >= a.T_src) {
      atomicCAS(&a.status->code, DEV_OK, DEV_BAD_ROW);
      s = -1;
    }
    idx[tid] = s;
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // The rows of the first kGtTmaWarps warps come by TMA (lanes of warp 0
  // issue one gather4 of four rows each, all on the tile's barrier); every
  // other warp copies its own 16 rows through the load path (16 bytes per lane
  // and row, channels past C filled with zeros), so that both copy engines
  // of the SM bring the tile in.
  if (kGtTmaWarps > 0 && w == 0) {
    if (l == 0) mbar_arrive_expect_tx(bar, kGtTmaWarps * 16 * kTileC * 2);
    __syncwarp();
    if (l < kGtTmaWarps * 4)
      tma_gather4_2d(tile + l * 4 * kTileC * 2, &a.tmx, bar, c0, max(idx[4 * l], 0),
                     max(idx[4 * l + 1], 0), max(idx[4 * l + 2], 0), max(idx[4 * l + 3], 0));
  }
  if (w >= kGtTmaWarps) {
    const uint16_t *x = static_cast<const uint16_t *>(a.x);
    const bool in = col < C;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const int r = 16 * w + i;
      const uint16_t *src = x + static_cast<int64_t>(max(idx[r], 0)) * C + (in ? col : 0);
      cp_async16(tile + r * (kTileC * 2) + l * 16, src, in ? 16u : 0u);
    }
    cp_async_commit();
  }
  if (kGtTmaWarps > 0 &&
      !mbar_wait(bar, 0, abort_flag, a.wait_limit_ns, a.status, 0x41, blockIdx.x)) {
    // gave up: let the copies in flight land (bounded) before the CTA exits
    mbar_wait(bar, 0, abort_flag, drain_limit_ns(a.wait_limit_ns), a.status, 0x42, blockIdx.x,
              false);
    if (w >= kGtTmaWarps) cp_async_wait_all();
    return;
  }
  if (w >= kGtTmaWarps) {
    cp_async_wait_all();
    __syncwarp();   // every lane's rows are visible to the warp
  }

  // ---- pass 1: packed 16-bit maxima of |x| over this thread's 16 rows
  uint32_t m[4] = {0, 0, 0, 0};
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    uint4 v = *reinterpret_cast<const uint4 *>(tile + (16 * w + i) * (kTileC * 2) + l * 16);
    if (idx[16 * w + i] < 0) v = make_uint4(0, 0, 0, 0);
    m[0] = __vmaxu2(m[0], v.x & 0x7FFF7FFFu);
    m[1] = __vmaxu2(m[1], v.y & 0x7FFF7FFFu);
    m[2] = __vmaxu2(m[2], v.z & 0x7FFF7FFFu);
    m[3] = __vmaxu2(m[3], v.w & 0x7FFF7FFFu);
  }
  red[w * 32 + l] = make_uint4(m[0], m[1], m[2], m[3]);
  __syncthreads();
  // one scale per (token block, column), computed once: its factor 2^-e and
  // its byte e + 127 (red as [warp][column] 16-bit maxima)
  constexpr int kWarps = (kGran == 128) ? 8 : 2;
  constexpr int kItems = (kTileT / kGran) * kTileC;
  const uint16_t *red16 = reinterpret_cast<const uint16_t *>(red);
#pragma unroll
  for (int it = tid; it < kItems; it += 256) {
    const int bb = it / kTileC, c = it % kTileC;
    uint32_t mx = 0;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) mx = max(mx, static_cast<uint32_t>(red16[(bb * kWarps + ww) * kTileC + c]));
    const int e = scale_exp_from_bf16(mx);
    mulS[it] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    sbS[it] = static_cast<uint8_t>(e + 127);
  }
  __syncthreads();
  const int blk = (16 * w) / kGran;
  float mul[8];
  {
    const float4 f0 = *reinterpret_cast<const float4 *>(mulS + blk * kTileC + 8 * l);
    const float4 f1 = *reinterpret_cast<const float4 *>(mulS + blk * kTileC + 8 * l + 4);
    mul[0] = f0.x; mul[1] = f0.y; mul[2] = f0.z; mul[3] = f0.w;
    mul[4] = f1.x; mul[5] = f1.y; mul[6] = f1.z; mul[7] = f1.w;
  }
  const uint2 sb2 = *reinterpret_cast<const uint2 *>(sbS + blk * kTileC + 8 * l);
  const uint32_t sfw[2] = {sb2.x, sb2.y};
  if (col_ok) {
    if constexpr (kGran == 128) {
      if (w == 0)
        *reinterpret_cast<uint2 *>(a.sf + (t0 / 128) * C + col) = make_uint2(sfw[0], sfw[1]);
    } else {
      const int64_t tb = t0 + 16 * w;
      if ((w & 1) == 0 && tb < a.T)
        *reinterpret_cast<uint2 *>(a.sf + (tb / 32) * C + col) = make_uint2(sfw[0], sfw[1]);
    }
  }

  // ---- pass 2: quantise and store (rows past T are not written)
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int64_t t = t0 + 16 * w + i;
    uint4 v = *reinterpret_cast<const uint4 *>(tile + (16 * w + i) * (kTileC * 2) + l * 16);
    if (idx[16 * w + i] < 0) v = make_uint4(0, 0, 0, 0);
    const uint2 o =
        make_uint2(quant_word(v.x, mul[0], mul[1]) | (quant_word(v.y, mul[2], mul[3]) << 16),
                   quant_word(v.z, mul[4], mul[5]) | (quant_word(v.w, mul[6], mul[7]) << 16));
    if (col_ok && t < a.T) __stcs(reinterpret_cast<uint2 *>(a.q + t * C + col), o);
  }
}

template <int kGran>
cudaError_t launch_gather_tma(const CastArgs &a, cudaStream_t stream) {
  // attributes set once per process (thread-safe static initialisation)
  static const cudaError_t setup = [] {
    cudaError_t e = cudaFuncSetAttribute(gather_cast_kernel<kGran>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kGtSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gather_cast_kernel<kGran>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    return e;
  }();
  if (setup != cudaSuccess) return setup;
  const dim3 grid(static_cast<unsigned>((a.T + kTileT - 1) / kTileT),
                  static_cast<unsigned>((a.C + kTileC - 1) / kTileC));
  gather_cast_kernel<kGran><<<grid, 256, kGtSmem, stream>>>(a);
  return cudaGetLastError();
}

template <bool kFp8Src, bool kGather>
cudaError_t launch_src(const CastArgs &a, int channel_major, int gran_k, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((a.T + kTileT - 1) / kTileT),
                  static_cast<unsigned>((a.C + kTileC - 1) / kTileC));
  if (gran_k == 128) {
    if (channel_major)
      cast_colblock_kernel<128, true, kFp8Src, kGather><<<grid, 256, 0, stream>>>(a);
    else
      cast_colblock_kernel<128, false, kFp8Src, kGather><<<grid, 256, 0, stream>>>(a);
  } else {
    if (channel_major)
      cast_colblock_kernel<32, true, kFp8Src, kGather><<<grid, 256, 0, stream>>>(a);
    else
      cast_colblock_kernel<32, false, kFp8Src, kGather><<<grid, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

template <bool kGather>
cudaError_t launch_requant_tm(const CastArgs &a, int gran_k, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((a.T + kTileT - 1) / kTileT),
                  static_cast<unsigned>((a.C + kRqTileC - 1) / kRqTileC));
  static const cudaError_t setup = [] {
    cudaError_t e = cudaFuncSetAttribute(requant_tm_kernel<128, kGather>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kRqSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(requant_tm_kernel<32, kGather>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kRqSmem);
    return e;
  }();
  if (setup != cudaSuccess) return setup;
  if (gran_k == 128)
    requant_tm_kernel<128, kGather><<<grid, 256, kRqSmem, stream>>>(a);
  else
    requant_tm_kernel<32, kGather><<<grid, 256, kRqSmem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cast_colblock(const CastArgs &a, int channel_major, int gran_k,
                                 cudaStream_t stream) {
  const bool fp8 = (a.x_sf != nullptr);
  const bool gather = (a.src_rows != nullptr);
  if (a.use_tmx)
    return gran_k == 128 ? launch_gather_tma<128>(a, stream) : launch_gather_tma<32>(a, stream);
  if (fp8 && !channel_major)
    return gather ? launch_requant_tm<true>(a, gran_k, stream)
                  : launch_requant_tm<false>(a, gran_k, stream);
  if (fp8)
    return gather ? launch_src<true, true>(a, channel_major, gran_k, stream)
                  : launch_src<true, false>(a, channel_major, gran_k, stream);
  return gather ? launch_src<false, true>(a, channel_major, gran_k, stream)
                : launch_src<false, false>(a, channel_major, gran_k, stream);
}

}  // namespace dg
