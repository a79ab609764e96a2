// Column-block FP8 cast (with optional physical transpose) for sm_103a.
//
// For every gran_k-token block and column of a BF16 matrix x[T, C]:
//   amax = max |x|, e = clamp(ceil(log2(amax / 448)), -127, 127),
//   sf = e + 127 (UE8M0), q = E4M3 round-to-nearest-even of x * 2^-e.
//
// HBM-bound: 2 bytes read and 1 (+1/gran_k) written per element.  One CTA
// covers 128 tokens x 256 channels (64 KiB of input).  Each thread loads 16
// rows x 16 bytes with independent vector loads, reduces |x| with packed
// 16-bit maxima on the BF16 bit patterns (exact: non-negative floats order like
// their bit patterns), combines the eight warps' partial maxima in shared
// memory, and converts with the hardware's saturating RNE E4M3 conversion.
// The channel-major variant transposes 4x4 byte blocks in registers and
// stages the tile in a swizzled shared-memory buffer so that both the shared
// stores and the 128-byte global row stores are conflict-free and coalesced.
#include <cstdint>
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

// Two floats -> two E4M3 bytes (lo in the low byte), RNE, saturating.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return static_cast<uint32_t>(r);
}

__device__ __forceinline__ uint32_t quant_word(uint32_t w, float m_lo, float m_hi) {
  const float lo = __uint_as_float(w << 16) * m_lo;
  const float hi = __uint_as_float(w & 0xFFFF0000u) * m_hi;
  return cvt_e4m3x2(lo, hi);
}

template <int kGran, bool kChannel>
__global__ void __launch_bounds__(256, 2)
    quant_colblock_kernel(const uint16_t *__restrict__ x, int64_t T, int C,
                          uint8_t *__restrict__ q, uint8_t *__restrict__ sf) {
  __shared__ uint4 red[8][32];
  __shared__ __align__(16) uint8_t tq[kChannel ? kTileC * kTileT : 16];
  const int w = threadIdx.x >> 5;
  const int l = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTileT;
  const int c0 = blockIdx.y * kTileC;
  const int col = c0 + 8 * l;
  const bool col_ok = col < C;

  uint4 v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int64_t t = t0 + 16 * w + i;
    if (col_ok && t < T)
      v[i] = __ldcs(reinterpret_cast<const uint4 *>(x + t * C + col));
    else
      v[i] = make_uint4(0, 0, 0, 0);
  }
  uint32_t m[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    m[0] = __vmaxu2(m[0], v[i].x & 0x7FFF7FFFu);
    m[1] = __vmaxu2(m[1], v[i].y & 0x7FFF7FFFu);
    m[2] = __vmaxu2(m[2], v[i].z & 0x7FFF7FFFu);
    m[3] = __vmaxu2(m[3], v[i].w & 0x7FFF7FFFu);
  }
  red[w][l] = make_uint4(m[0], m[1], m[2], m[3]);
  __syncthreads();
  uint4 a;
  if constexpr (kGran == 128) {
    a = red[0][l];
#pragma unroll
    for (int ww = 1; ww < 8; ++ww) {
      const uint4 r = red[ww][l];
      a.x = __vmaxu2(a.x, r.x);
      a.y = __vmaxu2(a.y, r.y);
      a.z = __vmaxu2(a.z, r.z);
      a.w = __vmaxu2(a.w, r.w);
    }
  } else {
    const uint4 r0 = red[w & ~1][l], r1 = red[w | 1][l];
    a = make_uint4(__vmaxu2(r0.x, r1.x), __vmaxu2(r0.y, r1.y), __vmaxu2(r0.z, r1.z),
                   __vmaxu2(r0.w, r1.w));
  }
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
  float mul[8];
  uint32_t sfw[2] = {0, 0};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = scale_exp_from_bf16((aw[k] >> (16 * h)) & 0xFFFFu);
      mul[2 * k + h] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
      sfw[k >> 1] |= static_cast<uint32_t>(e + 127) << (8 * (2 * (k & 1) + h));
    }
  }
  if (col_ok) {
    if constexpr (kGran == 128) {
      if (w == 0)
        *reinterpret_cast<uint2 *>(sf + (t0 / 128) * C + col) = make_uint2(sfw[0], sfw[1]);
    } else {
      const int64_t tb = t0 + 16 * w;
      if ((w & 1) == 0 && tb < T)
        *reinterpret_cast<uint2 *>(sf + (tb / 32) * C + col) = make_uint2(sfw[0], sfw[1]);
    }
  }

  uint2 o[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    o[i].x = quant_word(v[i].x, mul[0], mul[1]) | (quant_word(v[i].y, mul[2], mul[3]) << 16);
    o[i].y = quant_word(v[i].z, mul[4], mul[5]) | (quant_word(v[i].w, mul[6], mul[7]) << 16);
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

}  // namespace

cudaError_t launch_quant_colblock(const void *x, int64_t T, int C, void *q, uint8_t *sf,
                                  int channel_major, int gran_k, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((T + kTileT - 1) / kTileT),
                  static_cast<unsigned>((C + kTileC - 1) / kTileC));
  const auto *xp = static_cast<const uint16_t *>(x);
  auto *qp = static_cast<uint8_t *>(q);
  if (gran_k == 128) {
    if (channel_major)
      quant_colblock_kernel<128, true><<<grid, 256, 0, stream>>>(xp, T, C, qp, sf);
    else
      quant_colblock_kernel<128, false><<<grid, 256, 0, stream>>>(xp, T, C, qp, sf);
  } else {
    if (channel_major)
      quant_colblock_kernel<32, true><<<grid, 256, 0, stream>>>(xp, T, C, qp, sf);
    else
      quant_colblock_kernel<32, false><<<grid, 256, 0, stream>>>(xp, T, C, qp, sf);
  }
  return cudaGetLastError();
}

}  // namespace dg
