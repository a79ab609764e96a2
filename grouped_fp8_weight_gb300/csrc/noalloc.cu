// dg_k_grouped_fp8_wgrad_noalloc: the FP8 K-grouped weight gradient for
// callers that cannot allocate device memory.
//
// The ordinary entry point allocates one small status record per device with
// cudaMalloc on its first call (the kernel writes timeouts and ks_dev
// mismatches there) and takes scratch for the packed scale factors from a
// memory pool on every call.  Some callers cannot let a library do that: a
// framework whose caching allocator has already reserved the device memory it
// is allowed to use, or a thread that must not take the implicit device
// synchronisation a cudaMalloc can cause.  This variant runs the same kernels
// with both placed in a file-scope __device__ array instead, so it allocates
// nothing.
//
// Scratch: kScratchBytes = 256 bytes for the 16-byte status record plus
// kScaleBytes (32 MiB) for the packed scale records, whose size is
// (scale groups) x (2 * ceil(M / 256) + ceil(N / BN) * ceil(BN / 128)) x 512
// bytes, with one scale group per four k-blocks of each expert (gran_k 128) or
// per k-block (gran_k 32); larger problems are rejected with
// DG_ERR_UNSUPPORTED.  Every GPU that loads this part of the library holds the
// array until the process exits.  All calls on a device share it: each call
// clears the record and rewrites the scale records on its stream before the
// GEMM, and calls that overlap on the GPU (different streams) race on it.  This entry point never
// synchronises, so it does not report what the kernel records there; the
// kernel's waits are still bounded, so a wait that runs out ends the kernel
// early and leaves D unspecified.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "dg_wgrad.h"
#include "wgrad_params.h"

namespace dg {
void set_last_error(const char *msg);   // api.cu
}

namespace {

constexpr size_t kStatusBytes = 256;
constexpr size_t kScaleBytes = size_t(32) << 20;
constexpr size_t kScratchBytes = kStatusBytes + kScaleBytes;
static_assert(sizeof(dg::DevStatus) <= kStatusBytes, "status record must fit the scratch");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

thread_local dg::WgradParams t_params;   // reused per thread: no per-call heap allocation
thread_local dg::PackParams t_pack;

dg_status nfail(dg_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  dg::set_last_error(buf);
  return s;
}

struct NoAllocDevice {
  bool ready = false;
  int sms = 0;
  dg::DevStatus *scratch = nullptr;   // device address of g_noalloc_scratch
  unsigned char *scales = nullptr;    // the packed scale records, kStatusBytes in
};

constexpr int kMaxDev = 64;
std::mutex n_mu;
NoAllocDevice n_dev[kMaxDev];
PFN_cuTensorMapEncodeTiled_v12000 n_encode = nullptr;

// Once per device, with that device current: query it, resolve the scratch
// array's device address and the tensor-map encoder.  No allocation.
dg_status setup(NoAllocDevice **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return nfail(DG_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDev) return nfail(DG_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(n_mu);
  NoAllocDevice &st = n_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev)) !=
            cudaSuccess)
      return nfail(DG_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    if (major != 10 || minor != 3)
      return nfail(DG_ERR_UNSUPPORTED, "device is sm_%d%d; built for sm_103a only", major, minor);
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return nfail(DG_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    st.scratch = static_cast<dg::DevStatus *>(ptr);
    st.scales = static_cast<unsigned char *>(ptr) + kStatusBytes;
    if (n_encode == nullptr) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q{};
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q);
      if (e != cudaSuccess || fn == nullptr || q != cudaDriverEntryPointSuccess)
        return nfail(DG_ERR_CUDA, "cuTensorMapEncodeTiled not available");
      n_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    st.ready = true;
  }
  *out = &st;
  return DG_OK;
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dg_status map2d(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t inner,
                uint64_t outer, uint64_t row_bytes, uint32_t b0, uint32_t b1,
                CUtensorMapSwizzle sw, CUtensorMapL2promotion l2, const char *what) {
  const cuuint64_t dims[2] = {inner, outer}, strides[1] = {row_bytes};
  const cuuint32_t box[2] = {b0, b1}, es[2] = {1, 1};
  CUresult r = n_encode(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return nfail(DG_ERR_CUDA, "tensor map for %s failed (%d)", what, (int)r);
  return DG_OK;
}

dg_status map_out(CUtensorMap *m, bool bf16, const void *ptr, uint64_t M, uint64_t N,
                  uint64_t G, const char *what) {
  const uint64_t es = bf16 ? 2 : 4;
  const cuuint64_t dims[3] = {N, M, G}, strides[2] = {es * N, es * N * M};
  const cuuint32_t box[3] = {dg::kEpiCols, 32, 1}, ones[3] = {1, 1, 1};
  CUresult r = n_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                        3, const_cast<void *>(ptr), dims, strides, box, ones,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, dg::epi_swizzle(bf16 ? 2 : 4),
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return nfail(DG_ERR_CUDA, "tensor map for %s failed (%d)", what, (int)r);
  return DG_OK;
}

}  // namespace

extern "C" dg_status dg_k_grouped_fp8_wgrad_noalloc(
    const void *a, const uint8_t *sfa, const void *b, const uint8_t *sfb, void *d,
    dg_dtype d_dtype, const float *c, int G, int M, int N, int64_t sum_k, const int *ks_host,
    const int *ks_dev, int gran_k, dg_stream_t stream) {
  const char *fn = "dg_k_grouped_fp8_wgrad_noalloc";
  // The status record needs the same 16 bytes for every problem; the sizes
  // below are the limits of the kernel's schedule, as in the ordinary call.
  if (G < 0) return nfail(DG_ERR_INVALID_ARG, "%s: G = %d < 0", fn, G);
  if (G > DG_MAX_GROUPS)
    return nfail(DG_ERR_UNSUPPORTED, "%s: G = %d above the maximum of %d experts", fn, G,
                 DG_MAX_GROUPS);
  if (M <= 0 || N <= 0 || M % 16 || N % 16)
    return nfail(DG_ERR_INVALID_ARG, "%s: M = %d, N = %d must be positive multiples of 16", fn,
                 M, N);
  if (sum_k < 0) return nfail(DG_ERR_INVALID_ARG, "%s: sum_k < 0", fn);
  if (sum_k > (int64_t)0x7FFFFF00)
    return nfail(DG_ERR_UNSUPPORTED, "%s: sum_k above the maximum of 2^31 - 256", fn);
  if (gran_k != 32 && gran_k != 128)
    return nfail(DG_ERR_INVALID_ARG, "%s: gran_k = %d (must be 32 or 128)", fn, gran_k);
  if (d_dtype != DG_F32 && d_dtype != DG_BF16)
    return nfail(DG_ERR_INVALID_ARG, "%s: unknown output dtype %d", fn, (int)d_dtype);
  if (d_dtype == DG_BF16 && c != nullptr)
    return nfail(DG_ERR_INVALID_ARG, "%s: an accumulator needs FP32 output", fn);
  if (G == 0) {
    if (sum_k != 0) return nfail(DG_ERR_INVALID_ARG, "%s: G = 0 but sum_k != 0", fn);
    dg::set_last_error("");
    return DG_OK;
  }
  if (ks_host == nullptr || ks_dev == nullptr)
    return nfail(DG_ERR_INVALID_ARG, "%s: ks_host and ks_dev are required", fn);
  int64_t total = 0;
  for (int e = 0; e < G; ++e) {
    if (ks_host[e] < 0 || ks_host[e] % 128)
      return nfail(DG_ERR_INVALID_ARG, "%s: ks[%d] = %d must be a non-negative multiple of 128",
                   fn, e, ks_host[e]);
    total += ks_host[e];
  }
  if (total != sum_k)
    return nfail(DG_ERR_INVALID_ARG, "%s: sum of ks (%lld) != sum_k (%lld)", fn,
                 (long long)total, (long long)sum_k);
  if (d == nullptr || !al16(d) || (c != nullptr && c != d && !al16(c)))
    return nfail(DG_ERR_INVALID_ARG, "%s: d and c must be 16-byte aligned device pointers", fn);
  if (sum_k > 0 && (a == nullptr || b == nullptr || sfa == nullptr || sfb == nullptr ||
                    !al16(a) || !al16(b) || !al16(sfa) || !al16(sfb)))
    return nfail(DG_ERR_INVALID_ARG, "%s: a, b, sfa, sfb must be 16-byte aligned device pointers",
                 fn);
  // The schedule and the size check need no device: an over-size problem is
  // rejected before any CUDA call.
  dg::WgradParams &p = t_params;
  std::memset(&p, 0, sizeof(p));
  // Longest experts first; then experts that only need their output written.
  int n = 0;
  int64_t off = 0;
  int order_len = 0;
  static thread_local int order[DG_MAX_GROUPS];
  static thread_local int64_t offs[DG_MAX_GROUPS];
  for (int e = 0; e < G; ++e) {
    offs[e] = off;
    off += ks_host[e];
    if (ks_host[e] > 0) order[order_len++] = e;
  }
  std::stable_sort(order, order + order_len, [&](int u, int v) { return ks_host[u] > ks_host[v]; });
  const int n_mma = order_len;
  if (c != d)
    for (int e = 0; e < G; ++e)
      if (ks_host[e] == 0) order[order_len++] = e;
  for (n = 0; n < order_len; ++n) {
    p.sched[n].expert = order[n];
    p.sched[n].k_off = static_cast<int>(offs[order[n]]);
    p.sched[n].k_len = ks_host[order[n]];
    p.sched[n].k_exp = ks_host[order[n]];
  }
  const int bn = dg::fp8_pick_block_n(N);
  p.M = M;
  p.N = N;
  p.G = G;
  p.m_tiles = (M + dg::kPairM - 1) / dg::kPairM;
  p.n_tiles = (N + bn - 1) / bn;
  p.tiles_per_group = p.m_tiles * p.n_tiles;
  p.num_mma_tiles = n_mma * p.tiles_per_group;
  p.num_tiles = order_len * p.tiles_per_group;
  p.gran_k = gran_k;
  p.chunk = dg::kFp8Chunk;
  p.m_fastest = (M <= N) ? 1 : 0;
  p.out_mode = (d_dtype == DG_BF16) ? dg::OUT_BF16
               : (c == nullptr)     ? dg::OUT_F32
               : (c == d)           ? dg::OUT_F32_REDUCE
                                    : dg::OUT_F32_C;
  long ms = 4000;
  if (const char *env = std::getenv("DG_WAIT_LIMIT_MS")) {
    char *end = nullptr;
    const long v = std::strtol(env, &end, 10);
    if (end != env && v > 0) ms = v;
  }
  p.wait_limit_ns = static_cast<uint64_t>(ms) * 1000000ull;
  p.ks_dev = ks_dev;
  dg::PackParams &pk = t_pack;
  std::memset(&pk, 0, sizeof(pk));
  const size_t sf_bytes = (n_mma > 0) ? dg::plan_scale_pack(p, pk, n_mma, gran_k, bn) : 0;
  if (sf_bytes > kScaleBytes)
    return nfail(DG_ERR_UNSUPPORTED,
                 "%s: the packed scale factors need %zu bytes, above this entry point's %zu",
                 fn, sf_bytes, kScaleBytes);
  NoAllocDevice *dev = nullptr;
  dg_status s = setup(&dev);
  if (s != DG_OK) return s;
  p.status = dev->scratch;
  if (p.num_tiles == 0) {
    dg::set_last_error("");
    return DG_OK;
  }
  const uint64_t SK = sum_k;
  if (p.num_mma_tiles > 0) {
    dg::bind_scale_pack(pk, dev->scales, sfa, sfb);
    const uint64_t groups = static_cast<uint64_t>(pk.n_groups);
    if ((s = map2d(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, M, SK, M, 128, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "a")) ||
        (s = map2d(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, N, SK, N,
                   static_cast<uint32_t>(std::min(128, bn / 2)), 128,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "b")) ||
        (s = map2d(&p.tmSFA, CU_TENSOR_MAP_DATA_TYPE_UINT32, pk.sfa_p, 128, groups * pk.MC, 512,
                   128, 1, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   "sfa records")) ||
        (s = map2d(&p.tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT32, pk.sfb_p, 128,
                   groups * pk.NT * pk.CB, 512, 128, static_cast<uint32_t>(pk.CB),
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, "sfb records")))
      return s;
  }
  if ((s = map_out(&p.tmD, d_dtype == DG_BF16, d, M, N, G, "d"))) return s;
  if (p.out_mode == dg::OUT_F32_C && (s = map_out(&p.tmC, false, c, M, N, G, "c"))) return s;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(dev->scratch, 0, sizeof(dg::DevStatus), st);
  if (e != cudaSuccess) return nfail(DG_ERR_CUDA, "%s: clearing scratch: %s", fn, cudaGetErrorString(e));
  if (sf_bytes > 0 && (e = dg::launch_pack_scales(pk, st)) != cudaSuccess)
    return nfail(DG_ERR_CUDA, "%s: scale pack launch failed: %s", fn, cudaGetErrorString(e));
  dg::set_derived(p, order_len);
  e = dg::launch_kgrouped_fp8(p, bn, std::min(dev->sms / 2, p.num_tiles), st);
  if (e != cudaSuccess) return nfail(DG_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  dg::set_last_error("");
  return DG_OK;
}
