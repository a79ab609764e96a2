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
// It runs the same validation, schedule (longest experts first, transposed
// tiles where N is not a multiple of 224 but M is, the split of long experts
// along K for in-place accumulation) and kernels as dg_k_grouped_fp8_wgrad
// (grouped_plan.h); only the place of the status record and of the packed
// scale records differs.
//
// Scratch: kScratchBytes = 256 bytes for the 16-byte status record plus
// kScaleBytes (32 MiB) for the packed scale records, whose size is
// (scale groups) x (2 * ceil(M / 256) + ceil(N / BN) * ceil(BN / 128)) x 512
// bytes, with one scale group per four k-blocks of each schedule entry
// (gran_k 128) or per k-block (gran_k 32, about four times as many bytes);
// larger problems are rejected with DG_ERR_UNSUPPORTED.  Every GPU that loads
// this part of the library holds the array until the process exits.  All
// calls on a device share it: each call clears the record and rewrites the
// scale records on its stream before the GEMM, and calls that overlap on the
// GPU (different streams) race on it.  This entry point never synchronises; a
// device-side wait that runs out (the kernel then ends early and leaves D
// unspecified) or a ks_dev mismatch stays in the record until the next call
// clears it, and dg_sync_check reads and clears it (noalloc_take_status).
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "dg_wgrad.h"
#include "grouped_plan.h"
#include "wgrad_params.h"

namespace {

constexpr size_t kStatusBytes = 256;
constexpr size_t kScaleBytes = size_t(32) << 20;
constexpr size_t kScratchBytes = kStatusBytes + kScaleBytes;
static_assert(sizeof(dg::DevStatus) <= kStatusBytes, "status record must fit the scratch");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

thread_local dg::WgradParams t_params;   // reused per thread: no per-call heap allocation
thread_local dg::PackParams t_pack;

struct NoAllocDevice {
  bool ready = false;
  int sms = 0;
  dg::DevStatus *scratch = nullptr;   // device address of g_noalloc_scratch
  unsigned char *scales = nullptr;    // the packed scale records, kStatusBytes in
};

constexpr int kMaxDev = 64;
std::mutex n_mu;
NoAllocDevice n_dev[kMaxDev];

// Once per device, with that device current: query it and resolve the scratch
// array's device address.  No allocation.
dg_status setup(NoAllocDevice **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return dg::failf(DG_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDev) return dg::failf(DG_ERR_UNSUPPORTED, "device index %d", dev);
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
      return dg::failf(DG_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    if (major != 10 || minor != 3)
      return dg::failf(DG_ERR_UNSUPPORTED, "device is sm_%d%d; built for sm_103a only", major,
                       minor);
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return dg::failf(DG_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    if (dg::tensor_map_encoder() == nullptr)
      return dg::failf(DG_ERR_CUDA, "cuTensorMapEncodeTiled not available");
    st.scratch = static_cast<dg::DevStatus *>(ptr);
    st.scales = static_cast<unsigned char *>(ptr) + kStatusBytes;
    st.ready = true;
  }
  *out = &st;
  return DG_OK;
}

}  // namespace

namespace dg {
// For dg_sync_check: reads and clears this device's record of the
// allocation-free entry point (after the caller has synchronised), if that
// entry point has run on the device.  No allocation.
cudaError_t noalloc_take_status(DevStatus *out, bool *present) {
  *present = false;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaSuccess;
  dg::DevStatus *rec = nullptr;
  {
    std::lock_guard<std::mutex> lock(n_mu);
    if (n_dev[dev].ready) rec = n_dev[dev].scratch;
  }
  if (rec == nullptr) return cudaSuccess;
  if ((e = cudaMemcpy(out, rec, sizeof(*out), cudaMemcpyDeviceToHost)) != cudaSuccess) return e;
  *present = true;
  if (out->code != DEV_OK) e = cudaMemset(rec, 0, sizeof(*out));
  return e;
}
}  // namespace dg

extern "C" dg_status dg_k_grouped_fp8_wgrad_noalloc(
    const void *a, const uint8_t *sfa, const void *b, const uint8_t *sfb, void *d,
    dg_dtype d_dtype, const float *c, int G, int M, int N, int64_t sum_k, const int *ks_host,
    const int *ks_dev, int gran_k, dg_stream_t stream) {
  const char *fn = "dg_k_grouped_fp8_wgrad_noalloc";
  dg::GroupedArgs x{fn, true, false, a, b, sfa, sfb, d, d_dtype, c, G, M, N, sum_k,
                    ks_host, ks_dev, gran_k, reinterpret_cast<cudaStream_t>(stream)};
  dg_status s = dg::grouped_validate(x);
  if (s != DG_OK) return s;
  if (G == 0) {
    dg::set_last_error("");
    return DG_OK;
  }
  dg::WgradParams &p = t_params;
  dg::PackParams &pk = t_pack;
  dg::GroupedPlan g{};
  // The schedule without the split of long in-place experts needs no device:
  // a problem whose packed scale records cannot fit even so is rejected
  // before any CUDA call.  (The split adds at most a few groups.)
  dg::grouped_schedule(x, 0, p, pk, g);
  if (g.sf_bytes > kScaleBytes)
    return dg::failf(DG_ERR_UNSUPPORTED,
                     "%s: the packed scale factors need %zu bytes, above this entry point's "
                     "maximum of %zu",
                     fn, g.sf_bytes, kScaleBytes);
  NoAllocDevice *dev = nullptr;
  if ((s = setup(&dev)) != DG_OK) return s;
  // The same schedule as the ordinary entry point (split of long in-place
  // experts included), now that the SM count is known.
  dg::grouped_schedule(x, dev->sms, p, pk, g);
  if (g.sf_bytes > kScaleBytes)
    return dg::failf(DG_ERR_UNSUPPORTED,
                     "%s: the packed scale factors need %zu bytes, above this entry point's "
                     "maximum of %zu",
                     fn, g.sf_bytes, kScaleBytes);
  p.status = dev->scratch;
  p.wait_limit_ns = dg::wait_limit_ns();
  if (p.num_tiles == 0) {
    dg::set_last_error("");
    return DG_OK;
  }
  if ((s = dg::grouped_maps(x, g, p)) != DG_OK) return s;
  if (g.sf_bytes > 0 && (s = dg::grouped_scale_maps(x, g, dev->scales, p, pk)) != DG_OK) return s;
  cudaStream_t st = x.stream;
  cudaError_t e = cudaMemsetAsync(dev->scratch, 0, sizeof(dg::DevStatus), st);
  if (e != cudaSuccess)
    return dg::failf(DG_ERR_CUDA, "%s: clearing scratch: %s", fn, cudaGetErrorString(e));
  if (g.sf_bytes > 0 && (e = dg::launch_pack_scales(pk, st)) != cudaSuccess)
    return dg::failf(DG_ERR_CUDA, "%s: scale pack launch failed: %s", fn, cudaGetErrorString(e));
  p.pdl = (g.sf_bytes > 0 && dg::pdl_requested()) ? 1 : 0;
  if ((e = dg::grouped_launch(x, g, p, dev->sms)) != cudaSuccess)
    return dg::failf(DG_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  dg::set_last_error("");
  return DG_OK;
}
