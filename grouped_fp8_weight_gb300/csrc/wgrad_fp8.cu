// FP8 (E4M3, UE8M0 block-scaled) instantiations of the K-grouped kernel.
#include "wgrad_kernel.cuh"

namespace dg {

// 224 columns keep two FP32 accumulators plus the scale buffers inside the
// 512 tensor-memory columns; other widths fall back to 128.  (Block 256, the
// mixed 256 / 224 variant, is chosen by the schedule on top of 224.)
int fp8_pick_block_n(int N) { return (N % 224 == 0) ? 224 : 128; }

cudaError_t launch_kgrouped_fp8(const WgradParams &p, int block_n, int pairs,
                                cudaStream_t stream) {
  switch (block_n) {
    case 256: return launch_wgrad_bn<true, 256>(p, pairs, stream);
    case 224: return launch_wgrad_bn<true, 224>(p, pairs, stream);
    case 128: return launch_wgrad_bn<true, 128>(p, pairs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg
