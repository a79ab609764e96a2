// BF16-input instantiations of the K-grouped kernel.
#include "wgrad_kernel.cuh"

namespace dg {

int bf16_pick_block_n(int N) { return N >= 256 ? 256 : 128; }

cudaError_t launch_kgrouped_bf16(const WgradParams &p, int block_n, int pairs,
                                 cudaStream_t stream) {
  switch (block_n) {
    case 256: return launch_wgrad_bn<false, 256>(p, pairs, stream);
    case 128: return launch_wgrad_bn<false, 128>(p, pairs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg
