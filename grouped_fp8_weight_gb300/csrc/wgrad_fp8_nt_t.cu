// FP8 instantiations of the K-grouped kernel with transposed output tiles on
// K-major (NT) operands.
#include "wgrad_kernel.cuh"

namespace dg {

cudaError_t launch_kgrouped_fp8_nt_t(const WgradParams &p, int block_n, int pairs,
                                     cudaStream_t stream) {
  if (block_n != 224) return cudaErrorInvalidValue;
  return launch_wgrad_bn<true, 224, true, true>(p, pairs, stream);
}

}  // namespace dg
