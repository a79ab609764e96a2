// FP8 instantiations of the K-grouped kernel with transposed output tiles on
// K-major (NT) operands.
#include "wgrad_kernel.cuh"

namespace dg {

cudaError_t launch_kgrouped_fp8_nt_t(const WgradParams &p, int block_n, int pairs,
                                     cudaStream_t stream) {
  switch (block_n) {
    case 256: return launch_wgrad_bn<true, 256, true, true>(p, pairs, stream);
    case 224: return launch_wgrad_bn<true, 224, true, true>(p, pairs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg
