// FP8 instantiations of the K-grouped kernel for K-major (NT) operands:
// A [M, sum_k] and B [N, sum_k], token axis contiguous.
#include "wgrad_kernel.cuh"

namespace dg {

cudaError_t launch_kgrouped_fp8_nt(const WgradParams &p, int block_n, int pairs,
                                   cudaStream_t stream) {
  switch (block_n) {
    case 256: return launch_wgrad_bn<true, 256, true>(p, pairs, stream);
    case 224: return launch_wgrad_bn<true, 224, true>(p, pairs, stream);
    case 128: return launch_wgrad_bn<true, 128, true>(p, pairs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg
