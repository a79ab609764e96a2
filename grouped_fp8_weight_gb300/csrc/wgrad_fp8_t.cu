// FP8 instantiations of the K-grouped kernel with transposed output tiles
// (the kernel computes D^T = B^T A in 256 x 224 tiles, or mixed 256 x 256 /
// 256 x 224 ones, and writes them into D transposed): token-major operands.
#include "wgrad_kernel.cuh"

namespace dg {

cudaError_t launch_kgrouped_fp8_t(const WgradParams &p, int block_n, int pairs,
                                  cudaStream_t stream) {
  switch (block_n) {
    case 256: return launch_wgrad_bn<true, 256, false, true>(p, pairs, stream);
    case 224: return launch_wgrad_bn<true, 224, false, true>(p, pairs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg
