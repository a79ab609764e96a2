// FP8 instantiations of the persistent GEMM kernel in its M-grouped mode:
// the data gradient dx_e = dy_e W_e of a MoE expert, dy's token rows of every
// expert contiguous ([sum_m, K], K contiguous), W [G, K, N] (N contiguous).
#include "wgrad_kernel.cuh"

namespace dg {

cudaError_t launch_mgrouped_fp8(const WgradParams &p, int block_n, int pairs,
                                cudaStream_t stream) {
  switch (block_n) {
    case 224: return launch_mgrouped_bn<224>(p, pairs, stream);
    case 128: return launch_mgrouped_bn<128>(p, pairs, stream);
  }
  return cudaErrorInvalidValue;
}

// The same with the weights stored K-major, W [G, N, K] (tmB maps them as {K, G * N}).
cudaError_t launch_mgrouped_fp8_nt(const WgradParams &p, int block_n, int pairs,
                                   cudaStream_t stream) {
  switch (block_n) {
    case 224: return launch_mgrouped_bn<224, true>(p, pairs, stream);
    case 128: return launch_mgrouped_bn<128, true>(p, pairs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg
