// vq_decode_balanced.cu -- the split attention kernel (vq_decode_kernel.cuh)
// with length-balanced units: the (sequence, KV head) pairs' 32-token blocks
// are divided evenly over the grid whatever the sequence lengths (batches of
// two or more sequences; DecodeParams::balanced).
#include "vq_decode_kernel.cuh"

namespace vqk {

cudaError_t launch_decode_balanced(const DecodeParams& p, int k_sub, int k_bits, int v_sub, int v_bits,
                                   int grid, size_t smem, cudaStream_t stream, bool overlap, int method) {
  return dispatch_decode<true>(p, k_sub, k_bits, v_sub, v_bits, grid, smem, stream, overlap, method);
}

}  // namespace vqk
