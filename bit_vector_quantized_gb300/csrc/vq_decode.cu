// vq_decode.cu -- the split attention kernel (vq_decode_kernel.cuh) with fixed
// splits: each (sequence, KV head) is cut into `splits` ranges of max_seq_len
// and the units go round-robin over the grid.  Length-balanced launches are
// instantiated in vq_decode_balanced.cu, a translation unit of its own so the
// two families compile in parallel.
#include "vq_decode_kernel.cuh"

namespace vqk {

cudaError_t launch_decode(const DecodeParams& p, int k_sub, int k_bits, int v_sub, int v_bits,
                          int grid, size_t smem, cudaStream_t stream, bool overlap, int method) {
  if (p.balanced) return launch_decode_balanced(p, k_sub, k_bits, v_sub, v_bits, grid, smem, stream, overlap, method);
  return dispatch_decode<false>(p, k_sub, k_bits, v_sub, v_bits, grid, smem, stream, overlap, method);
}

}  // namespace vqk
