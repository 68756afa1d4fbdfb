// decode_paged_split.cu — instantiations of the decode kernel for the f16
// paged cache under the split-KV schedule (decode_attn_split_partial), one
// operand per Q/P part.
#include "launch_impl.cuh"

namespace da {

cudaError_t launch_paged_split_unpacked(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                        cudaStream_t stream) {
  return launch_paged_split_pk<false>(D, KVB, p, grid, smem, stream);
}

}  // namespace da
