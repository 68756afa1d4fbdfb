// decode_paged_sparse.cu — instantiations of the decode kernel for the
// block-sparse f16 paged cache (one operand per Q/P part).
#include "launch_impl.cuh"

namespace da {

cudaError_t launch_paged_sparse_unpacked(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                         cudaStream_t stream) {
  return launch_paged_sparse_pk<false>(D, KVB, p, grid, smem, stream);
}

}  // namespace da
