// decode_paged_split_packed.cu — instantiations of the decode kernel for the
// f16 paged cache under the split-KV schedule, with the Q/P parts packed into
// one MMA operand (at most four query heads per kv head).
#include "launch_impl.cuh"

namespace da {

cudaError_t launch_paged_split_packed(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                      cudaStream_t stream) {
  return launch_paged_split_pk<true>(D, KVB, p, grid, smem, stream);
}

}  // namespace da
