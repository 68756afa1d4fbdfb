// decode_tiered_f16_packed.cu — instantiations of the decode kernel for the
// f16-cold / f16-hot tiered cache with the Q/P parts packed into one MMA
// operand (at most four query heads per kv head).
#include "launch_impl.cuh"

namespace da {

cudaError_t launch_tiered_f16_packed(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                     cudaStream_t stream) {
  return launch_tiered_f16_pk<true>(D, KVB, p, grid, smem, stream);
}

}  // namespace da
