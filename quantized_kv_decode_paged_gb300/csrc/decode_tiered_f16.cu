// decode_tiered_f16.cu — instantiations of the decode kernel for the f16-cold /
// f16-hot tiered cache (one operand per Q/P part).
#include "launch_impl.cuh"

namespace da {

cudaError_t launch_tiered_f16_unpacked(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                       cudaStream_t stream) {
  return launch_tiered_f16_pk<false>(D, KVB, p, grid, smem, stream);
}

}  // namespace da
