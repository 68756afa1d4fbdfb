// decode_tiered.cu — instantiations of the decode kernel for the int8-cold /
// f16-hot tiered cache.
#include "decode_kernel.cuh"
#include "launch.h"

namespace da {

template <int KIND, int D, int GROUPS>
cudaError_t launch_decode_impl(const KParams& p, dim3 grid, int smem, cudaStream_t stream) {
  static int configured[128] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < 128 && !configured[dev]) {
    err = cudaFuncSetAttribute(decode_attn_kernel<KIND, D, GROUPS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (err != cudaSuccess) return err;
    configured[dev] = 1;
  }
  decode_attn_kernel<KIND, D, GROUPS><<<grid, cta_threads(GROUPS), smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tiered(int D, const KParams& p, dim3 grid, int smem, cudaStream_t stream) {
  switch (D) {
    case 128: return launch_decode_impl<KIND_TIERED, 128, 2>(p, grid, smem, stream);
    case 256: return launch_decode_impl<KIND_TIERED, 256, 1>(p, grid, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace da
