// decode_tiered.cu — instantiations of the decode kernel for the int8-cold /
// f16-hot tiered cache.
#include "decode_kernel.cuh"
#include "launch.h"

namespace da {

template <int KIND, int D, int KVB>
cudaError_t launch_decode_impl(const KParams& p, dim3 grid, int smem, cudaStream_t stream) {
  static int configured[128] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < 128 && !configured[dev]) {
    err = cudaFuncSetAttribute(decode_attn_kernel<KIND, D, KVB>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (err != cudaSuccess) return err;
    configured[dev] = 1;
  }
  decode_attn_kernel<KIND, D, KVB><<<grid, Geo<KIND, D, KVB>::THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int KIND, int D, int KVB>
GeoInfo geo_info() {
  using Gm = Geo<KIND, D, KVB>;
  return GeoInfo{Gm::W, Gm::TOK, Gm::TOKH, Gm::REGION, Gm::THREADS};
}

bool geo_tiered(int D, int KVB, GeoInfo* g) {
  if (D == 128 && KVB == 1) { *g = geo_info<KIND_TIERED, 128, 1>(); return true; }
  if (D == 128 && KVB == 2) { *g = geo_info<KIND_TIERED, 128, 2>(); return true; }
  if (D == 128 && KVB == 4) { *g = geo_info<KIND_TIERED, 128, 4>(); return true; }
  if (D == 256 && KVB == 1) { *g = geo_info<KIND_TIERED, 256, 1>(); return true; }
  if (D == 256 && KVB == 2) { *g = geo_info<KIND_TIERED, 256, 2>(); return true; }
  return false;
}

cudaError_t launch_tiered(int D, int KVB, const KParams& p, dim3 grid, int smem,
                          cudaStream_t stream) {
  if (D == 128 && KVB == 1) return launch_decode_impl<KIND_TIERED, 128, 1>(p, grid, smem, stream);
  if (D == 128 && KVB == 2) return launch_decode_impl<KIND_TIERED, 128, 2>(p, grid, smem, stream);
  if (D == 128 && KVB == 4) return launch_decode_impl<KIND_TIERED, 128, 4>(p, grid, smem, stream);
  if (D == 256 && KVB == 1) return launch_decode_impl<KIND_TIERED, 256, 1>(p, grid, smem, stream);
  if (D == 256 && KVB == 2) return launch_decode_impl<KIND_TIERED, 256, 2>(p, grid, smem, stream);
  return cudaErrorInvalidValue;
}

}  // namespace da
