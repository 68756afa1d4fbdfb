// decode_paged.cu — instantiations of the decode kernel for the f16 paged
// cache, plus the launch switch shared with the tiered unit.
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

cudaError_t launch_tiered(int D, int KVB, const KParams& p, dim3 grid, int smem,
                          cudaStream_t stream);
bool geo_tiered(int D, int KVB, GeoInfo* g);

GeoInfo decode_geo(int kind, int D, int KVB) {
  GeoInfo g{0, 0, 0, 0, 0};
  if (kind == KIND_TIERED) {
    geo_tiered(D, KVB, &g);
    return g;
  }
  if (D == 64 && KVB == 1) return geo_info<KIND_PAGED, 64, 1>();
  if (D == 64 && KVB == 2) return geo_info<KIND_PAGED, 64, 2>();
  if (D == 64 && KVB == 4) return geo_info<KIND_PAGED, 64, 4>();
  if (D == 128 && KVB == 1) return geo_info<KIND_PAGED, 128, 1>();
  if (D == 128 && KVB == 2) return geo_info<KIND_PAGED, 128, 2>();
  if (D == 128 && KVB == 4) return geo_info<KIND_PAGED, 128, 4>();
  if (D == 256 && KVB == 1) return geo_info<KIND_PAGED, 256, 1>();
  return g;
}

cudaError_t launch_decode(int kind, int D, int KVB, const KParams& p, dim3 grid, int smem,
                          cudaStream_t stream) {
  if (kind == KIND_TIERED) return launch_tiered(D, KVB, p, grid, smem, stream);
  if (D == 64 && KVB == 1) return launch_decode_impl<KIND_PAGED, 64, 1>(p, grid, smem, stream);
  if (D == 64 && KVB == 2) return launch_decode_impl<KIND_PAGED, 64, 2>(p, grid, smem, stream);
  if (D == 64 && KVB == 4) return launch_decode_impl<KIND_PAGED, 64, 4>(p, grid, smem, stream);
  if (D == 128 && KVB == 1) return launch_decode_impl<KIND_PAGED, 128, 1>(p, grid, smem, stream);
  if (D == 128 && KVB == 2) return launch_decode_impl<KIND_PAGED, 128, 2>(p, grid, smem, stream);
  if (D == 128 && KVB == 4) return launch_decode_impl<KIND_PAGED, 128, 4>(p, grid, smem, stream);
  if (D == 256 && KVB == 1) return launch_decode_impl<KIND_PAGED, 256, 1>(p, grid, smem, stream);
  return cudaErrorInvalidValue;
}

}  // namespace da
