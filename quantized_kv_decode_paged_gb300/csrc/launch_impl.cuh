// launch_impl.cuh — the launch wrapper of one kernel instantiation, shared by
// the translation units that instantiate the decode kernel.
#pragma once

#include <atomic>

#include "decode_kernel.cuh"
#include "launch.h"

namespace da {

// The shared-memory opt-in of each instantiation is set once per device.
// The flags are atomics: host threads making their first call together may
// each set the (idempotent) attribute.
template <int KIND, int D, int KVB, bool PK>
cudaError_t launch_decode_impl(const KParams& p, dim3 grid, int smem, cudaStream_t stream) {
  static std::atomic<int> configured[128];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 128 || !configured[dev].load(std::memory_order_acquire)) {
    err = cudaFuncSetAttribute(decode_attn_kernel<KIND, D, KVB, PK>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 128) configured[dev].store(1, std::memory_order_release);
  }
  decode_attn_kernel<KIND, D, KVB, PK><<<grid, Geo<KIND, D, KVB>::THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int KIND, int D, int KVB>
GeoInfo geo_info() {
  using Gm = Geo<KIND, D, KVB>;
  return GeoInfo{Gm::W, Gm::TOK, Gm::TOKH, Gm::REGION, Gm::THREADS};
}

// Instantiations of one cache kind and packing mode, by (D, KVB).
template <bool PK>
cudaError_t launch_paged_pk(int D, int KVB, const KParams& p, dim3 grid, int smem,
                            cudaStream_t stream) {
  if (D == 64 && KVB == 1) return launch_decode_impl<KIND_PAGED, 64, 1, PK>(p, grid, smem, stream);
  if (D == 64 && KVB == 2) return launch_decode_impl<KIND_PAGED, 64, 2, PK>(p, grid, smem, stream);
  if (D == 64 && KVB == 4) return launch_decode_impl<KIND_PAGED, 64, 4, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 1) return launch_decode_impl<KIND_PAGED, 128, 1, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 2) return launch_decode_impl<KIND_PAGED, 128, 2, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 4) return launch_decode_impl<KIND_PAGED, 128, 4, PK>(p, grid, smem, stream);
  if (D == 256 && KVB == 1) return launch_decode_impl<KIND_PAGED, 256, 1, PK>(p, grid, smem, stream);
  return cudaErrorInvalidValue;
}

template <bool PK>
cudaError_t launch_paged_split_pk(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                  cudaStream_t stream) {
  if (D == 64 && KVB == 1) return launch_decode_impl<KIND_PAGED_SPLIT, 64, 1, PK>(p, grid, smem, stream);
  if (D == 64 && KVB == 2) return launch_decode_impl<KIND_PAGED_SPLIT, 64, 2, PK>(p, grid, smem, stream);
  if (D == 64 && KVB == 4) return launch_decode_impl<KIND_PAGED_SPLIT, 64, 4, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 1) return launch_decode_impl<KIND_PAGED_SPLIT, 128, 1, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 2) return launch_decode_impl<KIND_PAGED_SPLIT, 128, 2, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 4) return launch_decode_impl<KIND_PAGED_SPLIT, 128, 4, PK>(p, grid, smem, stream);
  if (D == 256 && KVB == 1) return launch_decode_impl<KIND_PAGED_SPLIT, 256, 1, PK>(p, grid, smem, stream);
  return cudaErrorInvalidValue;
}

template <bool PK>
cudaError_t launch_tiered_pk(int D, int KVB, const KParams& p, dim3 grid, int smem,
                             cudaStream_t stream) {
  if (D == 128 && KVB == 1) return launch_decode_impl<KIND_TIERED, 128, 1, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 2) return launch_decode_impl<KIND_TIERED, 128, 2, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 4) return launch_decode_impl<KIND_TIERED, 128, 4, PK>(p, grid, smem, stream);
  if (D == 256 && KVB == 1) return launch_decode_impl<KIND_TIERED, 256, 1, PK>(p, grid, smem, stream);
  if (D == 256 && KVB == 2) return launch_decode_impl<KIND_TIERED, 256, 2, PK>(p, grid, smem, stream);
  return cudaErrorInvalidValue;
}

template <bool PK>
cudaError_t launch_tiered_f16_pk(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                 cudaStream_t stream) {
  if (D == 64 && KVB == 1) return launch_decode_impl<KIND_TIERED_F16, 64, 1, PK>(p, grid, smem, stream);
  if (D == 64 && KVB == 2) return launch_decode_impl<KIND_TIERED_F16, 64, 2, PK>(p, grid, smem, stream);
  if (D == 64 && KVB == 4) return launch_decode_impl<KIND_TIERED_F16, 64, 4, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 1) return launch_decode_impl<KIND_TIERED_F16, 128, 1, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 2) return launch_decode_impl<KIND_TIERED_F16, 128, 2, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 4) return launch_decode_impl<KIND_TIERED_F16, 128, 4, PK>(p, grid, smem, stream);
  if (D == 256 && KVB == 1) return launch_decode_impl<KIND_TIERED_F16, 256, 1, PK>(p, grid, smem, stream);
  return cudaErrorInvalidValue;
}

template <bool PK>
cudaError_t launch_paged_multi_pk(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                  cudaStream_t stream) {
  if (D == 64 && KVB == 1) return launch_decode_impl<KIND_PAGED_MULTI, 64, 1, PK>(p, grid, smem, stream);
  if (D == 64 && KVB == 2) return launch_decode_impl<KIND_PAGED_MULTI, 64, 2, PK>(p, grid, smem, stream);
  if (D == 64 && KVB == 4) return launch_decode_impl<KIND_PAGED_MULTI, 64, 4, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 1) return launch_decode_impl<KIND_PAGED_MULTI, 128, 1, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 2) return launch_decode_impl<KIND_PAGED_MULTI, 128, 2, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 4) return launch_decode_impl<KIND_PAGED_MULTI, 128, 4, PK>(p, grid, smem, stream);
  if (D == 256 && KVB == 1) return launch_decode_impl<KIND_PAGED_MULTI, 256, 1, PK>(p, grid, smem, stream);
  return cudaErrorInvalidValue;
}

template <bool PK>
cudaError_t launch_paged_sparse_pk(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                   cudaStream_t stream) {
  if (D == 64 && KVB == 1) return launch_decode_impl<KIND_PAGED_SPARSE, 64, 1, PK>(p, grid, smem, stream);
  if (D == 64 && KVB == 2) return launch_decode_impl<KIND_PAGED_SPARSE, 64, 2, PK>(p, grid, smem, stream);
  if (D == 64 && KVB == 4) return launch_decode_impl<KIND_PAGED_SPARSE, 64, 4, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 1) return launch_decode_impl<KIND_PAGED_SPARSE, 128, 1, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 2) return launch_decode_impl<KIND_PAGED_SPARSE, 128, 2, PK>(p, grid, smem, stream);
  if (D == 128 && KVB == 4) return launch_decode_impl<KIND_PAGED_SPARSE, 128, 4, PK>(p, grid, smem, stream);
  if (D == 256 && KVB == 1) return launch_decode_impl<KIND_PAGED_SPARSE, 256, 1, PK>(p, grid, smem, stream);
  return cudaErrorInvalidValue;
}

// Defined in the instantiating translation units.
cudaError_t launch_paged_unpacked(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                  cudaStream_t stream);
cudaError_t launch_paged_packed(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                cudaStream_t stream);
cudaError_t launch_paged_split_unpacked(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                        cudaStream_t stream);
cudaError_t launch_paged_split_packed(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                      cudaStream_t stream);
cudaError_t launch_tiered_unpacked(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                   cudaStream_t stream);
cudaError_t launch_tiered_packed(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                 cudaStream_t stream);
cudaError_t launch_paged_multi_unpacked(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                        cudaStream_t stream);
cudaError_t launch_paged_multi_packed(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                      cudaStream_t stream);
cudaError_t launch_tiered_f16_unpacked(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                       cudaStream_t stream);
cudaError_t launch_tiered_f16_packed(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                     cudaStream_t stream);
cudaError_t launch_paged_sparse_unpacked(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                         cudaStream_t stream);
cudaError_t launch_paged_sparse_packed(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                       cudaStream_t stream);

}  // namespace da
