// decode_paged.cu — instantiations of the decode kernel for the f16 paged
// cache (one operand per Q/P part), plus the geometry and launch switches
// over every cache kind.
#include "launch_impl.cuh"

namespace da {

cudaError_t launch_paged_unpacked(int D, int KVB, const KParams& p, dim3 grid, int smem,
                                  cudaStream_t stream) {
  return launch_paged_pk<false>(D, KVB, p, grid, smem, stream);
}

GeoInfo decode_geo(int kind, int D, int KVB) {
  GeoInfo g{0, 0, 0, 0, 0};
  if (kind == KIND_PAGED_MULTI) {
    if (D == 64 && KVB == 1) return geo_info<KIND_PAGED_MULTI, 64, 1>();
    if (D == 64 && KVB == 2) return geo_info<KIND_PAGED_MULTI, 64, 2>();
    if (D == 64 && KVB == 4) return geo_info<KIND_PAGED_MULTI, 64, 4>();
    if (D == 128 && KVB == 1) return geo_info<KIND_PAGED_MULTI, 128, 1>();
    if (D == 128 && KVB == 2) return geo_info<KIND_PAGED_MULTI, 128, 2>();
    if (D == 128 && KVB == 4) return geo_info<KIND_PAGED_MULTI, 128, 4>();
    if (D == 256 && KVB == 1) return geo_info<KIND_PAGED_MULTI, 256, 1>();
    return g;
  }
  if (kind == KIND_PAGED_SPARSE) {
    if (D == 64 && KVB == 1) return geo_info<KIND_PAGED_SPARSE, 64, 1>();
    if (D == 64 && KVB == 2) return geo_info<KIND_PAGED_SPARSE, 64, 2>();
    if (D == 64 && KVB == 4) return geo_info<KIND_PAGED_SPARSE, 64, 4>();
    if (D == 128 && KVB == 1) return geo_info<KIND_PAGED_SPARSE, 128, 1>();
    if (D == 128 && KVB == 2) return geo_info<KIND_PAGED_SPARSE, 128, 2>();
    if (D == 128 && KVB == 4) return geo_info<KIND_PAGED_SPARSE, 128, 4>();
    if (D == 256 && KVB == 1) return geo_info<KIND_PAGED_SPARSE, 256, 1>();
    return g;
  }
  if (kind == KIND_TIERED_F16) {
    if (D == 64 && KVB == 1) return geo_info<KIND_TIERED_F16, 64, 1>();
    if (D == 64 && KVB == 2) return geo_info<KIND_TIERED_F16, 64, 2>();
    if (D == 64 && KVB == 4) return geo_info<KIND_TIERED_F16, 64, 4>();
    if (D == 128 && KVB == 1) return geo_info<KIND_TIERED_F16, 128, 1>();
    if (D == 128 && KVB == 2) return geo_info<KIND_TIERED_F16, 128, 2>();
    if (D == 128 && KVB == 4) return geo_info<KIND_TIERED_F16, 128, 4>();
    if (D == 256 && KVB == 1) return geo_info<KIND_TIERED_F16, 256, 1>();
    return g;
  }
  if (kind == KIND_TIERED) {
    if (D == 128 && KVB == 1) return geo_info<KIND_TIERED, 128, 1>();
    if (D == 128 && KVB == 2) return geo_info<KIND_TIERED, 128, 2>();
    if (D == 128 && KVB == 4) return geo_info<KIND_TIERED, 128, 4>();
    if (D == 256 && KVB == 1) return geo_info<KIND_TIERED, 256, 1>();
    if (D == 256 && KVB == 2) return geo_info<KIND_TIERED, 256, 2>();
    return g;
  }
  // KIND_PAGED and KIND_PAGED_SPLIT (the same geometry)
  if (D == 64 && KVB == 1) return geo_info<KIND_PAGED, 64, 1>();
  if (D == 64 && KVB == 2) return geo_info<KIND_PAGED, 64, 2>();
  if (D == 64 && KVB == 4) return geo_info<KIND_PAGED, 64, 4>();
  if (D == 128 && KVB == 1) return geo_info<KIND_PAGED, 128, 1>();
  if (D == 128 && KVB == 2) return geo_info<KIND_PAGED, 128, 2>();
  if (D == 128 && KVB == 4) return geo_info<KIND_PAGED, 128, 4>();
  if (D == 256 && KVB == 1) return geo_info<KIND_PAGED, 256, 1>();
  return g;
}

cudaError_t launch_decode(int kind, int D, int KVB, bool packed, const KParams& p, dim3 grid,
                          int smem, cudaStream_t stream) {
  if (kind == KIND_TIERED)
    return packed ? launch_tiered_packed(D, KVB, p, grid, smem, stream)
                  : launch_tiered_unpacked(D, KVB, p, grid, smem, stream);
  if (kind == KIND_TIERED_F16)
    return packed ? launch_tiered_f16_packed(D, KVB, p, grid, smem, stream)
                  : launch_tiered_f16_unpacked(D, KVB, p, grid, smem, stream);
  if (kind == KIND_PAGED_SPARSE)
    return packed ? launch_paged_sparse_packed(D, KVB, p, grid, smem, stream)
                  : launch_paged_sparse_unpacked(D, KVB, p, grid, smem, stream);
  if (kind == KIND_PAGED_MULTI)
    return packed ? launch_paged_multi_packed(D, KVB, p, grid, smem, stream)
                  : launch_paged_multi_unpacked(D, KVB, p, grid, smem, stream);
  if (kind == KIND_PAGED_SPLIT)
    return packed ? launch_paged_split_packed(D, KVB, p, grid, smem, stream)
                  : launch_paged_split_unpacked(D, KVB, p, grid, smem, stream);
  return packed ? launch_paged_packed(D, KVB, p, grid, smem, stream)
                : launch_paged_unpacked(D, KVB, p, grid, smem, stream);
}

}  // namespace da
