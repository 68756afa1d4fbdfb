// launch.h — host-side entry points into the kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "kernel_params.h"

namespace da {

// Consumer groups of the decode kernel for head dimension D (two groups
// need about 180 registers per thread; D = 256 keeps one).
inline int decode_groups(int D) { return D <= 128 ? 2 : 1; }

// Launches the decode kernel of `kind` for head dimension D (64/128/256 for
// paged, 128/256 for tiered) with decode_groups(D) consumer groups.  Returns
// cudaErrorInvalidValue for a D that has no instantiation.
cudaError_t launch_decode(int kind, int D, const KParams& p, dim3 grid, int smem_bytes,
                          cudaStream_t stream);

// out/lse from max_splits partial states per (b, h).
cudaError_t launch_split_merge(int rows, int max_splits, int D, const float* o_part,
                               const float* lse_part, float* out, float* lse,
                               cudaStream_t stream);

}  // namespace da
