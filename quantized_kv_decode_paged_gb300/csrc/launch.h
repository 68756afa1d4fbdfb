// launch.h — host-side entry points into the kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "kernel_params.h"

namespace da {

// kv heads per work unit for a cache of `kind` with head dimension D and
// Hkv kv heads: enough that one token row of the block is >= 512
// contiguous bytes, and a divisor of Hkv.
inline int decode_kvb(int kind, int D, int Hkv) {
  int pref = cold_int8(kind) ? (D == 128 ? 4 : 2) : (D == 64 ? 4 : D == 128 ? 2 : 1);
  while (pref > 1 && Hkv % pref != 0) pref /= 2;
  return pref;
}

// Geometry numbers of the instantiation (kind, D, KVB) for the host.
struct GeoInfo {
  int W, TOK, TOKH, REGION, THREADS;
};
GeoInfo decode_geo(int kind, int D, int KVB);

// Launches the decode kernel of (kind, D, KVB); `packed` selects the variant
// that packs the f16 and remainder parts of Q and P into one MMA operand
// (valid when p.NH <= 4).  Returns cudaErrorInvalidValue for a combination
// that has no instantiation.
cudaError_t launch_decode(int kind, int D, int KVB, bool packed, const KParams& p, dim3 grid,
                          int smem_bytes, cudaStream_t stream);

// Bytes at the start of a stream-K workspace that hold the ticket counters
// on the current device (they must be zero when a call starts); 0 when the
// device cannot be queried.
size_t workspace_ticket_bytes();

// out/lse from max_splits partial states per (b, h).
cudaError_t launch_split_merge(int rows, int max_splits, int D, const float* o_part,
                               const float* lse_part, float* out, float* lse,
                               cudaStream_t stream);

}  // namespace da
