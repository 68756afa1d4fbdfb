// split_merge.cu — second half of flash-decoding: merge S partial softmax
// states (o_s, lse_s) of each (b, h) into out / lse with the log-sum-exp
// form of the (m, d) pair merge of com.microsoft.SparseAttention
// combine_partials:  M = max lse_s, w_s = e^(lse_s - M),
// out = sum w_s o_s / sum w_s, lse = M + ln sum w_s.
#include <math.h>

#include "launch.h"

namespace da {

namespace {

constexpr int kMergeWarps = 4;

__global__ void __launch_bounds__(kMergeWarps * 32)
    split_merge_kernel(int rows, int S, int D, const float* __restrict__ o_part,
                       const float* __restrict__ lse_part, float* __restrict__ out,
                       float* __restrict__ lse) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kMergeWarps + warp;
  if (row >= rows) return;
  const float* lp = lse_part + row * S;
  const float* op = o_part + row * S * D;
  const float ninf = -INFINITY;
  float M = ninf;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, lp[s]);
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (M == ninf) {
    for (int d = lane; d < D; d += 32) out[row * D + d] = 0.f;
    if (lane == 0 && lse) lse[row] = ninf;
    return;
  }
  float wsum = 0.f;
  for (int s = lane; s < S; s += 32) wsum += (lp[s] == ninf) ? 0.f : expf(lp[s] - M);
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  const float inv = 1.f / wsum;
  for (int d = lane; d < D; d += 32) {
    float acc = 0.f;
    for (int s = 0; s < S; ++s) {
      const float ls = lp[s];
      if (ls != ninf) acc += expf(ls - M) * op[(long long)s * D + d];
    }
    out[row * D + d] = acc * inv;
  }
  if (lane == 0 && lse) lse[row] = M + logf(wsum);
}

}  // namespace

cudaError_t launch_split_merge(int rows, int S, int D, const float* o_part, const float* lse_part,
                               float* out, float* lse, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int blocks = (rows + kMergeWarps - 1) / kMergeWarps;
  split_merge_kernel<<<blocks, kMergeWarps * 32, 0, stream>>>(rows, S, D, o_part, lse_part, out,
                                                               lse);
  return cudaGetLastError();
}

}  // namespace da
