// append.cu — the steps either side of a decode step on the cache: writing
// the new token's K/V rows (paged cache, or the hot ring of a tiered cache)
// and, when the ring is full, moving its oldest token into the cold tier —
// quantized to int8 with one f16 scale per (token, kv head), or copied as
// f16.  The cold layout is the one the tiered decode reads: page
// block_table[b][t / block_size], row t % block_size, value d of a row in
// byte lane d % 4 of word d / 4.
//
// These kernels move a few KB per sequence; one CTA per sequence, one warp
// per kv head at a time, 16-byte copies.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/decode_attn.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// 16-byte copy of `bytes` (a multiple of 16) by the CTA's threads.
__device__ __forceinline__ void copy_row(void* dst, const void* src, int bytes) {
  const uint4* s = static_cast<const uint4*>(src);
  uint4* d = static_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < bytes / 16; i += blockDim.x) d[i] = s[i];
}

__global__ void __launch_bounds__(kThreads) append_paged_kernel(
    int Hkv, int D, int bs, int max_blocks, int num_blocks, const uint16_t* k_new,
    const uint16_t* v_new, const int32_t* positions, const int32_t* block_table,
    uint16_t* k_pool, uint16_t* v_pool, int32_t* dev_status) {
  const int b = blockIdx.x;
  const long long pos = positions[b];
  int flag = 0;
  if (pos < 0 || pos >= (long long)max_blocks * bs) {
    flag = DA_DEV_BAD_SEQ_LEN;
  } else {
    const int blk = block_table[(long long)b * max_blocks + pos / bs];
    if (blk < 0 || blk >= num_blocks) {
      flag = DA_DEV_BAD_BLOCK;
    } else {
      const long long row = (long long)blk * bs + pos % bs;
      const long long n = (long long)Hkv * D;
      copy_row(k_pool + row * n, k_new + (long long)b * n, (int)(n * 2));
      copy_row(v_pool + row * n, v_new + (long long)b * n, (int)(n * 2));
    }
  }
  if (flag && threadIdx.x == 0 && dev_status) atomicOr(dev_status, flag);
}

// One row of D f16 values (lane-strided words of four values) to int8 codes:
// scale s16 = f16(max|x| / 127) with the division in f32; code =
// rint(x / f32(s16)) clamped to [-127, 127]; code 0 when s16 is 0 or the
// ratio is not a number.
__device__ void quantize_row(const uint16_t* x, int D, uint32_t* words, uint16_t* scale) {
  const int lane = threadIdx.x & 31;
  const uint2* xv = reinterpret_cast<const uint2*>(x);  // four f16 per uint2
  float m = 0.f;
  for (int w = lane; w < D / 4; w += 32) {
    const uint2 u = xv[w];
    const __half2 a = *reinterpret_cast<const __half2*>(&u.x);
    const __half2 c = *reinterpret_cast<const __half2*>(&u.y);
    m = fmaxf(m, fabsf(__low2float(a)));
    m = fmaxf(m, fabsf(__high2float(a)));
    m = fmaxf(m, fabsf(__low2float(c)));
    m = fmaxf(m, fabsf(__high2float(c)));
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  const __half s16 = __float2half_rn(__fdiv_rn(m, 127.f));
  const float s = __half2float(s16);
  for (int w = lane; w < D / 4; w += 32) {
    const uint2 u = xv[w];
    const __half2 a = *reinterpret_cast<const __half2*>(&u.x);
    const __half2 c = *reinterpret_cast<const __half2*>(&u.y);
    const float v[4] = {__low2float(a), __high2float(a), __low2float(c), __high2float(c)};
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int code = 0;
      if (s != 0.f) {
        const float r = __fdiv_rn(v[i], s);
        if (r == r) code = (int)fminf(fmaxf(rintf(r), -127.f), 127.f);
      }
      word |= (uint32_t)(code & 0xff) << (8 * i);
    }
    words[w] = word;
  }
  if (lane == 0) *scale = __half_as_ushort(s16);
}

// One append step per sequence of a tiered cache (see decode_attn.h).
template <bool F16>
__global__ void __launch_bounds__(kThreads) append_tiered_kernel(
    int Hkv, int D, int bs, int max_blocks, int num_blocks, int W, int cap,
    const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_hot, uint16_t* v_hot,
    void* k_cold, void* v_cold, uint16_t* k_scale, uint16_t* v_scale,
    const int32_t* block_table, int32_t* cold_lens, int32_t* hot_lens, int32_t* hot_starts,
    int32_t* dev_status) {
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  long long cl = cold_lens[b], hl = hot_lens[b], hs = hot_starts[b];
  int flag = 0;
  if (hl < 0 || hl > W || cl < 0 || hs < 0) flag = DA_DEV_BAD_TIER;
  long long cold_row = -1;
  if (!flag && hl == W) {
    if (cl != hs) {
      flag = DA_DEV_BAD_TIER;
    } else if (cl >= (long long)max_blocks * bs) {
      flag = DA_DEV_BAD_SEQ_LEN;
    } else {
      const int blk = block_table[(long long)b * max_blocks + cl / bs];
      if (blk < 0 || blk >= num_blocks)
        flag = DA_DEV_BAD_BLOCK;
      else
        cold_row = (long long)blk * bs + cl % bs;
    }
  }
  if (flag) {
    if (threadIdx.x == 0 && dev_status) atomicOr(dev_status, flag);
    return;  // the sequence is left unchanged (uniform over the CTA)
  }
  const long long n = (long long)Hkv * D;  // values of one token
  if (cold_row >= 0) {
    // the oldest hot token (position hs, slot hs % W) moves to cold position cl
    const long long hot_row = (long long)b * cap + hs % W;
    if constexpr (F16) {
      copy_row(static_cast<uint16_t*>(k_cold) + cold_row * n, k_hot + hot_row * n, (int)(n * 2));
      copy_row(static_cast<uint16_t*>(v_cold) + cold_row * n, v_hot + hot_row * n, (int)(n * 2));
    } else {
      for (int kv = warp; kv < Hkv; kv += kWarps) {
        const long long r = cold_row * Hkv + kv;
        quantize_row(k_hot + (hot_row * Hkv + kv) * D, D,
                     static_cast<uint32_t*>(k_cold) + r * (D / 4), k_scale + r);
        quantize_row(v_hot + (hot_row * Hkv + kv) * D, D,
                     static_cast<uint32_t*>(v_cold) + r * (D / 4), v_scale + r);
      }
    }
    ++cl;
    ++hs;
    --hl;
  }
  __syncthreads();  // the old row of the slot is read before it is overwritten
  const long long slot_row = (long long)b * cap + (hs + hl) % W;
  copy_row(k_hot + slot_row * n, k_new + (long long)b * n, (int)(n * 2));
  copy_row(v_hot + slot_row * n, v_new + (long long)b * n, (int)(n * 2));
  if (threadIdx.x == 0) {
    cold_lens[b] = (int32_t)cl;
    hot_lens[b] = (int32_t)(hl + 1);
    hot_starts[b] = (int32_t)hs;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Geometry shared by the append entry points.
int check_append(const da_params* p) {
  if (!p) return DA_ERR_INVALID;
  if (p->batch < 0 || p->num_kv_heads <= 0 || p->head_dim <= 0) return DA_ERR_INVALID;
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256) return DA_ERR_UNSUPPORTED;
  if (p->block_size <= 0 || p->max_blocks_per_seq <= 0 || p->num_blocks <= 0)
    return DA_ERR_INVALID;
  if ((long long)p->num_blocks * p->block_size > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
  if ((long long)p->max_blocks_per_seq * p->block_size > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
  if ((long long)p->num_kv_heads * p->head_dim * 2 > (1LL << 30)) return DA_ERR_UNSUPPORTED;
  return DA_OK;
}

template <bool F16>
int append_tiered(const da_params* p, int32_t hot_window, int32_t hot_capacity,
                  const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_hot, uint16_t* v_hot,
                  void* k_cold, void* v_cold, uint16_t* k_scale, uint16_t* v_scale,
                  const int32_t* block_table, int32_t* cold_lens, int32_t* hot_lens,
                  int32_t* hot_starts, int32_t* dev_status, void* stream) {
  int st = check_append(p);
  if (st != DA_OK) return st;
  if (hot_window <= 0 || hot_capacity < hot_window) return DA_ERR_INVALID;
  if (!k_new || !v_new || !k_hot || !v_hot || !k_cold || !v_cold || !block_table ||
      !cold_lens || !hot_lens || !hot_starts)
    return DA_ERR_INVALID;
  if (!F16 && (!k_scale || !v_scale)) return DA_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_hot) || !aligned16(v_hot) ||
      !aligned16(k_cold) || !aligned16(v_cold))
    return DA_ERR_INVALID;
  if (p->batch == 0) return DA_OK;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  append_tiered_kernel<F16><<<p->batch, kThreads, 0, s>>>(
      p->num_kv_heads, p->head_dim, p->block_size, p->max_blocks_per_seq, p->num_blocks,
      hot_window, hot_capacity, k_new, v_new, k_hot, v_hot, k_cold, v_cold, k_scale, v_scale,
      block_table, cold_lens, hot_lens, hot_starts, dev_status);
  return cudaGetLastError() == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

}  // namespace

extern "C" {

int decode_attn_append_paged(const da_params* p, const uint16_t* k_new, const uint16_t* v_new,
                             const int32_t* positions, const int32_t* block_table,
                             uint16_t* k_pool, uint16_t* v_pool, int32_t* dev_status,
                             void* stream) {
  int st = check_append(p);
  if (st != DA_OK) return st;
  if (!k_new || !v_new || !positions || !block_table || !k_pool || !v_pool) return DA_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
    return DA_ERR_INVALID;
  if (p->batch == 0) return DA_OK;
  append_paged_kernel<<<p->batch, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      p->num_kv_heads, p->head_dim, p->block_size, p->max_blocks_per_seq, p->num_blocks, k_new,
      v_new, positions, block_table, k_pool, v_pool, dev_status);
  return cudaGetLastError() == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

int decode_attn_append_tiered_int8(const da_params* p, int32_t hot_window, int32_t hot_capacity,
                                   const uint16_t* k_new, const uint16_t* v_new,
                                   uint16_t* k_hot, uint16_t* v_hot, uint32_t* k_cold,
                                   uint32_t* v_cold, uint16_t* k_scale, uint16_t* v_scale,
                                   const int32_t* block_table, int32_t* cold_lens,
                                   int32_t* hot_lens, int32_t* hot_starts, int32_t* dev_status,
                                   void* stream) {
  return append_tiered<false>(p, hot_window, hot_capacity, k_new, v_new, k_hot, v_hot, k_cold,
                              v_cold, k_scale, v_scale, block_table, cold_lens, hot_lens,
                              hot_starts, dev_status, stream);
}

int decode_attn_append_tiered_f16(const da_params* p, int32_t hot_window, int32_t hot_capacity,
                                  const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_hot,
                                  uint16_t* v_hot, uint16_t* k_cold, uint16_t* v_cold,
                                  const int32_t* block_table, int32_t* cold_lens,
                                  int32_t* hot_lens, int32_t* hot_starts, int32_t* dev_status,
                                  void* stream) {
  return append_tiered<true>(p, hot_window, hot_capacity, k_new, v_new, k_hot, v_hot, k_cold,
                             v_cold, nullptr, nullptr, block_table, cold_lens, hot_lens,
                             hot_starts, dev_status, stream);
}

}  // extern "C"
