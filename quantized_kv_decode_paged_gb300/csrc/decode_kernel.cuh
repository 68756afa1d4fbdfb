// decode_kernel.cuh — single-query GQA attention over a paged (optionally
// int8-tiered) KV cache for sm_103a.
//
// What is computed (per sequence b, query head h, kv = h / (Hq/Hkv)):
//   s_t = scale * <q, k_t>, then cap * tanh(s_t / cap) when cap > 0
//   (@simulatte/doppler 0.1.0 "attention_f16kv.wgsl", softcap step),
//   keys masked by the causal / sliding-window rule of is_masked there,
//   out = softmax(s) V and lse = max + ln(sum)
//   (boostr "paged_attention.wgsl", paged_attention_fwd_f32).
//   The int8 cold tier decodes byte d%4 of word d/4 as a signed value times
//   the f16 scale of its (token, kv head), and hot key j sits in ring slot
//   (hot_start + j) % W (doppler "attention_decode_tiered_int8_f16kv.wgsl",
//   read_cold_k / get_hot_pos).
//
// How (GB300 design, not the pages' WGSL):
//   * A work unit is (sequence, block of KVB kv heads, group of <= 8 query
//     heads per kv head).  The KVB heads make every token row read from the
//     pool at least 512 contiguous bytes (Geo in kernel_params.h), and the
//     query heads of one kv head share each K/V byte: they are the n = 8
//     dimension of mma.m16n8k16, so QK^T is S^T[16 keys x 8 heads] =
//     K[16 x D] * Q^T and PV is O^T[D x 8] += V^T[D x 16] * P^T[16 x 8].
//   * f32 Q and P enter the f16 tensor cores as hi + lo f16 pairs, so the
//     products keep ~22 bits; accumulation is f32.  int8 values become exact
//     f16 integers (byte bias + magic-number subtraction); the per-key
//     scales multiply the score (K) and fold into the weight (V).
//   * One producer warp streams tiles through TMA into a ring of shared-
//     memory stages guarded by mbarriers.  The tensor maps put the token
//     dimension inside the (128-byte slice, kv head) dimensions, so one box
//     per page covers KVB heads x all of D, and the 128-byte swizzle keeps
//     eight consecutive keys of one slice in distinct banks.  Each consumer
//     warp owns one kv head of the block and 16-key groups of every tile,
//     with its own online-softmax state; the warps of a head merge their
//     states through a register-level tree at the end of a unit.
//   * Stream-K split-KV: the key tiles of all units are concatenated and cut
//     into one equal share per CTA.  A unit cut between CTAs leaves partial
//     (o, lse) states in the workspace; the last CTA to finish the unit
//     (atomic ticket, no waiting) merges them with the log-sum-exp form of
//     com.microsoft.SparseAttention combine_partials.
#pragma once

#include "kernel_params.h"
#include "ptx.cuh"

namespace da {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_inff();

enum { DEST_OUT = 0, DEST_PARTIAL = 1, DEST_SPLIT = 2 };
enum { TK_PAGED = 0, TK_COLD = 1, TK_HOT = 2 };

struct Seg {
  int b, kvb, hg, unit;  // kvb: index of the kv-head block
  int i0, i1;            // unit-local tile range
  int vlo, vhi;          // visible absolute key positions of this segment
  int dest, slot;
  int pidx;              // index of b's plan entry
};

struct SegIter {
  long long g, g_end;  // next position and end of this CTA's range
  long long s0;        // start of the range
  long long fwd_end;   // end of the forward pass
  long long last0;     // start of the range's last segment when it goes first, else -1
  int n;
};

struct Misc {
  int flags;
  int ticket;
  int abort;  // set when a wait gave up: see note_abort
};

// A wait that gave up (its time limit passed, or another warp had already
// given up) puts the CTA in abort mode: every later wait returns at once,
// the producer issues no more copies, and every warp still runs its loops
// to the end -- on whatever is in shared memory -- so that the barriers
// stay matched and the kernel ends.  The host sees DEV_TIMEOUT.
__device__ __forceinline__ void note_abort(Misc* misc) {
  *reinterpret_cast<volatile int*>(&misc->abort) = 1;
  atomicOr(&misc->flags, DEV_TIMEOUT);
}
__device__ __forceinline__ const volatile int* abort_flag(Misc* misc) {
  return reinterpret_cast<const volatile int*>(&misc->abort);
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.b16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128_zero(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// ------------------------------------------------------------------ plan
__device__ __forceinline__ int ceil_div_i(long long a, int b) { return (int)((a + b - 1) / b); }

// Plan of sequence b (lengths validated, visible range, tile counts for
// paged / cold tiles of TOK keys and hot tiles of TOKH slots); returns
// device-status bits.
template <int KIND, int TOK, int TOKH>
__device__ __forceinline__ int plan_sequence(const KParams& p, int b, SeqPlan& e) {
  int flags = 0;
  const long long cap = (long long)p.max_blocks * p.bs;
  e.ntiles = 0;
  e.t0 = 0;
  e.ncold = 0;
  e.ha0 = e.ha1 = e.hb0 = e.hb1 = 0;
  e.hot_start = e.hot_len = 0;
  e.cold_len = 0;
  long long qp;
  bool empty = false;
  long long L = 0;  // paged: keys 0..L-1
  long long cl = 0, hl = 0, hs = 0;
  if (is_paged(KIND)) {
    L = p.seq_lens[b];
    if (L < 0) { flags |= DEV_BAD_SEQ_LEN; L = 0; }
    if (L > cap) { flags |= DEV_BAD_SEQ_LEN; L = cap; }
    // the block-sparse bitmasks cover the host's length bound
    if (KIND == KIND_PAGED_SPARSE && L > p.sp_max_len) { flags |= DEV_BAD_SEQ_LEN; L = p.sp_max_len; }
    qp = L - p.q_len;  // query token 0; the T new tokens are the last T keys
  } else {
    cl = p.cold_lens ? p.cold_lens[b] : p.cold_len;
    hl = p.hot_lens ? p.hot_lens[b] : p.hot_len;
    hs = p.hot_starts ? p.hot_starts[b] : p.hot_start;
    if (cl < 0) { flags |= DEV_BAD_TIER; cl = 0; }
    if (cl > cap) { flags |= DEV_BAD_SEQ_LEN; cl = cap; }
    const long long hot_limit = p.hot_window > 0 ? p.hot_window : p.hot_cap;
    if (hl < 0) { flags |= DEV_BAD_TIER; hl = 0; }
    if (hl > hot_limit) { flags |= DEV_BAD_TIER; hl = hot_limit; }
    if (hs < 0) { flags |= DEV_BAD_TIER; hs = 0; }
    qp = hl > 0 ? hs + hl - 1 : cl - 1;
  }
  if (p.q_pos) {
    qp = p.q_pos[b];
    if (qp < 0) { flags |= DEV_BAD_QPOS; empty = true; }
  }
  e.qp0 = (int)qp;
  // is_masked: causal hides keys after a token's position qp + t; a window W
  // hides keys below qp + t - W + 1 once qp + t >= W.  [lo, hi) is the union
  // over the T tokens (token 0's lower bound, token T-1's upper bound).
  long long lo = (p.window > 0 && qp >= p.window) ? qp - p.window + 1 : 0;
  long long hi = p.causal ? qp + p.q_len : (long long)0x7fffffff;
  if (lo < 0) lo = 0;
  if (hi > 0x7fffffff) hi = 0x7fffffff;
  e.lo = (int)lo;
  e.hi = (int)hi;
  if (is_paged(KIND)) e.cold_len = empty ? 0 : (int)L;  // the clamped length
  if (empty) return flags;
  if (is_paged(KIND)) {
    long long vh = hi < L ? hi : L;
    e.hi = (int)vh;
    if (vh > lo) {
      e.t0 = (int)(lo / TOK);
      e.ntiles = ceil_div_i(vh, TOK) - e.t0;
    }
  } else {
    e.cold_len = (int)cl;
    e.hot_start = (int)hs;
    e.hot_len = (int)hl;
    long long ch = hi < cl ? hi : cl;
    if (ch > lo) {
      e.t0 = (int)(lo / TOK);
      e.ncold = ceil_div_i(ch, TOK) - e.t0;
    }
    long long j0 = lo - hs > 0 ? lo - hs : 0;
    long long j1 = hi - hs < hl ? hi - hs : hl;
    int nhot = 0;
    if (j1 > j0) {
      if (p.hot_window > 0) {
        // visible ring slots: [s0, s0 + n) modulo W, as one or two tile runs
        const int W = p.hot_window;
        const int nT = ceil_div_i(W, TOKH);
        long long s0 = (hs + j0) % W;
        long long n = j1 - j0;
        if (s0 + n <= W) {
          e.ha0 = (int)(s0 / TOKH);
          e.ha1 = ceil_div_i(s0 + n, TOKH);
        } else {
          int te = ceil_div_i(s0 + n - W, TOKH);
          int ts = (int)(s0 / TOKH);
          if (te > ts) {
            e.ha0 = 0;
            e.ha1 = nT;
          } else {
            e.ha0 = 0;
            e.ha1 = te;
            e.hb0 = ts;
            e.hb1 = nT;
          }
        }
      } else {
        e.ha0 = (int)(j0 / TOKH);
        e.ha1 = ceil_div_i(j1, TOKH);
      }
      nhot = (e.ha1 - e.ha0) + (e.hb1 - e.hb0);
    }
    e.ntiles = e.ncold + nhot;
  }
  return flags;
}

// Shared-memory plan storage: 4 ints per sequence for the one-token paged
// kernels, the whole SeqPlan for the others.
template <int KIND>
struct PlanStore {
  uint8_t* base;
  __device__ __forceinline__ void put(int b, const SeqPlan& e) const {
    if constexpr (one_token_paged(KIND)) {
      reinterpret_cast<SeqPlanPaged*>(base)[b] = SeqPlanPaged{e.lo, e.hi, e.t0, e.ntiles};
    } else {
      reinterpret_cast<SeqPlan*>(base)[b] = e;
    }
  }
  __device__ __forceinline__ SeqPlan get(int b) const {
    SeqPlan e;
    if constexpr (one_token_paged(KIND)) {
      const SeqPlanPaged s = reinterpret_cast<const SeqPlanPaged*>(base)[b];
      e.lo = s.lo;
      e.hi = s.hi;
      e.t0 = s.t0;
      e.ntiles = s.ntiles;
      e.qp0 = s.hi - 1;  // (not used: one query token)
      e.ncold = s.ntiles;
      e.hot_start = e.hot_len = e.ha0 = e.ha1 = e.hb0 = e.hb1 = e.cold_len = 0;
    } else {
      e = reinterpret_cast<const SeqPlan*>(base)[b];
    }
    return e;
  }
  __device__ __forceinline__ int ntiles(int b) const {
    if constexpr (one_token_paged(KIND)) {
      return reinterpret_cast<const SeqPlanPaged*>(base)[b].ntiles;
    } else {
      return reinterpret_cast<const SeqPlan*>(base)[b].ntiles;
    }
  }
};

// Exclusive prefix of ntiles * units_per_seq over the batch (one warp).
template <int KIND>
__device__ __forceinline__ void plan_prefix(const PlanStore<KIND>& plan, int* pre, int B, int upb,
                                            int lane) {
  const int per = (B + 31) / 32;
  const int b0 = lane * per;
  long long sum = 0;
#pragma unroll 1
  for (int i = 0; i < per; ++i)
    if (b0 + i < B) sum += (long long)plan.ntiles(b0 + i) * upb;
  long long incl = sum;
  for (int off = 1; off < 32; off <<= 1) {
    long long v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  long long run = incl - sum;
#pragma unroll 1
  for (int i = 0; i < per; ++i) {
    if (b0 + i < B) {
      pre[b0 + i] = (int)run;
      run += (long long)plan.ntiles(b0 + i) * upb;
    }
  }
  if (lane == 31) pre[B] = (int)incl;
}

// ----------------------------------------------------------- scheduling
__device__ __forceinline__ int stream_cta_of(long long g, long long T, int grid) {
  return (int)(((g + 1) * grid - 1) / T);
}
__device__ __forceinline__ long long stream_start(int c, long long T, int grid) {
  // floor(c * T / grid) in 32-bit steps (tile counts fit in int; c <= grid)
  const unsigned t = (unsigned)T, g = (unsigned)grid, uc = (unsigned)c;
  const unsigned q = t / g, r = t - q * g;
  return (long long)(uc * q + (uc * r) / g);
}
// CTAs that share the key tiles in the STREAM schedule: never more than the
// tiles, so every participating CTA owns at least one tile.
__device__ __forceinline__ int stream_grid(const KParams& p, long long T) {
  return (int)(T < p.grid ? T : p.grid);
}
__device__ __forceinline__ int units_per_seq(const KParams& p) { return (p.Hkv / p.KVU) * p.HGN; }

// Query rows (virtual heads) of head group hg of a kv head: kHeadTile, or
// fewer in the last group.  Virtual head j = t*G + g is head g of the kv
// head's group for query token t.
__device__ __forceinline__ int unit_nh(const KParams& p, int hg) {
  const int n = p.Gv - hg * kHeadTile;
  return n < kHeadTile ? n : kHeadTile;
}

// kv head and head group of warp slot ks of a unit (kv-head block kvb, first
// head group hg0).  Only the four-slot instantiations share a unit between
// head groups; the others keep one head group per unit at compile time.
template <int KVB>
__device__ __forceinline__ int hgu_shift(const KParams& p) {
  if constexpr (KVB == 4) return p.hgu_shift;
  else return 0;
}
template <int KVB>
__device__ __forceinline__ int slot_kv(const KParams& p, int kvb, int ks) {
  if constexpr (KVB == 4) return kvb * p.KVU + (ks >> p.hgu_shift);
  else return kvb * KVB + ks;
}
template <int KVB>
__device__ __forceinline__ int slot_hg(const KParams& p, int hg0, int ks) {
  if constexpr (KVB == 4) return hg0 + (ks & (p.HGU - 1));
  else return hg0;
}

// Row of out / lse ([B, T, Hq]) of virtual head h of head group hg of kv head kv.
template <int KIND>
__device__ __forceinline__ long long out_row(const KParams& p, int b, int kv, int hg, int h) {
  const int j = hg * kHeadTile + h;
  if constexpr (KIND != KIND_PAGED_MULTI) {
    return (long long)b * p.Hq + (long long)kv * p.G + j;  // one token
  } else {
    const int t = j / p.G, g = j - t * p.G;
    return ((long long)b * p.q_len + t) * p.Hq + (long long)kv * p.G + g;
  }
}

// Query row of q ([B, T, Hq, D]) for the same virtual head (the same index).
template <int KIND>
__device__ __forceinline__ long long q_row(const KParams& p, int b, int kv, int hg, int h) {
  return out_row<KIND>(p, b, kv, hg, h);
}

// Sequence whose tile positions contain g: the largest b with pre[b] <= g.
__device__ __forceinline__ int seq_of(const KParams& p, const int* pre, long long g) {
  int lo = 0, hi = p.B;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (pre[mid] <= g) lo = mid; else hi = mid;
  }
  return lo;
}

// STREAM order inside a CTA's range: when the range ends inside a unit that
// continues in the next CTA, that last segment goes first, then the rest in
// order.  Every unit cut between CTAs is then worked on at the start of its
// participants' ranges, so the partial states, tickets and the merge happen
// early, and a CTA's range ends with whole units (no cross-CTA work at the
// end of the kernel).
template <int KIND>
__device__ __forceinline__ void seg_init(const KParams& p, const PlanStore<KIND>& plan,
                                         const int* pre, SegIter& it) {
  it.n = 0;
  it.last0 = -1;
  if constexpr (KIND == KIND_PAGED_SPLIT) {
    it.g = 0;
    it.g_end = 1;
    return;
  }
  if (p.sched == SCHED_STREAM) {
    const long long T = pre[p.B];
    const int sg = stream_grid(p, T);
    if ((int)blockIdx.x >= sg) {
      it.g = it.g_end = it.s0 = it.fwd_end = 0;
      return;
    }
    it.g = it.s0 = stream_start(blockIdx.x, T, sg);
    it.g_end = it.fwd_end = stream_start(blockIdx.x + 1, T, sg);
    if (it.g_end > it.g) {
      const int b = seq_of(p, pre, it.g_end - 1);
      const int nt = plan.ntiles(b);
      const int off = (int)(it.g_end - 1 - pre[b]);
      const long long u0 = pre[b] + (long long)(off / nt * nt);  // unit start
      if (u0 > it.s0 && u0 + nt > it.g_end) {
        it.last0 = u0;
        it.fwd_end = u0;
      }
    }
  } else if (p.sched == SCHED_UNITS) {
    const long long U = (long long)p.B * units_per_seq(p);
    it.g = (long long)blockIdx.x * U / p.grid;
    it.g_end = (long long)(blockIdx.x + 1) * U / p.grid;
  } else {
    it.g = 0;
    it.g_end = 1;
  }
}

template <int KIND, int TOK>
__device__ __forceinline__ bool seg_next(const KParams& p, const PlanStore<KIND>& plan,
                                         const int* pre, SegIter& it, Seg& s) {
  const int upb = units_per_seq(p);
  if (KIND != KIND_PAGED_SPLIT && p.sched == SCHED_STREAM) {
    // the range's last segment first (see seg_init), then [s0, fwd_end)
    const bool last_first = it.last0 >= 0;
    const long long g = last_first ? it.last0 : it.g;
    const long long end = last_first ? it.g_end : it.fwd_end;
    if (g >= end) return false;
    const int b = seq_of(p, pre, g);
    const SeqPlan e = plan.get(b);
    const int nt = e.ntiles;
    const long long local = g - pre[b];
    const int li = (int)local;  // tile counts fit in int
    const int uib = li / nt;
    s.b = b;
    s.pidx = b;
    s.kvb = uib / p.HGN;
    s.hg = (uib % p.HGN) * p.HGU;
    s.unit = b * upb + uib;
    s.i0 = li - uib * nt;
    const long long rem = end - g;
    s.i1 = (int)((long long)s.i0 + rem < nt ? s.i0 + rem : nt);
    s.vlo = e.lo;
    s.vhi = e.hi;
    s.dest = (s.i0 == 0 && s.i1 == nt) ? DEST_OUT : DEST_PARTIAL;
    // partial slot: 0 for the segment at the start of the range, 1 for the
    // one at its end (the only two that can be partial)
    s.slot = g == it.s0 ? 0 : 1;
    if (last_first)
      it.last0 = -1;
    else
      it.g += s.i1 - s.i0;
    it.n++;
    return true;
  }
  if (KIND != KIND_PAGED_SPLIT && p.sched == SCHED_UNITS) {
    while (it.g < it.g_end) {
      const int u = (int)it.g++;
      const int b = u / upb;
      const SeqPlan e = plan.get(b);
      if (e.ntiles == 0) continue;
      const int uib = u % upb;
      s.b = b;
      s.pidx = b;
      s.kvb = uib / p.HGN;
      s.hg = (uib % p.HGN) * p.HGU;
      s.unit = u;
      s.i0 = 0;
      s.i1 = e.ntiles;
      s.vlo = e.lo;
      s.vhi = e.hi;
      s.dest = DEST_OUT;
      s.slot = 0;
      it.n++;
      return true;
    }
    return false;
  }
  // SCHED_SPLIT (its own kind): one segment, split blockIdx.x of unit blockIdx.y
  if constexpr (KIND != KIND_PAGED_SPLIT) return false;
  if (it.n > 0) return false;
  it.n = 1;
  const int u = blockIdx.y;
  const int b = u / upb;
  const int uib = u % upb;
  const SeqPlan e = plan.get(0);
  s.b = b;
  s.pidx = 0;
  s.kvb = uib / p.HGN;
  s.hg = (uib % p.HGN) * p.HGU;
  s.unit = u;
  s.dest = DEST_SPLIT;
  s.slot = blockIdx.x;
  const long long st0 = (long long)blockIdx.x * p.split_tokens;
  const long long st1 = st0 + p.split_tokens;
  long long vlo = e.lo > st0 ? e.lo : st0;
  long long vhi = e.hi < st1 ? e.hi : st1;
  s.i0 = s.i1 = 0;
  s.vlo = (int)vlo;
  s.vhi = (int)(vhi > vlo ? vhi : vlo);
  if (e.ntiles > 0 && vhi > vlo) {
    s.i0 = (int)(vlo / TOK) - e.t0;
    s.i1 = ceil_div_i(vhi, TOK) - e.t0;
  }
  return true;
}

// Flat index of the partial slot of participant c of a unit whose first
// tile is g0 (STREAM): slot 1 when the unit starts after c's range does
// (it is the segment at the end of c's range), else slot 0.
__device__ __forceinline__ int stream_slot(int c, int c0, long long g0, long long T, int grid) {
  const int j = (c == c0 && stream_start(c, T, grid) < g0) ? 1 : 0;
  return c * 2 + j;
}

// Block-sparse kind: the sequence's area of `words` words (sparse_words).
__device__ __forceinline__ const uint32_t* sparse_area(const uint32_t* sp_base, const KParams& p,
                                                       int b) {
  return sp_base + (size_t)b * p.sp_words;
}

// Tile of the i-th set bit of a sequence's tile bitmask: the last word
// whose count of earlier set bits is <= i holds it.
__device__ __forceinline__ int sparse_select(const uint32_t* area, int tw, int i) {
  const uint32_t* pc = area + tw;
  int lo = 0, hi = tw;  // pc[lo] <= i
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int)pc[mid] <= i) lo = mid; else hi = mid;
  }
  const int bit = (int)__fns(area[lo], 0u, i - (int)pc[lo] + 1);
  return 32 * lo + bit;
}

// The tiles of a segment of the block-sparse kind in order: the i0-th set
// bit of the sequence's tile bitmask (a select), then each following set bit
// (the lowest remaining bit of the current word, or of the next non-zero
// word).  A segment asks for no more tiles than the bitmask has bits.
struct SparseTiles {
  const uint32_t* words;
  int w;
  uint32_t rest;  // bits of word w after the last tile returned
  int first;
  __device__ __forceinline__ void init(const uint32_t* area, int tw, int i0) {
    first = sparse_select(area, tw, i0);
    words = area;
    w = first >> 5;
    rest = area[w] & ~((2u << (first & 31)) - 1u);
  }
  __device__ __forceinline__ int next() {
    while (rest == 0u) rest = words[++w];
    const int t = 32 * w + __ffs(rest) - 1;
    rest &= rest - 1u;
    return t;
  }
};

// Absolute tile of unit-local tile i (tiered: hot tiles follow cold ones).
template <int KIND>
__device__ __forceinline__ int tile_of(const SeqPlan& e, int i, bool& is_hot) {
  if (is_tiered(KIND) && i >= e.ncold) {
    is_hot = true;
    const int hi_ = i - e.ncold;
    const int na = e.ha1 - e.ha0;
    return hi_ < na ? e.ha0 + hi_ : e.hb0 + (hi_ - na);
  }
  is_hot = false;
  return e.t0 + i;
}

// Rows of one TMA box of a paged / cold tile and its page split.
struct BoxGeo {
  int R;         // rows (keys) per box: min(block_size, TOK)
  int log2R;
  int npg;       // boxes (pages) per tile
  int box_bytes; // bytes of one box (KVB heads x all slices x R rows)
};

// ============================================================== producer
template <int KIND, int D, int KVB>
__device__ __forceinline__ void producer_loop(const KParams& p, const PlanStore<KIND>& plan,
                                              const int* pre, uint8_t* stages, uint8_t* hdrs,
                                              uint8_t* qslot, const SmemLayout& L,
                                              const BoxGeo& bg, uint64_t* full, uint64_t* empty,
                                              uint64_t* qfull, uint64_t* qempty, Misc* misc,
                                              const uint32_t* sp_base) {
  using Gm = Geo<KIND, D, KVB>;
  constexpr int OPS = cold_int8(KIND) ? 4 : 2;  // copies per page: K, V (+ 2 scale slabs)
  const int lane = threadIdx.x & 31;
  const int nstages = p.stages;
  const int bs = p.bs, log2_bs = p.log2_bs, max_blocks = p.max_blocks, nblocks = p.num_blocks;
  const int Hkv = p.Hkv;
  const uint32_t page_bytes =
      (uint32_t)(2 * bg.box_bytes + (cold_int8(KIND) ? 2 * bg.R * Hkv * 2 : 0));
  SegIter it;
  seg_init<KIND>(p, plan, pre, it);
  Seg s;
  int stage = 0;
  uint32_t round = 0;
  int qn = 0;  // non-empty segments so far (Q slot phase)
  // stages (bit j) holding an issued copy, and the phase parity it completes
  uint32_t iss_mask = 0, iss_par = 0;
  bool q_iss = false;
  uint32_t q_par = 0;
  int bt_b = -1, bt_base = 0, bt_cur = -1, bt_nxt = -1;
  int flags = 0;
  // The f16 pages are read once: their L2 lines go first (measured: the
  // paged and long-context steps 1-2% faster).  The tiered kernels measured
  // slower with the hinted copies and keep the plain ones.
  const uint64_t stream_pol = is_paged(KIND) ? l2_evict_first_policy() : 0ull;
  while (seg_next<KIND, Gm::TOK>(p, plan, pre, it, s)) {
    if (s.i0 >= s.i1) continue;
    const SeqPlan e = plan.get(s.pidx);
    const int kv0 = s.kvb * (KVB >> hgu_shift<KVB>(p));  // first kv head of the unit's boxes
    const int* bt_row = p.block_table + (long long)s.b * max_blocks;
    // ---- Q rows of the unit (KVB slots x NH heads) into the Q slot
    {
      if (!mbar_wait(qempty, (qn & 1) ^ 1, abort_flag(misc), p.wait_ns) && lane == 0) note_abort(misc);
      const bool live = !__any_sync(0xffffffffu, *abort_flag(misc) != 0);
      if (live) {
        q_iss = true;
        q_par = qn & 1;
      }
      if (lane == 0 && live) {
        // slot layout [KVB][NH][D]; slot j takes the nh rows of its
        // (kv head, head group)
        const uint32_t row = (uint32_t)(D * 4);
        const uint32_t per = (uint32_t)p.NH * row;
        if (KIND != KIND_PAGED_MULTI && p.HG == 1) {
          // one token, one group: the unit's KVB x G rows are contiguous
          const int nh = unit_nh(p, 0);
          mbar_arrive_expect_tx(qfull, (uint32_t)(nh * KVB) * row);
          bulk_load(qslot, p.q + q_row<KIND>(p, s.b, kv0, 0, 0) * D, (uint32_t)(nh * KVB) * row, qfull);
        } else {
          int rows = 0;
          for (int j = 0; j < KVB; ++j) rows += unit_nh(p, slot_hg<KVB>(p, s.hg, j));
          mbar_arrive_expect_tx(qfull, (uint32_t)rows * row);
          for (int j = 0; j < KVB; ++j) {
            const int kv = slot_kv<KVB>(p, s.kvb, j), hg = slot_hg<KVB>(p, s.hg, j);
            const int nh = unit_nh(p, hg);
            if (KIND != KIND_PAGED_MULTI) {
              bulk_load(qslot + j * per, p.q + q_row<KIND>(p, s.b, kv, hg, 0) * D,
                        (uint32_t)nh * row, qfull);
            } else {
              // several tokens: rows of different tokens are Hq rows apart
              for (int h = 0; h < nh; ++h)
                bulk_load(qslot + j * per + h * row, p.q + q_row<KIND>(p, s.b, kv, hg, h) * D, row,
                          qfull);
            }
          }
        }
      }
      ++qn;
    }
    SparseTiles spt;
    if constexpr (KIND == KIND_PAGED_SPARSE) spt.init(sparse_area(sp_base, p, s.pidx), p.sp_tw, s.i0);
    for (int i = s.i0; i < s.i1; ++i) {
      if (!mbar_wait(&empty[stage], (round & 1) ^ 1, abort_flag(misc), p.wait_ns) && lane == 0)
        note_abort(misc);
      uint8_t* st = stages + (size_t)stage * L.stage_bytes;
      bool is_hot = false;
      int at;
      if constexpr (KIND == KIND_PAGED_SPARSE) at = i == s.i0 ? spt.first : spt.next();
      else at = tile_of<KIND>(e, i, is_hot);
      if (__any_sync(0xffffffffu, *abort_flag(misc) != 0) ||
          (p.test_skip_arm && blockIdx.x == 0 && iss_mask == 0)) {
        // abort mode (or the test knob): no copy, the stage stays unarmed
      } else if (!is_hot) {
        // ----- pages through the block table
        const int tok0 = at * Gm::TOK;
        const int p_first = tok0 >> log2_bs;
        const int row_off = (bs > Gm::TOK) ? (tok0 & (bs - 1)) : 0;
        // keep a 64-entry window of block-table entries in two registers
        if (s.b != bt_b || p_first < bt_base || p_first + bg.npg > bt_base + 64) {
          if (s.b == bt_b && p_first >= bt_base + 32 && p_first + bg.npg <= bt_base + 96) {
            bt_cur = bt_nxt;
            bt_base += 32;
          } else {
            bt_base = p_first;
            const int pc = bt_base + lane;
            bt_cur = pc < max_blocks ? __ldg(bt_row + pc) : -1;
          }
          const int pn = bt_base + 32 + lane;
          bt_nxt = pn < max_blocks ? __ldg(bt_row + pn) : -1;
          bt_b = s.b;
        }
        // lane j < npg: page j of the tile
        const int idx = p_first + lane - bt_base;
        const int vc = __shfl_sync(0xffffffffu, bt_cur, idx & 31);
        const int vn = __shfl_sync(0xffffffffu, bt_nxt, idx & 31);
        const int pg = p_first + lane;
        const int blk = (lane < bg.npg && pg < max_blocks) ? (idx < 32 ? vc : vn) : -1;
        const int vhi_keys = is_tiered(KIND) ? min(s.vhi, e.cold_len) : s.vhi;
        const int r0 = tok0 + lane * bg.R;
        const bool needed = lane < bg.npg && (r0 < vhi_keys) && (r0 + bg.R > s.vlo);
        const bool ok = needed && blk >= 0 && blk < nblocks;
        const uint32_t need_mask = __ballot_sync(0xffffffffu, ok);
        const uint32_t bad_mask = __ballot_sync(0xffffffffu, needed && !ok);
        if (bad_mask) flags |= DEV_BAD_BLOCK;
        if (lane == 0) {
          *reinterpret_cast<volatile uint32_t*>(hdrs + stage * 16) = bad_mask;
          mbar_arrive_expect_tx(&full[stage], (uint32_t)__popc(need_mask) * page_bytes);
        }
        __syncwarp();
        iss_mask |= 1u << stage;
        iss_par = (iss_par & ~(1u << stage)) | ((round & 1u) << stage);
        for (int base = 0; base < bg.npg * OPS; base += 32) {
          const int op = base + lane;
          const int j = op / OPS;
          const int bj = __shfl_sync(0xffffffffu, blk, j & 31);
          if (op < bg.npg * OPS && ((need_mask >> j) & 1u)) {
            const int r = op % OPS;
            const int row = bj * bs + row_off;
            if (r < 2) {
              uint8_t* dst = st + (r ? L.off_v : L.off_k) + j * bg.box_bytes;
              if constexpr (is_paged(KIND))
                tma_load_4d_hint(dst, r ? &p.tm_v : &p.tm_k, &full[stage], 0, row, 0, kv0,
                                 stream_pol);
              else
                tma_load_4d(dst, r ? &p.tm_v : &p.tm_k, &full[stage], 0, row, 0, kv0);
            } else if constexpr (cold_int8(KIND)) {
              // the box's rows of the page's [rows, Hkv] f16 scale slab
              const int isv = r - 2;
              const uint16_t* src = (isv ? p.v_scale : p.k_scale) + (long long)row * Hkv;
              uint8_t* dst = st + L.off_sc + isv * (Gm::TOK * Hkv * 2) + j * bg.R * Hkv * 2;
              bulk_load(dst, src, (uint32_t)(bg.R * Hkv * 2), &full[stage]);
            }
          }
        }
      } else if constexpr (is_tiered(KIND)) {
        // ----- hot ring tile: slots [at*TOKH, at*TOKH + TOKH) of sequence b
        if (lane == 0) {
          *reinterpret_cast<volatile uint32_t*>(hdrs + stage * 16) = 0u;
          mbar_arrive_expect_tx(&full[stage], (uint32_t)(2 * (Gm::REGION >> hgu_shift<KVB>(p))));
        }
        __syncwarp();
        iss_mask |= 1u << stage;
        iss_par = (iss_par & ~(1u << stage)) | ((round & 1u) << stage);
        if (lane < 2) {
          uint8_t* dst = st + (lane ? L.off_v : L.off_k);
          tma_load_5d(dst, lane ? &p.tm_vh : &p.tm_kh, &full[stage], 0, at * Gm::TOKH, 0, kv0,
                      s.b + p.hot_b0);
        }
      }
      if (++stage == nstages) {
        stage = 0;
        ++round;
      }
    }
  }
  // No copy may still be in flight when the CTA exits: wait (bounded, and
  // also in abort mode) for the last one issued into each stage and the Q slot.
  for (int j = 0; j < nstages; ++j)
    if (((iss_mask >> j) & 1u) && !mbar_wait_lazy(&full[j], (iss_par >> j) & 1u, p.wait_ns))
      flags |= DEV_TIMEOUT;
  if (q_iss && !mbar_wait_lazy(qfull, q_par, p.wait_ns)) flags |= DEV_TIMEOUT;
  if (flags && lane == 0) atomicOr(&misc->flags, flags);
}

// ============================================================== consumer
template <int D>
struct Acc {
  float o[D / 16][4];  // O^T fragments: (d row r (+8) of m-tile mt, head 2c (+1))
  float m[2], l[2];    // heads 2c, 2c+1 (base-2 units)
};

// Q^T B fragments.  Unpacked: hi and lo parts as two operands (one MMA
// each).  Packed (at most four heads per kv head): hi holds columns 0-3 =
// f16 part of heads 0-3 and columns 4-7 = remainder of the same heads, so
// one MMA yields both parts of every score; lo is unused.
template <int D>
struct QFrag {
  uint32_t hi[D / 16][2], lo[D / 16][2];
};

// Head-dimension index held by accumulator row r (+8 when hi8) of m-tile mt:
// every V load (f16 and int8 transposed fragments) keeps the natural order.
template <int KIND>
__device__ __forceinline__ int o_row_d(int mt, int r, int hi8) {
  return 16 * mt + r + 8 * hi8;
}

// Q rows of the head group, prescaled (scale*log2 e), as hi/lo f16 B
// fragments.  Natural order: k-step ks covers d = 16ks + {2c, 2c+1} and
// {2c+8, 2c+9}; permuted order (tiered): d = 16ks + 4c + {0, 1} and {2, 3}.
template <int KIND, int D, bool PK>
__device__ __forceinline__ void load_q(uint32_t qs, int NH, float qscale, int r, int c,
                                       QFrag<D>& q) {
  const int hq = PK ? (r & 3) : r;  // head of B column r
  const bool hv = hq < NH;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    int d0, d2;
    if constexpr (!cold_int8(KIND)) {
      d0 = 16 * ks + 2 * c;
      d2 = d0 + 8;
    } else {
      // tiered d order: k-steps 2j and 2j + 1 take, from lane c, the 8
      // consecutive values d = 32j + 8c .. + 7 of a key (4 each)
      d0 = 32 * (ks >> 1) + 8 * c + 4 * (ks & 1);
      d2 = d0 + 2;
    }
    float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
    if (hv) {
      const uint32_t row = qs + (uint32_t)(hq * D) * 4u;
      const uint2 a = lds64(row + d0 * 4);
      const uint2 b = lds64(row + d2 * 4);
      x0 = __uint_as_float(a.x) * qscale;
      x1 = __uint_as_float(a.y) * qscale;
      x2 = __uint_as_float(b.x) * qscale;
      x3 = __uint_as_float(b.y) * qscale;
    }
    split_half2(x0, x1, q.hi[ks][0], q.lo[ks][0]);
    split_half2(x2, x3, q.hi[ks][1], q.lo[ks][1]);
    if constexpr (PK) {
      if (r >= 4) {
        q.hi[ks][0] = q.lo[ks][0];
        q.hi[ks][1] = q.lo[ks][1];
      }
    }
  }
}

// Two signed bytes of a word already biased by 0x80 (so byte = x + 128) to
// an exact f16x2 pair: 0x64XX is 1024 + XX as f16, minus 1152 gives x.
// `sel` picks the bytes (0x4140: bytes 0,1; 0x4342: bytes 2,3).
__device__ __forceinline__ uint32_t biased_i8x2_to_h2(uint32_t wb, uint32_t sel) {
  uint32_t t = __byte_perm(wb, 0x64646464u, sel);
  __half2 h = *reinterpret_cast<__half2*>(&t);
  h = __hsub2(h, __half2half2(__ushort_as_half((unsigned short)0x6480u)));  // 1152
  return *reinterpret_cast<uint32_t*>(&h);
}

// Where the rows of one kv head live in a stage.  Row of key k:
//   base + (k >> log2R) * box_bytes + (k & (R-1)) * 128, slice ch adds
//   ch * R * 128, and 16-byte unit u of a slice sits at (u ^ (k & 7)) * 16.
struct RowMap {
  uint32_t base;  // stage region + kv-head offset inside a box
  int log2R;
  int box_bytes;
  int cstride;    // R * 128
  __device__ __forceinline__ uint32_t row(int k) const {
    return base + (uint32_t)((k >> log2R) * box_bytes + (k & ((1 << log2R) - 1)) * 128);
  }
};

// S^T[16 keys x 8 heads] of keys k0..k0+15 into NCH accumulators (summed
// by the caller): unpacked, half take the hi Q part and half the lo part;
// packed, k-step ks goes to accumulator ks mod NCH.  Several accumulators
// keep the MMA dependency chains short.
template <int TK, int D, bool PK, int NCH>
__device__ __forceinline__ void qk_mma(float (&s4)[NCH][4], int ks, uint32_t a0, uint32_t a1,
                                       uint32_t a2, uint32_t a3, const QFrag<D>& q) {
  if constexpr (PK) {
    mma_f16_16816(s4[ks % NCH], a0, a1, a2, a3, q.hi[ks][0], q.hi[ks][1]);
  } else {
    constexpr int H = NCH / 2;
    mma_f16_16816(s4[ks % H], a0, a1, a2, a3, q.hi[ks][0], q.hi[ks][1]);
    mma_f16_16816(s4[H + ks % H], a0, a1, a2, a3, q.lo[ks][0], q.lo[ks][1]);
  }
}

template <int TK, int D, bool PK, int NCH>
__device__ __forceinline__ void tile_qk(const RowMap& km, int k0, int lane, const QFrag<D>& q,
                                        float (&s4)[NCH][4]) {
  const int r = lane >> 2, c = lane & 3;
  if constexpr (TK == TK_PAGED) {
    const int mat = lane >> 3;
    const int key = k0 + (lane & 7) + ((mat & 1) << 3);
    const uint32_t rowaddr = km.row(key);
    const int x = lane & 7;
    const int dh = mat >> 1;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int ug = 2 * ks + dh;
      uint32_t a0, a1, a2, a3;
      ldsm_x4(rowaddr + (ug >> 3) * km.cstride + (((ug & 7) ^ x) << 4), a0, a1, a2, a3);
      qk_mma<TK, D, PK, NCH>(s4, ks, a0, a1, a2, a3, q);
    }
  } else if constexpr (TK == TK_COLD) {
    // int8 rows of D bytes; k-steps 2j and 2j + 1 take the 8 bytes
    // d = 32j + 8c .. + 7 of rows r and r + 8 (one 8-byte load each): the
    // 16-byte unit (2j + (c >> 1)) & 7 of slice j >> 2, at byte 8 (c & 1).
    // Rows start on 128-byte boundaries, so the swizzled unit is set with an
    // xor on a per-tile base.
    const uint32_t lb = (uint32_t)(8 * (c & 1)) | (uint32_t)((((c >> 1) ^ r) & 7) << 4);
    const uint32_t x0 = km.row(k0 + r) | lb;
    const uint32_t x1 = km.row(k0 + r + 8) | lb;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
      const uint32_t cs = (j >> 2) * km.cstride;
      const uint32_t sw = (uint32_t)(((2 * j) & 7) << 4);
      const uint2 w0 = lds64((x0 + cs) ^ sw);
      const uint2 w1 = lds64((x1 + cs) ^ sw);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint32_t u0 = (t ? w0.y : w0.x) ^ 0x80808080u;
        const uint32_t u1 = (t ? w1.y : w1.x) ^ 0x80808080u;
        const uint32_t a0 = biased_i8x2_to_h2(u0, 0x4140u), a2 = biased_i8x2_to_h2(u0, 0x4342u);
        const uint32_t a1 = biased_i8x2_to_h2(u1, 0x4140u), a3 = biased_i8x2_to_h2(u1, 0x4342u);
        qk_mma<TK, D, PK, NCH>(s4, 2 * j + t, a0, a1, a2, a3, q);
      }
    }
  } else {
    // f16 rows; k-steps 2j and 2j + 1 take the 8 values d = 32j + 8c .. + 7
    // of rows r and r + 8 (one 16-byte load each): unit (4j + c) & 7 of
    // slice j >> 1
    const uint32_t lb = (uint32_t)(((c ^ r) & 7) << 4);
    const uint32_t x0 = km.row(k0 + r) | lb;
    const uint32_t x1 = km.row(k0 + r + 8) | lb;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
      const uint32_t cs = (j >> 1) * km.cstride;
      const uint32_t sw = (uint32_t)(((4 * j) & 7) << 4);
      const uint4 v0 = lds128((x0 + cs) ^ sw);
      const uint4 v1 = lds128((x1 + cs) ^ sw);
      qk_mma<TK, D, PK, NCH>(s4, 2 * j, v0.x, v1.x, v0.y, v1.y, q);
      qk_mma<TK, D, PK, NCH>(s4, 2 * j + 1, v0.z, v1.z, v0.w, v1.w, q);
    }
  }
}

// One m-tile of O^T += V^T P^T: hi then lo P parts, or the packed operand
// alone (columns 0-3 f16 part, 4-7 remainder).
template <bool PK>
__device__ __forceinline__ void pv_mma(float (&o)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t bh0, uint32_t bh1, uint32_t bl0,
                                       uint32_t bl1) {
  mma_f16_16816(o, a0, a1, a2, a3, bh0, bh1);
  if constexpr (!PK) mma_f16_16816(o, a0, a1, a2, a3, bl0, bl1);
}

// O^T += V^T P^T for keys k0..k0+15; b* are the P^T fragments.
template <int TK, int D, bool PK>
__device__ __forceinline__ void tile_pv(const RowMap& vm, int k0, int lane, float (&o)[D / 16][4],
                                        uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
  if constexpr (TK == TK_PAGED || TK == TK_HOT) {
    // f16 rows: 8x8 transposed fragments (d rows of m-tile mt, keys k0 ..)
    const int mat = lane >> 3;
    const int key = k0 + (lane & 7) + ((mat >> 1) << 3);
    const uint32_t rowaddr = vm.row(key);
    const int x = lane & 7;
    const int dh = mat & 1;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      const int ug = 2 * mt + dh;
      uint32_t a0, a1, a2, a3;
      ldsm_x4_trans(rowaddr + (ug >> 3) * vm.cstride + (((ug & 7) ^ x) << 4), a0, a1, a2, a3);
      pv_mma<PK>(o[mt], a0, a1, a2, a3, bh0, bh1, bl0, bl1);
    }
  } else {
    // int8 rows: 16 keys x 16 d bytes per transposed 8-bit load, two m-tiles
    // at once.  Lane (r, c) gets keys k0+4c .. k0+4c+3 at d = 16 mt + r and
    // + 8, so the MMA's k index 2c + j (+8) stands for key 4c + j (+2); the
    // caller orders P^T the same way.  Lane l gives the address of row l & 15
    // of m-tile 2 mp + (l >> 4): unit (mt & 7) ^ (key & 7) of slice mt >> 3,
    // split into a per-lane part and an xor by 2 mp & 7 (rows on 128-byte
    // boundaries).
    const int j = lane & 15;
    const uint32_t xb = vm.row(k0 + j) | ((uint32_t)(((lane >> 4) ^ j) & 7) << 4);
#pragma unroll
    for (int mp = 0; mp < D / 32; ++mp) {
      const uint32_t addr = (xb + (mp >> 2) * vm.cstride) ^ ((uint32_t)((2 * mp) & 7) << 4);
      uint32_t w[4];
      ldsm_b8_x2_trans(addr, w[0], w[1], w[2], w[3]);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint32_t u0 = w[2 * m] ^ 0x80808080u, u1 = w[2 * m + 1] ^ 0x80808080u;
        const uint32_t a0 = biased_i8x2_to_h2(u0, 0x4140u), a1 = biased_i8x2_to_h2(u1, 0x4140u);
        const uint32_t a2 = biased_i8x2_to_h2(u0, 0x4342u), a3 = biased_i8x2_to_h2(u1, 0x4342u);
        pv_mma<PK>(o[2 * mp + m], a0, a1, a2, a3, bh0, bh1, bl0, bl1);
      }
    }
  }
}

// P^T fragments for the int8 V loads: the natural B fragments hold keys
// (2c, 2c+1) in b0 and (2c+8, 2c+9) in b1; lane (r, c) takes keys (4c, 4c+1)
// and (4c+2, 4c+3) instead, from lanes 2c and 2c + 1 (mod 4) of its quad:
// their b0 for c < 2, their b1 for c >= 2.
__device__ __forceinline__ void key_order_4c(int lane, uint32_t& b0, uint32_t& b1) {
  const int q = lane & ~3, c = lane & 3;
  const int s0 = q | ((2 * c) & 3), s1 = q | ((2 * c + 1) & 3);
  const uint32_t t0 = __shfl_sync(0xffffffffu, b0, s0), t1 = __shfl_sync(0xffffffffu, b1, s0);
  const uint32_t t2 = __shfl_sync(0xffffffffu, b0, s1), t3 = __shfl_sync(0xffffffffu, b1, s1);
  b0 = c < 2 ? t0 : t1;
  b1 = c < 2 ? t2 : t3;
}

// Per-column masks of a multi-token query: the lane's two score columns
// belong to query tokens whose own causal / window bounds [lo, hi) cut the
// keys (absolute position kbase + tile key index).
struct ColMask {
  bool on;
  int kbase;
  int lo[2], hi[2];
};

// Softcap in base-2 score units: cap2 * tanh(y), y = x / cap2, cap2 = cap *
// log2(e).  tanh comes from the identity tanh(y) = 1 - 2 / (e^(2y) + 1),
// e^(2y) = 2^(2 log2(e) y): one exp2 and one approximate division.  Its
// absolute error, about 3e-7 (the rounding of e^(2y) next to 1), becomes
// 3e-7 * cap2 in the score: at most 3e-5 up to cap2 = 100, and the form
// saturates to +-1 without overflow and keeps NaN.  Above cap2 = 100, where
// that error would grow with the cap, |y| <= 1/2 takes the Taylor series of
// tanh about 0 instead (coefficients 2^2n (2^2n - 1) B_2n / (2n)! from the
// Bernoulli numbers, through y^13: the first omitted term is below 1e-7 of
// tanh(y) at |y| = 1/2), whose error is relative to y; beyond |y| = 1/2 the
// identity's 3e-7 is below 1e-6 of tanh(y).  The cap is uniform across a
// launch, so the branch is too.
constexpr float kSoftcapSeriesAbove = 100.f;

__device__ __forceinline__ float tanh_series(float y) {
  const float y2 = y * y;
  float t = 21844.f / 6081075.f;
  t = fmaf(t, y2, -1382.f / 155925.f);
  t = fmaf(t, y2, 62.f / 2835.f);
  t = fmaf(t, y2, -17.f / 315.f);
  t = fmaf(t, y2, 2.f / 15.f);
  t = fmaf(t, y2, -1.f / 3.f);
  return fmaf(t * y2, y, y);
}

__device__ __forceinline__ float softcap_b2(float x, float cap2, float inv_cap2) {
  const float y = x * inv_cap2;
  float t = 1.f - __fdividef(2.f, ex2_ftz(y * 2.8853900817779268f) + 1.f);
  if (cap2 > kSoftcapSeriesAbove && fabsf(y) <= 0.5f) t = tanh_series(y);
  return cap2 * t;
}

// NG 16-key groups of this warp (keys k0[g] .. k0[g]+15) in one online-
// softmax step: the QK products, one running-max update, then the PV
// products.  v[2g], v[2g+1]: validity of keys k0[g]+r and k0[g]+r+8;
// ks / vs: their K and V scales in the int8 tier (1 otherwise).  Taking two
// groups at once halves the serial max/rescale work per key and gives the
// warp two independent QK chains to interleave.
template <int TK, int D, bool PK, int NG>
__device__ __forceinline__ void groups_compute(const RowMap& km, const RowMap& vm,
                                               float2 cap, const int (&k0)[NG], int lane,
                                               const QFrag<D>& q, Acc<D>& a,
                                               const bool (&v)[2 * NG],
                                               const float (&ks)[2 * NG],
                                               const float (&vs)[2 * NG],
                                               const ColMask& cm) {
  constexpr int NCH = NG == 1 ? 4 : 2;
  float s4[NG][NCH][4];
#pragma unroll
  for (int g = 0; g < NG; ++g)
#pragma unroll
    for (int i = 0; i < NCH; ++i) s4[g][i][0] = s4[g][i][1] = s4[g][i][2] = s4[g][i][3] = 0.f;
#pragma unroll
  for (int g = 0; g < NG; ++g) tile_qk<TK, D, PK, NCH>(km, k0[g], lane, q, s4[g]);
  float sc[NG][4];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float x = s4[g][0][j];
#pragma unroll
      for (int i = 1; i < NCH; ++i) x += s4[g][i][j];
      // packed: column h + 4 (lane c ^ 2) holds the remainder part of head h
      if constexpr (PK) x += __shfl_xor_sync(0xffffffffu, x, 2);
      if constexpr (TK == TK_COLD) x *= ks[2 * g + (j >> 1)];
      if (cap.x > 0.f) x = softcap_b2(x, cap.x, cap.y);
      sc[g][j] = x;
    }
    if (!v[2 * g]) sc[g][0] = sc[g][1] = kNegInf;
    if (!v[2 * g + 1]) sc[g][2] = sc[g][3] = kNegInf;
    if (cm.on) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = cm.kbase + k0[g] + (lane >> 2) + 8 * (j >> 1);
        if (key < cm.lo[j & 1] || key >= cm.hi[j & 1]) sc[g][j] = kNegInf;
      }
    }
  }
  // ---- online softmax (base 2)
  float mx0 = fmaxf(sc[0][0], sc[0][2]), mx1 = fmaxf(sc[0][1], sc[0][3]);
#pragma unroll
  for (int g = 1; g < NG; ++g) {
    mx0 = fmaxf(mx0, fmaxf(sc[g][0], sc[g][2]));
    mx1 = fmaxf(mx1, fmaxf(sc[g][1], sc[g][3]));
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const float mn0 = fmaxf(a.m[0], mx0), mn1 = fmaxf(a.m[1], mx1);
  const float al0 = (mn0 == kNegInf) ? 1.f : ex2_ftz(a.m[0] - mn0);
  const float al1 = (mn1 == kNegInf) ? 1.f : ex2_ftz(a.m[1] - mn1);
  const float mu0 = (mn0 == kNegInf) ? 0.f : mn0;
  const float mu1 = (mn1 == kNegInf) ? 0.f : mn1;
  float pr[NG][4];
  float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    pr[g][0] = ex2_ftz(sc[g][0] - mu0);
    pr[g][1] = ex2_ftz(sc[g][1] - mu1);
    pr[g][2] = ex2_ftz(sc[g][2] - mu0);
    pr[g][3] = ex2_ftz(sc[g][3] - mu1);
    ls0 += pr[g][0] + pr[g][2];
    ls1 += pr[g][1] + pr[g][3];
  }
  a.l[0] = a.l[0] * al0 + ls0;
  a.l[1] = a.l[1] * al1 + ls1;
  a.m[0] = mn0;
  a.m[1] = mn1;
  if (!__all_sync(0xffffffffu, al0 == 1.f && al1 == 1.f)) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      a.o[mt][0] *= al0;
      a.o[mt][1] *= al1;
      a.o[mt][2] *= al0;
      a.o[mt][3] *= al1;
    }
  }
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    float p0 = pr[g][0], p1 = pr[g][1], p2 = pr[g][2], p3 = pr[g][3];
    if constexpr (TK == TK_COLD) {
      // the V scale of each key folds into its weight (masked keys: exactly 0)
      p0 = v[2 * g] ? p0 * vs[2 * g] : 0.f;
      p1 = v[2 * g] ? p1 * vs[2 * g] : 0.f;
      p2 = v[2 * g + 1] ? p2 * vs[2 * g + 1] : 0.f;
      p3 = v[2 * g + 1] ? p3 * vs[2 * g + 1] : 0.f;
    }
    // ---- P^T as the B operand (hi + lo), via an 8x8 transpose
    uint32_t h01, l01, h23, l23;
    split_half2(p0, p1, h01, l01);
    split_half2(p2, p3, h23, l23);
    if constexpr (PK) {
      // lanes c < 2 give columns 0-3 (f16 parts), lanes c >= 2 columns 4-7
      const bool lo_cols = (lane & 2) != 0;
      uint32_t b0 = movmatrix_trans(lo_cols ? l01 : h01);
      uint32_t b1 = movmatrix_trans(lo_cols ? l23 : h23);
      if constexpr (TK == TK_COLD) key_order_4c(lane, b0, b1);
      tile_pv<TK, D, PK>(vm, k0[g], lane, a.o, b0, b1, 0u, 0u);
    } else {
      uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
      uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);
      if constexpr (TK == TK_COLD) {
        key_order_4c(lane, bh0, bh1);
        key_order_4c(lane, bl0, bl1);
      }
      tile_pv<TK, D, PK>(vm, k0[g], lane, a.o, bh0, bh1, bl0, bl1);
    }
  }
}

// One 16-key group (keys k0 .. k0+15) of an f16 tile.
template <int TK, int D, bool PK>
__device__ __forceinline__ void group_compute(const RowMap& km, const RowMap& vm, float2 cap,
                                              int k0, int lane, const QFrag<D>& q, Acc<D>& a,
                                              bool vA, bool vB, const ColMask& cm) {
  const int k0s[1] = {k0};
  const bool v[2] = {vA, vB};
  const float one[2] = {1.f, 1.f};
  groups_compute<TK, D, PK, 1>(km, vm, cap, k0s, lane, q, a, v, one, one, cm);
}

// Zeroes the f16 V rows of masked keys among k0..k0+15 of this warp's head,
// so that a zero weight never meets a stale or non-finite value.
template <int D, typename OkFn>
__device__ __forceinline__ void zero_masked_v_rows(const RowMap& vm, int k0, int lane, OkFn ok) {
  constexpr int UPR = D / 8;  // 16-byte units per f16 row
  for (int u = lane; u < 16 * UPR; u += 32) {
    const int row = u / UPR, ug = u % UPR;
    const int k = k0 + row;
    if (!ok(k)) sts128_zero(vm.row(k) + (ug >> 3) * vm.cstride + (((ug & 7) ^ (k & 7)) << 4));
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// What a hot-ring tile can see: ring slot s holds hot key
// j = (s - hot_start) mod W (or j = s without a ring), visible when
// j0 <= j < j1.
struct HotView {
  int W, cap_eff, hs_mod;
  long long j0, j1;
};

__device__ __forceinline__ bool key_ok_hot(const HotView& hv, int slot0, int k) {
  const int sl = slot0 + k;
  if (sl >= hv.cap_eff) return false;
  const int j = hv.W > 0 ? (sl - hv.hs_mod + hv.W) % hv.W : sl;
  return j >= hv.j0 && j < hv.j1;
}

// The tree merge goes through shared memory in RP parts of the O
// fragments (m-tiles [part * MP, part * MP + MP), MP = D / 16 / RP); part 0
// also carries m and l and fixes the two weights of the merge, which later
// parts reuse.  A slot holds red_floats(D, RP) floats per lane set.
struct MergeW {
  float fa0, fb0, fa1, fb1;
};

// Combines two online-softmax states of the same heads (this warp's and a
// partner's, read back from shared memory in the same fragment layout).
template <int D, int RP>
__device__ __forceinline__ void merge_state(Acc<D>& a, const float* red, int lane, int part,
                                            MergeW& w) {
  constexpr int MP = D / 16 / RP;
  constexpr int NO = 4 * MP;
  if (part == 0) {
    const float mb0 = red[(NO + 0) * 32 + lane], mb1 = red[(NO + 1) * 32 + lane];
    const float lb0 = red[(NO + 2) * 32 + lane], lb1 = red[(NO + 3) * 32 + lane];
    const float mn0 = fmaxf(a.m[0], mb0), mn1 = fmaxf(a.m[1], mb1);
    w.fa0 = (a.m[0] == kNegInf) ? 0.f : exp2f(a.m[0] - mn0);
    w.fb0 = (mb0 == kNegInf) ? 0.f : exp2f(mb0 - mn0);
    w.fa1 = (a.m[1] == kNegInf) ? 0.f : exp2f(a.m[1] - mn1);
    w.fb1 = (mb1 == kNegInf) ? 0.f : exp2f(mb1 - mn1);
    a.l[0] = a.l[0] * w.fa0 + lb0 * w.fb0;
    a.l[1] = a.l[1] * w.fa1 + lb1 * w.fb1;
    a.m[0] = mn0;
    a.m[1] = mn1;
  }
#pragma unroll
  for (int q = 0; q < RP; ++q) {
    if (q != part) continue;
#pragma unroll
    for (int i = 0; i < MP; ++i) {
      const int mt = q * MP + i;
      a.o[mt][0] = a.o[mt][0] * w.fa0 + red[(4 * i + 0) * 32 + lane] * w.fb0;
      a.o[mt][1] = a.o[mt][1] * w.fa1 + red[(4 * i + 1) * 32 + lane] * w.fb1;
      a.o[mt][2] = a.o[mt][2] * w.fa0 + red[(4 * i + 2) * 32 + lane] * w.fb0;
      a.o[mt][3] = a.o[mt][3] * w.fa1 + red[(4 * i + 3) * 32 + lane] * w.fb1;
    }
  }
}

template <int D, int RP>
__device__ __forceinline__ void store_state(const Acc<D>& a, float* red, int lane, int part) {
  constexpr int MP = D / 16 / RP;
  constexpr int NO = 4 * MP;
#pragma unroll
  for (int q = 0; q < RP; ++q) {
    if (q != part) continue;
#pragma unroll
    for (int i = 0; i < MP; ++i) {
#pragma unroll
      for (int k = 0; k < 4; ++k) red[(4 * i + k) * 32 + lane] = a.o[q * MP + i][k];
    }
  }
  if (part == 0) {
    red[(NO + 0) * 32 + lane] = a.m[0];
    red[(NO + 1) * 32 + lane] = a.m[1];
    red[(NO + 2) * 32 + lane] = a.l[0];
    red[(NO + 3) * 32 + lane] = a.l[1];
  }
}

// Merges the warps of each kv head of segment s and writes the result.
template <int KIND, int D, int KVB, bool PK>
__device__ __forceinline__ void finish_segment(const KParams& p, const Seg& s, Acc<D>& a,
                                               float* red, Misc* misc, const int* pre,
                                               const PlanStore<KIND>& plan) {
  using Gm = Geo<KIND, D, KVB>;
  constexpr int TG = Gm::TG;
  constexpr int NCW = Gm::W;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  const int kvs = warp / TG, tg = warp % TG;
  const int hg = slot_hg<KVB>(p, s.hg, kvs);
  const int nh = unit_nh(p, hg);  // query rows of this warp's slot
  if constexpr (PK) {
    // fold the remainder columns (lane c ^ 2) into the f16-part columns;
    // both lanes of a pair then hold the same state
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int k = 0; k < 4; ++k) a.o[mt][k] += __shfl_xor_sync(0xffffffffu, a.o[mt][k], 2);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float l = a.l[j];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    a.l[j] = l;
  }
  constexpr int SROW = D + 4;  // floats a staged row: D values, the lse, padding
  constexpr int D4 = D / 4;
  auto row_dst = [&](int ks, int h, float*& dst, float*& ldst) {
    const int hgs = slot_hg<KVB>(p, s.hg, ks);
    if (s.dest == DEST_OUT) {
      const long long orow = out_row<KIND>(p, s.b, slot_kv<KVB>(p, s.kvb, ks), hgs, h);
      dst = p.out + orow * D;
      ldst = p.lse ? p.lse + orow : nullptr;
    } else if (KIND == KIND_PAGED_SPLIT && s.dest == DEST_SPLIT) {
      const long long pr =
          out_row<KIND>(p, s.b, slot_kv<KVB>(p, s.kvb, ks), hgs, h) * p.max_splits + s.slot;
      dst = p.o_part + pr * D;
      ldst = p.lse_part + pr;
    } else {
      const long long sl =
          ((long long)blockIdx.x * 2 + s.slot) * (KVB * kHeadTile) + ks * kHeadTile + h;
      dst = p.ws_o + sl * D;
      ldst = p.ws_lse + sl;
    }
  };
  // Flat merge (packed kernels, at most four rows a slot, when every warp's
  // rows fit in the merge buffer): every warp writes its unnormalised rows
  // and its (m, l) to shared memory, then each consumer thread merges one
  // float4 of one row over the TG warps of its slot and stores it.  Two
  // barriers; the tree merge below takes 2 log2(TG) + 2.
  constexpr int RPS = PK ? 4 : kHeadTile;  // staged rows a slot (tree path)
  constexpr bool STAGED = KVB * RPS * SROW <= (NCW / 2) * red_floats(D, Gm::RED_PARTS);
  constexpr int FR = 4;  // rows a slot in the flat buffer
  constexpr bool FLAT =
      PK && (TG * KVB * FR * SROW + 2 * TG * KVB * FR) <= (NCW / 2) * red_floats(D, Gm::RED_PARTS);
  if constexpr (FLAT) {
    float* ml = red + TG * KVB * FR * SROW;  // [kvs][tg][row][m, l]
    if (c < 2) {
      float* fb = red + ((kvs * TG + tg) * FR) * SROW;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = 2 * c + j;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          fb[h * SROW + o_row_d<KIND>(mt, r, 0)] = a.o[mt][j];
          fb[h * SROW + o_row_d<KIND>(mt, r, 1)] = a.o[mt][2 + j];
        }
        if (r == 0) {
          ml[((kvs * TG + tg) * FR + h) * 2 + 0] = a.m[j];
          ml[((kvs * TG + tg) * FR + h) * 2 + 1] = a.l[j];
        }
      }
    }
    named_bar_sync(kRedBarrier, NCW * 32);
#pragma unroll 1
    for (int idx = tid; idx < KVB * FR * D4; idx += NCW * 32) {
      const int d4 = idx % D4, lrow = idx / D4;
      const int ks = lrow / FR, h = lrow % FR;
      if (h >= unit_nh(p, slot_hg<KVB>(p, s.hg, ks))) continue;
      float M = kNegInf;
#pragma unroll
      for (int w = 0; w < TG; ++w) M = fmaxf(M, ml[((ks * TG + w) * FR + h) * 2]);
      float L = 0.f;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < TG; ++w) {
        const float mw = ml[((ks * TG + w) * FR + h) * 2];
        const float sc = (mw == kNegInf) ? 0.f : ex2_ftz(mw - M);
        L += ml[((ks * TG + w) * FR + h) * 2 + 1] * sc;
        const float4 v = *reinterpret_cast<const float4*>(red + ((ks * TG + w) * FR + h) * SROW + 4 * d4);
        O.x += sc * v.x; O.y += sc * v.y; O.z += sc * v.z; O.w += sc * v.w;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      float* dst;
      float* ldst;
      row_dst(ks, h, dst, ldst);
      reinterpret_cast<float4*>(dst)[d4] = make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
      if (d4 == 0 && ldst) *ldst = (M == kNegInf) ? kNegInf : (M + log2f(L)) * kLn2;
    }
    named_bar_sync(kRedBarrier, NCW * 32);  // rows read before the buffer is written again
  } else {
    // tree merge of the TG warps of each kv head; warp tg = 0 ends with the sum
    constexpr int RP = Gm::RED_PARTS;
#pragma unroll
    for (int st = TG / 2; st >= 1; st >>= 1) {
      MergeW w;
#pragma unroll
      for (int part = 0; part < RP; ++part) {
        if (tg >= st && tg < 2 * st)
          store_state<D, RP>(a, red + (kvs * (TG / 2) + (tg - st)) * red_floats(D, RP), lane, part);
        named_bar_sync(kRedBarrier, NCW * 32);
        if (tg < st) merge_state<D, RP>(a, red + (kvs * (TG / 2) + tg) * red_floats(D, RP), lane, part, w);
        named_bar_sync(kRedBarrier, NCW * 32);
      }
    }
    // Results go out through shared memory when the merge buffer (free again
    // after the tree merge's last barrier) holds every row of the unit: the
    // warps holding them (tg = 0) write normalized rows there, and all
    // consumer threads copy whole rows to global memory with 16-byte stores.
    // A slot has at most four rows in the packed kernels, else kHeadTile.
    // Otherwise (the unpacked int8 tiered kernel with four slots, whose merge
    // buffer is halved) the tg = 0 warps store their fragments directly.
    if (tg == 0 && (!PK || c < 2)) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = 2 * c + j;
        if (h >= nh) continue;
        const float L = a.l[j];
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const float lse = (a.m[j] == kNegInf) ? kNegInf : (a.m[j] + log2f(L)) * kLn2;
        float* dst;
        float* ldst;
        if constexpr (STAGED) {
          dst = red + (kvs * RPS + h) * SROW;
          ldst = dst + D;
        } else {
          row_dst(kvs, h, dst, ldst);
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          dst[o_row_d<KIND>(mt, r, 0)] = a.o[mt][j] * inv;
          dst[o_row_d<KIND>(mt, r, 1)] = a.o[mt][2 + j] * inv;
        }
        if (r == 0 && ldst) *ldst = lse;
      }
    }
    if constexpr (STAGED) {
      named_bar_sync(kRedBarrier, NCW * 32);
      for (int idx = tid; idx < KVB * RPS * D4; idx += NCW * 32) {
        const int d4 = idx % D4, lrow = idx / D4;
        const int ks = lrow / RPS, h = lrow % RPS;
        if (h >= unit_nh(p, slot_hg<KVB>(p, s.hg, ks))) continue;
        const float* row = red + lrow * SROW;
        float* dst;
        float* ldst;
        row_dst(ks, h, dst, ldst);
        reinterpret_cast<float4*>(dst)[d4] = *reinterpret_cast<const float4*>(row + 4 * d4);
        if (d4 == 0 && ldst) *ldst = row[D];
      }
      named_bar_sync(kRedBarrier, NCW * 32);  // rows read before the buffer is written again
    }
  }
  if (KIND == KIND_PAGED_SPLIT || s.dest != DEST_PARTIAL) return;
  if (FLAT || STAGED || tg == 0) __threadfence();  // the threads that stored the partial state
  named_bar_sync(kRedBarrier, NCW * 32);
  // ---- last-arriver merge of the unit's partial states
  const long long T = pre[p.B];
  const int sg = stream_grid(p, T);
  const int nt = plan.ntiles(s.pidx);
  const int uib = s.unit - s.b * units_per_seq(p);
  const long long g0 = pre[s.b] + (long long)uib * nt;
  const long long g1 = g0 + nt - 1;
  const int c0 = stream_cta_of(g0, T, sg);
  const int c1 = stream_cta_of(g1, T, sg);
  // A unit cut between CTAs is the segment at the end of its first CTA c0's
  // range, so c0 names the unit's ticket counter.
  if (tid == 0) misc->ticket = atomicAdd(&p.ws_cnt[c0], 1);
  named_bar_sync(kRedBarrier, NCW * 32);
  const int ticket = misc->ticket;
  if (ticket == c1 - c0) {
    __threadfence();
    // One float4 of one head row per thread; the participants' states are
    // read in batches of MB (all loads in flight together) and folded with a
    // running log-sum-exp.  A tiered unit spans five to eight CTAs of the
    // stream and takes batches of eight; the paged units have two or three
    // participants, and there a batch of two measured faster (smaller code
    // on a path every CTA fetches once: two-token steps 71.9 -> 69.9 us,
    // four-token 86.5 -> 83.9 us).
    constexpr int MB = is_tiered(KIND) ? 8 : 2;
    constexpr int D4 = D / 4;
    const int nk = c1 - c0 + 1;
    const int NHs = p.NH;  // rows per slot (the last head group's slots may use fewer)
#pragma unroll 1
    for (int idx = tid; idx < KVB * NHs * D4; idx += NCW * 32) {
      const int d4 = idx % D4;
      const int hh = idx / D4;
      const int ks = hh / NHs, h = hh % NHs;
      if (h >= unit_nh(p, slot_hg<KVB>(p, s.hg, ks))) continue;
      const int rowoff = ks * kHeadTile + h;
      float M = kNegInf, Wsum = 0.f;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
      for (int k0 = 0; k0 < nk; k0 += MB) {
        float ls[MB];
        float4 ov[MB];
#pragma unroll
        for (int j = 0; j < MB; ++j) {
          ls[j] = kNegInf;
          ov[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (k0 + j < nk) {
            const long long sl =
                (long long)stream_slot(c0 + k0 + j, c0, g0, T, sg) * (KVB * kHeadTile) + rowoff;
            ls[j] = __ldcg(p.ws_lse + sl);
            ov[j] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + sl * D) + d4);
          }
        }
        float mb = kNegInf;
#pragma unroll
        for (int j = 0; j < MB; ++j) mb = fmaxf(mb, ls[j]);
        const float mn = fmaxf(M, mb);
        if (mn == kNegInf) continue;
        const float f = (M == kNegInf) ? 0.f : expf(M - mn);
        Wsum *= f;
        O.x *= f; O.y *= f; O.z *= f; O.w *= f;
#pragma unroll
        for (int j = 0; j < MB; ++j) {
          const float w = (ls[j] == kNegInf) ? 0.f : expf(ls[j] - mn);
          Wsum += w;
          O.x += w * ov[j].x; O.y += w * ov[j].y; O.z += w * ov[j].z; O.w += w * ov[j].w;
        }
        M = mn;
      }
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      float lse = kNegInf;
      if (M != kNegInf) {
        const float inv = 1.f / Wsum;
        o = make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
        lse = M + logf(Wsum);
      }
      const long long orow = out_row<KIND>(p, s.b, slot_kv<KVB>(p, s.kvb, ks), slot_hg<KVB>(p, s.hg, ks), h);
      reinterpret_cast<float4*>(p.out + orow * D)[d4] = o;
      if (d4 == 0 && p.lse) p.lse[orow] = lse;
    }
    if (tid == 0) p.ws_cnt[c0] = 0;
  }
  named_bar_sync(kRedBarrier, NCW * 32);
}

template <int KIND, int D, int KVB, bool PK>
__device__ __forceinline__ void consumer_loop(const KParams& p, const PlanStore<KIND>& plan,
                                              const int* pre, uint8_t* stages, uint8_t* hdrs,
                                              uint8_t* qslot, const SmemLayout& L,
                                              const BoxGeo& bg, uint64_t* full, uint64_t* empty,
                                              uint64_t* qfull, uint64_t* qempty, float* red,
                                              Misc* misc, const uint32_t* sp_base) {
  using Gm = Geo<KIND, D, KVB>;
  constexpr int TG = Gm::TG;
  constexpr int NCW = Gm::W;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  const int kvs = warp / TG, tg = warp % TG;
  const int nstages = p.stages;
  const int bs = p.bs;
  const float2 cap = make_float2(p.softcap2, p.softcap_inv);
  const float qscale = p.qscale;
  const int NH = p.NH;
  const int Hkv = p.Hkv;

  // Sequences with no visible key: out = 0, lse = -inf.
  if (KIND != KIND_PAGED_SPLIT) {
#pragma unroll 1
    for (int b = blockIdx.x; b < p.B; b += p.grid) {
      if (plan.ntiles(b) != 0) continue;
      const long long rows = (long long)p.q_len * p.Hq;  // all tokens of sequence b
#pragma unroll 1
      for (long long idx = tid; idx < rows * D; idx += NCW * 32)
        p.out[(long long)b * rows * D + idx] = 0.f;
      if (p.lse)
#pragma unroll 1
        for (long long h = tid; h < rows; h += NCW * 32) p.lse[(long long)b * rows + h] = kNegInf;
    }
  }

  SegIter it;
  seg_init<KIND>(p, plan, pre, it);
  Seg s;
  int stage = 0;
  uint32_t round = 0;
  int qn = 0;
  Acc<D> a;
  QFrag<D> q;

  while (seg_next<KIND, Gm::TOK>(p, plan, pre, it, s)) {
    if (KIND == KIND_PAGED_SPLIT && s.i0 >= s.i1) {
      // SPLIT with no visible key: o = 0, lse = -inf
      const int NHs = p.NH;
      for (int idx = tid; idx < KVB * NHs * D; idx += NCW * 32) {
        const int d = idx % D, hh = idx / D;
        const int ks = hh / NHs, h = hh % NHs;
        const int hgs = slot_hg<KVB>(p, s.hg, ks);
        if (h >= unit_nh(p, hgs)) continue;
        const long long pr =
            out_row<KIND>(p, s.b, slot_kv<KVB>(p, s.kvb, ks), hgs, h) * p.max_splits + s.slot;
        p.o_part[pr * D + d] = 0.f;
        if (d == 0) p.lse_part[pr] = kNegInf;
      }
      continue;
    }
    const SeqPlan e = plan.get(s.pidx);
    const int kv = slot_kv<KVB>(p, s.kvb, kvs);
    const int hg = slot_hg<KVB>(p, s.hg, kvs);
    const int kvsm = kvs >> hgu_shift<KVB>(p);  // this slot's kv head in the stage's boxes
    {
      if (!mbar_wait(qfull, qn & 1, abort_flag(misc), p.wait_ns) && lane == 0) note_abort(misc);
      load_q<KIND, D, PK>(smem_u32(qslot + kvs * NH * D * 4), unit_nh(p, hg), qscale, r, c,
                          q);
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty);
      ++qn;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) a.o[mt][0] = a.o[mt][1] = a.o[mt][2] = a.o[mt][3] = 0.f;
    a.m[0] = a.m[1] = kNegInf;
    a.l[0] = a.l[1] = 0.f;
    // several query tokens: the causal / window bounds of this lane's two
    // score columns (padding columns take the last token's)
    ColMask cm;
    // several query tokens, or per-head key blocks: per-column bounds (the
    // other kinds take one query token and one key set per kv head)
    cm.on = KIND == KIND_PAGED_MULTI || KIND == KIND_PAGED_SPARSE;
    cm.kbase = 0;
    cm.lo[0] = cm.lo[1] = 0;
    cm.hi[0] = cm.hi[1] = 0x7fffffff;
    // block-sparse: shared-memory address of the block bitmask of the layout
    // each of this lane's two columns reads (0: a padding column)
    uint32_t sp_lay[2] = {0u, 0u};
    if constexpr (KIND == KIND_PAGED_SPARSE) {
      const uint32_t* area = sparse_area(sp_base, p, s.pidx);
#pragma unroll
      for (int col = 0; col < 2; ++col) {
        const int head = (PK ? 2 * (c & 1) : 2 * c) + col;
        if (head < unit_nh(p, hg)) {
          const int h = kv * p.G + hg * kHeadTile + head;  // query head of the column
          sp_lay[col] = smem_u32(area + 2 * p.sp_tw + (h % p.sp_nl) * p.sp_bw);
        }
      }
    }
    if (KIND == KIND_PAGED_MULTI) {
#pragma unroll
      for (int col = 0; col < 2; ++col) {
        const int head = (PK ? 2 * (c & 1) : 2 * c) + col;
        int t = (hg * kHeadTile + head) / p.G;
        t = t < p.q_len ? t : p.q_len - 1;
        const long long qp = (long long)e.qp0 + t;
        cm.lo[col] = (p.window > 0 && qp >= p.window) ? (int)(qp - p.window + 1) : 0;
        cm.hi[col] = p.causal ? (int)(qp + 1) : 0x7fffffff;
      }
    }
    HotView hv;
    if constexpr (is_tiered(KIND)) {
      hv.W = p.hot_window;
      hv.cap_eff = p.hot_window > 0 ? p.hot_window : p.hot_cap;
      hv.hs_mod = p.hot_window > 0 ? e.hot_start % p.hot_window : 0;
      const long long j0 = (long long)s.vlo - e.hot_start;
      const long long j1 = (long long)s.vhi - e.hot_start;
      hv.j0 = j0 > 0 ? j0 : 0;
      hv.j1 = j1 < e.hot_len ? j1 : e.hot_len;
    }
    // all ring slots below cap_eff hold visible keys (a full, unmasked ring)
    bool hot_all = false;
    if constexpr (is_tiered(KIND))
      hot_all = hv.j0 <= 0 && hv.j1 >= (hv.W > 0 ? (long long)hv.W : (long long)hv.cap_eff);
    const int vhc = is_tiered(KIND) ? min(s.vhi, e.cold_len) : s.vhi;

    SparseTiles spt;
    if constexpr (KIND == KIND_PAGED_SPARSE) spt.init(sparse_area(sp_base, p, s.pidx), p.sp_tw, s.i0);
    for (int i = s.i0; i < s.i1; ++i) {
      if (!mbar_wait(&full[stage], round & 1, abort_flag(misc), p.wait_ns) && lane == 0) note_abort(misc);
      uint8_t* st = stages + (size_t)stage * L.stage_bytes;
      const uint32_t bad_mask = lds32(smem_u32(hdrs + stage * 16));
      bool is_hot = false;
      int at;
      if constexpr (KIND == KIND_PAGED_SPARSE) at = i == s.i0 ? spt.first : spt.next();
      else at = tile_of<KIND>(e, i, is_hot);
      if (!is_hot) {
        RowMap km, vm;
        km.log2R = bg.log2R;
        km.box_bytes = bg.box_bytes;
        km.cstride = bg.R * 128;
        km.base = smem_u32(st + L.off_k) + (uint32_t)(kvsm * Gm::CHN * bg.R * 128);
        vm = km;
        vm.base = smem_u32(st + L.off_v) + (uint32_t)(kvsm * Gm::CHN * bg.R * 128);
        const int tok0 = at * Gm::TOK;
        auto ok = [&](int k) {
          const int t = tok0 + k;
          if (t < s.vlo || t >= vhc) return false;
          const int j = bs <= Gm::TOK ? (k >> bg.log2R) : 0;
          return ((bad_mask >> j) & 1u) == 0;
        };
        if constexpr (is_paged(KIND)) {
          static_assert(Gm::GPW == 1, "one key group per warp in an f16 tile");
          const int k0 = 16 * tg;
          bool vA = ok(k0 + r), vB = ok(k0 + r + 8);
          if constexpr (KIND == KIND_PAGED_SPARSE) {
            // the group's 16 keys lie in one sparse block (its size is a
            // multiple of 16); a column whose layout does not select it sees
            // none of them, and a group no column selects is skipped
            const int blk = (tok0 + k0) >> p.sp_log2_block;
            bool a0 = false, a1 = false;
            if (blk < 32 * p.sp_bw) {
              const uint32_t wo = (uint32_t)(blk >> 5) * 4u;
              if (sp_lay[0]) a0 = (lds32(sp_lay[0] + wo) >> (blk & 31)) & 1u;
              if (sp_lay[1]) a1 = (lds32(sp_lay[1] + wo) >> (blk & 31)) & 1u;
            }
            cm.lo[0] = a0 ? 0 : 0x7fffffff;
            cm.lo[1] = a1 ? 0 : 0x7fffffff;
            if (!__any_sync(0xffffffffu, a0 || a1)) vA = vB = false;
          }
          if (__any_sync(0xffffffffu, vA || vB)) {
            if (!__all_sync(0xffffffffu, vA && vB)) zero_masked_v_rows<D>(vm, k0, lane, ok);
            cm.kbase = tok0;
            group_compute<TK_PAGED, D, PK>(km, vm, cap, k0, lane, q, a, vA, vB, cm);
          }
        } else if constexpr (KIND == KIND_TIERED_F16) {
          // f16 cold rows, read like hot-ring rows (the tiered d order)
          static_assert(Gm::GPW == 1, "one key group per warp in an f16 tile");
          const int k0 = 16 * tg;
          const bool vA = ok(k0 + r), vB = ok(k0 + r + 8);
          if (__any_sync(0xffffffffu, vA || vB)) {
            if (!__all_sync(0xffffffffu, vA && vB)) zero_masked_v_rows<D>(vm, k0, lane, ok);
            group_compute<TK_PAGED, D, PK>(km, vm, cap, k0, lane, q, a, vA, vB, cm);
          }
        } else {
          // both key groups of the warp in one softmax step (int8 values are
          // always finite, so masked keys need only a zero weight)
          static_assert(Gm::GPW == 2, "two key groups per warp in a cold tile");
          const int k0[2] = {16 * tg, 16 * (tg + TG)};
          const bool v[4] = {ok(k0[0] + r), ok(k0[0] + r + 8), ok(k0[1] + r), ok(k0[1] + r + 8)};
          if (__any_sync(0xffffffffu, v[0] || v[1] || v[2] || v[3])) {
            const uint32_t sck = smem_u32(st + L.off_sc);
            const uint32_t scv = sck + Gm::TOK * Hkv * 2;
            float ks[4], vs[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t off = ((k0[i >> 1] + r + 8 * (i & 1)) * Hkv + kv) * 2;
              ks[i] = __half2float(__ushort_as_half(lds16(sck + off)));
              vs[i] = __half2float(__ushort_as_half(lds16(scv + off)));
            }
            groups_compute<TK_COLD, D, PK, 2>(km, vm, cap, k0, lane, q, a, v, ks, vs, cm);
          }
        }
      } else if constexpr (is_tiered(KIND)) {
        RowMap km, vm;
        km.log2R = 31 - __clz(Gm::TOKH);
        km.box_bytes = 0;
        km.cstride = Gm::TOKH * 128;
        km.base = smem_u32(st + L.off_k) + (uint32_t)(kvsm * Gm::CHH * Gm::TOKH * 128);
        vm = km;
        vm.base = smem_u32(st + L.off_v) + (uint32_t)(kvsm * Gm::CHH * Gm::TOKH * 128);
        const int slot0 = at * Gm::TOKH;
        // every slot of the tile holds a visible key: no per-key ring test
        const bool all_in = hot_all && slot0 + Gm::TOKH <= hv.cap_eff;
        auto ok = [&](int k) { return all_in || key_ok_hot(hv, slot0, k); };
        const int k0 = 16 * tg;
        const bool vA = ok(k0 + r), vB = ok(k0 + r + 8);
        if (__any_sync(0xffffffffu, vA || vB)) {
          if (!__all_sync(0xffffffffu, vA && vB)) zero_masked_v_rows<D>(vm, k0, lane, ok);
          group_compute<KIND == KIND_TIERED_F16 ? TK_PAGED : TK_HOT, D, PK>(km, vm, cap, k0, lane,
                                                                            q, a, vA, vB, cm);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == nstages) {
        stage = 0;
        ++round;
      }
    }
    finish_segment<KIND, D, KVB, PK>(p, s, a, red, misc, pre, plan);
  }
}

// Block-sparse selection of the launch's sequences, by every thread of the
// CTA (com.microsoft.SparseAttention sparse-attention.wgsl.jinja, the
// attention pass: head h reads layout h % NUM_LAYOUT, the query at qp reads
// CSR row qp / SPARSE_BLOCK, each listed column names a block of keys, and a
// repeated column adds nothing).  Per sequence and layout some head reads:
// the bitmask of the blocks its row lists.  Per sequence: the bitmask of
// the tiles of the visible range [lo, hi) that hold a key of a block some
// layout selects, its prefix counts, and the tile count, which replaces the
// plan's.  A row outside the layout, a malformed row and a column outside
// [0, rows) select nothing and raise DEV_BAD_BLOCK.  Returns the device
// flags of the sequences this CTA reports.
template <int KIND, int TOK, int THREADS>
__device__ int sparse_plan(const KParams& p, const PlanStore<KIND>& plan, uint32_t* sp, int tid) {
  const int B = p.B, nlu = p.sp_nlu, tw = p.sp_tw, bw = p.sp_bw, W = p.sp_words;
  const int lg = p.sp_log2_block;
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int NW = THREADS / 32;
  int flags = 0;
  // every (sequence, layout) by one thread: its CSR row's bounds, then its
  // columns, eight loads at a time, into the layout's block bitmask (which
  // only this thread writes)
#pragma unroll 1
  for (int q = tid; q < B * nlu; q += THREADS) {
    const int b = q / nlu, l = q - b * nlu;
    uint32_t* bits = sp + (size_t)b * W + 2 * tw + l * bw;
#pragma unroll 1
    for (int w = 0; w < bw; ++w) bits[w] = 0u;
    const SeqPlan e = plan.get(b);
    int start = 0, len = 0, f = 0;
    if (e.cold_len > 0 && e.qp0 >= 0) {
      const int row = e.qp0 >> lg;
      if (row >= p.sp_rows) {
        f |= DEV_BAD_BLOCK;
      } else {
        const int* rp = p.sp_row_ptr + (long long)l * (p.sp_rows + 1);
        const int s0 = __ldg(rp + row), s1 = __ldg(rp + row + 1);
        if (s0 < 0 || s1 < s0 || s1 > p.sp_nnz) {
          f |= DEV_BAD_BLOCK;
        } else {
          start = s0;
          len = s1 - s0;
        }
      }
    }
    const int* cols = p.sp_col_idx + (long long)l * p.sp_nnz + start;
#pragma unroll 1
    for (int e0 = 0; e0 < len; e0 += 8) {
      int c8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) c8[j] = e0 + j < len ? __ldg(cols + e0 + j) : -2;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = c8[j];
        if (e0 + j >= len) continue;
        if (c < 0 || c >= p.sp_rows) f |= DEV_BAD_BLOCK;
        else if (c < 32 * bw) bits[c >> 5] |= 1u << (c & 31);  // past the bound: no key
      }
    }
    if (b % p.grid == (int)blockIdx.x) flags |= f;
  }
  __syncthreads();
  // tiles of [lo, hi) holding a key of a block that some layout selects: a
  // warp per 32-tile word, lane j deciding tile 32w + j
#pragma unroll 1
  for (int q = warp; q < B * tw; q += NW) {
    const int b = q / tw, w = q - b * tw;
    const SeqPlan e = plan.get(b);
    const uint32_t* a = sp + (size_t)b * W;
    const int t = 32 * w + lane;
    bool on = false;
    if (t >= e.t0 && t < e.t0 + e.ntiles) {
      const int ka = max(t * TOK, e.lo), kb = min(t * TOK + TOK, e.hi);
      for (int blk = ka >> lg; !on && ka < kb && blk <= ((kb - 1) >> lg) && blk < 32 * bw; ++blk) {
        uint32_t u = 0u;
        for (int l = 0; l < nlu; ++l) u |= a[2 * tw + l * bw + (blk >> 5)];
        on = (u >> (blk & 31)) & 1u;
      }
    }
    const uint32_t word = __ballot_sync(0xffffffffu, on);
    if (lane == 0) sp[(size_t)b * W + w] = word;
  }
  __syncthreads();
  // prefix counts and the tile count of every sequence
#pragma unroll 1
  for (int b = tid; b < B; b += THREADS) {
    uint32_t* a = sp + (size_t)b * W;
    int run = 0;
    for (int w = 0; w < tw; ++w) {
      a[tw + w] = (uint32_t)run;
      run += __popc(a[w]);
    }
    SeqPlan e = plan.get(b);
    e.ntiles = run;
    plan.put(b, e);
  }
  __syncthreads();
  return flags;
}

// ================================================================ kernel
// PK: Q/P f16 and remainder parts packed into one MMA operand (requires at
// most four query heads per kv head).
template <int KIND, int D, int KVB, bool PK>
__global__ void __launch_bounds__(Geo<KIND, D, KVB>::THREADS, 1)
    decode_attn_kernel(const __grid_constant__ KParams p) {
  using Gm = Geo<KIND, D, KVB>;
  constexpr int NCW = Gm::W;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  // 1024-aligned base (128-byte TMA swizzle atoms), by pointer arithmetic so
  // the compiler keeps the shared address space.
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int nplan = (KIND == KIND_PAGED_SPLIT) ? 1 : p.B;
  const SmemLayout L = make_layout(KIND, D, KVB, NCW, Gm::REGION >> hgu_shift<KVB>(p), Gm::TOK,
                                   p.NH, p.Hkv, p.stages, nplan,
                                   KIND == KIND_PAGED_SPARSE ? p.sp_words : 0);
  uint8_t* stages = base + L.off_stages;
  uint8_t* hdrs = base + L.off_hdr;
  uint8_t* qslot = base + L.off_q;
  float* red = reinterpret_cast<float*>(base + L.off_red);
  PlanStore<KIND> plan{base + L.off_plan};
  int* pre = reinterpret_cast<int*>(base + L.off_pre);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + L.off_bar);
  uint64_t* empty = full + p.stages;
  uint64_t* qfull = empty + p.stages;
  uint64_t* qempty = qfull + 1;
  Misc* misc = reinterpret_cast<Misc*>(base + L.off_misc);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  BoxGeo bg;
  bg.R = p.bs < Gm::TOK ? p.bs : Gm::TOK;
  bg.log2R = 31 - __clz(bg.R);
  bg.npg = Gm::TOK / bg.R;
  bg.box_bytes = bg.R * Gm::CHN * (KVB >> hgu_shift<KVB>(p)) * 128;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    mbar_init(qfull, 1);
    mbar_init(qempty, NCW);
    fence_mbarrier_init();
    misc->flags = 0;
    misc->ticket = 0;
    misc->abort = 0;
  }
  if (warp == NCW && (tid & 31) == 0) {
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
    if (is_tiered(KIND)) {
      prefetch_tensormap(&p.tm_kh);
      prefetch_tensormap(&p.tm_vh);
    }
  }
  // A block-sparse layout's CSR arrays are read by the plan, behind the
  // lengths.  Each of their 128-byte lines (up to 16 MB of each) is
  // prefetched into L2 by one CTA here, so those dependent reads find them
  // in L2.
  if constexpr (KIND == KIND_PAGED_SPARSE) {
    const long long G = gridDim.x * gridDim.y, c = blockIdx.x + blockIdx.y * gridDim.x;
    auto pf = [&](const void* base, long long bytes) {
      const long long lines = min((bytes + 127) / 128, 1ll << 17);
      for (long long l = c + (long long)tid * G; l < lines; l += G * Gm::THREADS)
        prefetch_l2(reinterpret_cast<const char*>(base) + l * 128);
    };
    pf(p.sp_row_ptr, (long long)p.sp_nl * (p.sp_rows + 1) * 4);
    pf(p.sp_col_idx, (long long)p.sp_nl * p.sp_nnz * 4);
  }
  // ---- per-sequence plan
  int fl = 0;
  if (KIND == KIND_PAGED_SPLIT) {
    if (tid == 0) {
      const int b = blockIdx.y / units_per_seq(p);
      SeqPlan e;
      fl |= plan_sequence<KIND, Gm::TOK, Gm::TOKH>(p, b, e);
      plan.put(0, e);
      if (blockIdx.x == 0 && e.ntiles > 0 &&
          (long long)e.hi > (long long)p.max_splits * p.split_tokens)
        fl |= DEV_SPLIT_OVERFLOW;
    }
  } else {
#pragma unroll 1
    for (int b = tid; b < p.B; b += Gm::THREADS) {
      SeqPlan e;
      const int f = plan_sequence<KIND, Gm::TOK, Gm::TOKH>(p, b, e);
      plan.put(b, e);
      if (b % p.grid == (int)blockIdx.x) fl |= f;  // report once per sequence
    }
  }
  if (fl) atomicOr(&misc->flags, fl);
  __syncthreads();
  uint32_t* sp_base = reinterpret_cast<uint32_t*>(base + L.off_sparse);
  if constexpr (KIND == KIND_PAGED_SPARSE) {
    const int sf = sparse_plan<KIND, Gm::TOK, Gm::THREADS>(p, plan, sp_base, tid);
    if (sf) atomicOr(&misc->flags, sf);
  }
  if (KIND != KIND_PAGED_SPLIT && warp == 0) plan_prefix<KIND>(plan, pre, p.B, units_per_seq(p), tid & 31);
  __syncthreads();

  if (warp >= NCW) {
    if constexpr (Gm::REG_SPLIT) setmaxnreg_dec<Gm::REG_PROD>();
    if (warp == NCW)
      producer_loop<KIND, D, KVB>(p, plan, pre, stages, hdrs, qslot, L, bg, full, empty, qfull,
                                  qempty, misc, sp_base);
  } else {
    if constexpr (Gm::REG_SPLIT) setmaxnreg_inc<Gm::REG_CONS>();
    consumer_loop<KIND, D, KVB, PK>(p, plan, pre, stages, hdrs, qslot, L, bg, full, empty, qfull,
                                qempty, red, misc, sp_base);
  }
  __syncthreads();
  if (tid == 0 && misc->flags && p.dev_status) atomicOr(p.dev_status, misc->flags);
}

}  // namespace da
