// decode_kernel.cuh — single-query GQA attention over a paged (optionally
// int8-tiered) KV cache for sm_103a.
//
// What is computed (per sequence b, query head h, kv = h / (Hq/Hkv)):
//   s_t = scale * <q, k_t>, then cap * tanh(s_t / cap) when cap > 0
//   (@simulatte/doppler 0.1.0 "attention_f16kv.wgsl", softcap step),
//   keys masked by the causal / sliding-window rule of is_masked there,
//   out = softmax(s) V and lse = max + ln(sum)
//   (boostr "paged_attention.wgsl", paged_attention_fwd_f32).
//
// How (GB300 design, not the pages' WGSL):
//   * A work unit is (sequence, kv head, group of <= 8 query heads).  All
//     heads of the group share every K/V byte read from HBM: the group is the
//     n = 8 dimension of mma.m16n8k16, so QK^T is S^T[16 keys x 8 heads] =
//     K[16 x D] * Q^T and PV is O^T[D x 8] += V^T[D x 16] * P^T[16 x 8].
//   * f32 Q and P enter the f16 tensor cores as hi + lo f16 pairs, so the
//     products keep ~22 bits; accumulation is f32.
//   * One producer warp streams 64-key stages through TMA (3-D tensor maps
//     over the pool, one box per page and 64-wide slice of D, 128-byte
//     swizzle) into a ring of shared-memory stages guarded by mbarriers; four
//     consumer warps take 16 keys each and keep their own online-softmax
//     state, merged through shared memory at the end of a unit.
//   * Stream-K split-KV: the key tiles of all units are concatenated and cut
//     into one equal share per CTA.  A unit cut between CTAs leaves partial
//     (o, lse) states in the workspace; the last CTA to finish the unit
//     (atomic ticket, no waiting) merges them with the log-sum-exp rule of
//     com.microsoft.SparseAttention combine_partials.
#pragma once

#include "kernel_params.h"
#include "ptx.cuh"

namespace da {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_inff();

enum { DEST_OUT = 0, DEST_PARTIAL = 1, DEST_SPLIT = 2 };

struct Seg {
  int b, kv, hg, unit;
  int i0, i1;    // unit-local tile range
  int vlo, vhi;  // visible absolute key positions of this segment
  int dest, slot;
  int pidx;      // index of b's plan entry
};

struct SegIter {
  long long g, g_end;
  int n;
};

struct Misc {
  int flags;
  int ticket;
  int abort;
};

// ------------------------------------------------------------------ plan
__device__ __forceinline__ int ceil_div_i(long long a, int b) { return (int)((a + b - 1) / b); }

// Fills plan entry `e` for sequence b (lengths validated, visible range,
// tile counts); returns device-status bits.
template <int KIND>
__device__ int plan_sequence(const KParams& p, int b, SeqPlan& e) {
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
  if (KIND == KIND_PAGED) {
    L = p.seq_lens[b];
    if (L < 0) { flags |= DEV_BAD_SEQ_LEN; L = 0; }
    if (L > cap) { flags |= DEV_BAD_SEQ_LEN; L = cap; }
    qp = L - 1;
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
  // is_masked: causal hides keys after qp; a window W hides keys below
  // qp - W + 1 once qp >= W.
  long long lo = (p.window > 0 && qp >= p.window) ? qp - p.window + 1 : 0;
  long long hi = p.causal ? qp + 1 : (long long)0x7fffffff;
  if (lo < 0) lo = 0;
  if (hi > 0x7fffffff) hi = 0x7fffffff;
  e.lo = (int)lo;
  e.hi = (int)hi;
  if (empty) return flags;
  if (KIND == KIND_PAGED) {
    long long vh = hi < L ? hi : L;
    e.hi = (int)vh;
    if (vh > lo) {
      e.t0 = (int)(lo / kTile);
      e.ntiles = ceil_div_i(vh, kTile) - e.t0;
    }
  } else {
    e.cold_len = (int)cl;
    e.hot_start = (int)hs;
    e.hot_len = (int)hl;
    long long ch = hi < cl ? hi : cl;
    if (ch > lo) {
      e.t0 = (int)(lo / kTile);
      e.ncold = ceil_div_i(ch, kTile) - e.t0;
    }
    long long j0 = lo - hs > 0 ? lo - hs : 0;
    long long j1 = hi - hs < hl ? hi - hs : hl;
    int nhot = 0;
    if (j1 > j0) {
      if (p.hot_window > 0) {
        const int W = p.hot_window;
        const int nT = ceil_div_i(W, kTile);
        long long s0 = (hs + j0) % W;
        long long n = j1 - j0;
        if (s0 + n <= W) {
          e.ha0 = (int)(s0 / kTile);
          e.ha1 = ceil_div_i(s0 + n, kTile);
        } else {
          int te = ceil_div_i(s0 + n - W, kTile);
          int ts = (int)(s0 / kTile);
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
        e.ha0 = (int)(j0 / kTile);
        e.ha1 = ceil_div_i(j1, kTile);
      }
      nhot = (e.ha1 - e.ha0) + (e.hb1 - e.hb0);
    }
    e.ntiles = e.ncold + nhot;
  }
  return flags;
}

// Exclusive prefix of ntiles * units_per_seq over the batch (one warp).
__device__ __forceinline__ void plan_prefix(const SeqPlan* plan, int* pre, int B, int upb, int lane) {
  const int per = (B + 31) / 32;
  const int b0 = lane * per;
  long long sum = 0;
  for (int i = 0; i < per; ++i)
    if (b0 + i < B) sum += (long long)plan[b0 + i].ntiles * upb;
  long long incl = sum;
  for (int off = 1; off < 32; off <<= 1) {
    long long v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  long long run = incl - sum;
  for (int i = 0; i < per; ++i) {
    if (b0 + i < B) {
      pre[b0 + i] = (int)run;
      run += (long long)plan[b0 + i].ntiles * upb;
    }
  }
  if (lane == 31) pre[B] = (int)incl;
}

// ----------------------------------------------------------- scheduling
__device__ __forceinline__ int stream_cta_of(long long g, long long T, int grid) {
  return (int)(((g + 1) * grid - 1) / T);
}
__device__ __forceinline__ long long stream_start(int c, long long T, int grid) {
  return (long long)c * T / grid;
}

__device__ __forceinline__ void seg_init(const KParams& p, const int* pre, SegIter& it) {
  it.n = 0;
  if (p.sched == SCHED_STREAM) {
    const long long T = pre[p.B];
    it.g = stream_start(blockIdx.x, T, p.grid);
    it.g_end = stream_start(blockIdx.x + 1, T, p.grid);
  } else if (p.sched == SCHED_UNITS) {
    const long long U = (long long)p.B * p.Hkv * p.HG;
    it.g = (long long)blockIdx.x * U / p.grid;
    it.g_end = (long long)(blockIdx.x + 1) * U / p.grid;
  } else {
    it.g = 0;
    it.g_end = 1;
  }
}

__device__ __forceinline__ bool seg_next(const KParams& p, const SeqPlan* plan, const int* pre,
                                         SegIter& it, Seg& s) {
  const int upb = p.Hkv * p.HG;
  if (p.sched == SCHED_STREAM) {
    if (it.g >= it.g_end) return false;
    int lo = 0, hi = p.B;  // largest b with pre[b] <= g
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (pre[mid] <= it.g) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int nt = plan[b].ntiles;
    const long long local = it.g - pre[b];
    const int uib = (int)(local / nt);
    s.b = b;
    s.pidx = b;
    s.kv = uib / p.HG;
    s.hg = uib % p.HG;
    s.unit = b * upb + uib;
    s.i0 = (int)(local % nt);
    long long rem = it.g_end - it.g;
    s.i1 = (int)((long long)s.i0 + rem < nt ? s.i0 + rem : nt);
    s.vlo = plan[b].lo;
    s.vhi = plan[b].hi;
    s.dest = (s.i0 == 0 && s.i1 == nt) ? DEST_OUT : DEST_PARTIAL;
    s.slot = it.n == 0 ? 0 : 1;
    it.g += s.i1 - s.i0;
    it.n++;
    return true;
  }
  if (p.sched == SCHED_UNITS) {
    while (it.g < it.g_end) {
      const int u = (int)it.g++;
      const int b = u / upb;
      if (plan[b].ntiles == 0) continue;
      const int uib = u % upb;
      s.b = b;
      s.pidx = b;
      s.kv = uib / p.HG;
      s.hg = uib % p.HG;
      s.unit = u;
      s.i0 = 0;
      s.i1 = plan[b].ntiles;
      s.vlo = plan[b].lo;
      s.vhi = plan[b].hi;
      s.dest = DEST_OUT;
      s.slot = 0;
      it.n++;
      return true;
    }
    return false;
  }
  // SCHED_SPLIT: one segment, the keys of split blockIdx.x of unit blockIdx.y
  if (it.n > 0) return false;
  it.n = 1;
  const int u = blockIdx.y;
  const int b = u / upb;
  const int uib = u % upb;
  s.b = b;
  s.pidx = 0;
  s.kv = uib / p.HG;
  s.hg = uib % p.HG;
  s.unit = u;
  s.dest = DEST_SPLIT;
  s.slot = blockIdx.x;
  const long long st0 = (long long)blockIdx.x * p.split_tokens;
  const long long st1 = st0 + p.split_tokens;
  long long vlo = plan[0].lo > st0 ? plan[0].lo : st0;
  long long vhi = plan[0].hi < st1 ? plan[0].hi : st1;
  s.i0 = s.i1 = 0;
  s.vlo = (int)vlo;
  s.vhi = (int)(vhi > vlo ? vhi : vlo);
  if (plan[0].ntiles > 0 && vhi > vlo) {
    s.i0 = (int)(vlo / kTile) - plan[0].t0;
    s.i1 = ceil_div_i(vhi, kTile) - plan[0].t0;
  }
  return true;
}

// Flat index of the last CTA's partial slot for participant c of a unit
// whose first tile is g0 (STREAM).
__device__ __forceinline__ int stream_slot(int c, int c0, long long g0, long long T, int grid) {
  const int j = (c == c0 && stream_start(c, T, grid) < g0) ? 1 : 0;
  return c * 2 + j;
}

// ---------------------------------------------------------- tile geometry
// Paged / cold tile: absolute tile `at` covers keys [at*64, at*64+64).
struct PageSpan {
  int p_first;  // first page of the tile
  int npg;      // pages in the tile
  int rows;     // rows per box (min(bs, 64))
  int row_off;  // row offset inside the page (bs > 64)
};

__device__ __forceinline__ PageSpan page_span(const KParams& p, int at) {
  PageSpan ps;
  const int tok0 = at * kTile;
  ps.p_first = tok0 >> p.log2_bs;
  if (p.bs <= kTile) {
    ps.npg = kTile >> p.log2_bs;
    ps.rows = p.bs;
    ps.row_off = 0;
  } else {
    ps.npg = 1;
    ps.rows = kTile;
    ps.row_off = tok0 & (p.bs - 1);
  }
  return ps;
}

// ============================================================== producer
template <int KIND, int D>
__device__ void producer_loop(const KParams& p, const SeqPlan* plan, const int* pre,
                              uint8_t* stages, const SmemLayout& L, uint64_t* full,
                              uint64_t* empty, Misc* misc) {
  const int lane = threadIdx.x & 31;
  constexpr int CH = D / 64;  // 64-element slices of D (f16 boxes)
  SegIter it;
  seg_init(p, pre, it);
  Seg s;
  int stage = 0;
  uint32_t round = 0;
  int bt_b = -1, bt_base = 0, bt_cur = -1, bt_nxt = -1;
  int flags = 0;
  const int* bt_all = p.block_table;
  while (seg_next(p, plan, pre, it, s)) {
    if (s.i0 >= s.i1) continue;
    const SeqPlan& e = plan[s.pidx];
    const int* bt_row = bt_all + (long long)s.b * p.max_blocks;
    for (int i = s.i0; i < s.i1; ++i) {
      if (!mbar_wait(&empty[stage], (round & 1) ^ 1)) {
        if (lane == 0) atomicOr(&misc->flags, DEV_TIMEOUT);
        misc->abort = 1;
        return;
      }
      uint8_t* st = stages + (size_t)stage * L.stage_bytes;
      uint32_t bytes = 0;
      uint32_t bad_mask = 0;
      const bool q_load = (i == s.i0);
      if (q_load) bytes += (uint32_t)p.NH * D * 4;
      bool is_hot = false;
      int at = 0;
      if (KIND == KIND_TIERED && i >= e.ncold) {
        is_hot = true;
        const int hi_ = i - e.ncold;
        const int na = e.ha1 - e.ha0;
        at = hi_ < na ? e.ha0 + hi_ : e.hb0 + (hi_ - na);
      } else {
        at = e.t0 + i;
      }
      if (!is_hot) {
        // ----- pages through the block table
        const PageSpan ps = page_span(p, at);
        // keep a 64-entry window of block-table entries in two registers
        if (s.b != bt_b || ps.p_first < bt_base || ps.p_first + ps.npg > bt_base + 64) {
          if (s.b == bt_b && ps.p_first >= bt_base + 32 && ps.p_first + ps.npg <= bt_base + 96) {
            bt_cur = bt_nxt;
            bt_base += 32;
          } else {
            bt_base = ps.p_first;
            const int pc = bt_base + lane;
            bt_cur = pc < p.max_blocks ? __ldg(bt_row + pc) : -1;
          }
          const int pn = bt_base + 32 + lane;
          bt_nxt = pn < p.max_blocks ? __ldg(bt_row + pn) : -1;
          bt_b = s.b;
        }
        const int vhi_keys = (KIND == KIND_TIERED) ? min(s.vhi, e.cold_len) : s.vhi;
        // page ids of this lane's copies (lane -> page lane / (2*CH'))
        constexpr int OPS = (KIND == KIND_PAGED) ? 2 * CH : 2 * (D / 128) + 2;
        int my_blk0 = -1, my_blk1 = -1;
        uint32_t need_mask = 0;
        for (int j = 0; j < ps.npg; ++j) {
          const int pg = ps.p_first + j;
          const int idx = pg - bt_base;
          const int vc = __shfl_sync(0xffffffffu, bt_cur, idx & 31);
          const int vn = __shfl_sync(0xffffffffu, bt_nxt, idx & 31);
          const int blk = pg < p.max_blocks ? (idx < 32 ? vc : vn) : -1;
          const int r0 = at * kTile + j * ps.rows;
          const bool needed = (r0 < vhi_keys) && (r0 + ps.rows > s.vlo);
          if (!needed) continue;
          if (blk < 0 || blk >= p.num_blocks) {
            bad_mask |= 1u << j;
            continue;
          }
          need_mask |= 1u << j;
          if constexpr (KIND == KIND_PAGED) {
            bytes += (uint32_t)(2 * CH * ps.rows * 128);
          } else {
            bytes += (uint32_t)(2 * (D / 128) * ps.rows * 128 + 2 * p.bs * p.Hkv * 2);
          }
          if (lane / OPS == j) my_blk0 = blk;
          if ((lane + 32) / OPS == j) my_blk1 = blk;
        }
        if (bad_mask) flags |= DEV_BAD_BLOCK;
        if (lane == 0) {
          *reinterpret_cast<uint32_t*>(st + L.off_hdr) = bad_mask;
          mbar_arrive_expect_tx(&full[stage], bytes);
        }
        __syncwarp();
        // issue the copies: op = lane (and lane + 32)
#pragma unroll
        for (int rep = 0; rep < 2; ++rep) {
          const int op = lane + rep * 32;
          const int j = op / OPS;
          const int blk = rep ? my_blk1 : my_blk0;
          if (j < ps.npg && ((need_mask >> j) & 1u)) {
            const int r = op % OPS;
            const int row = blk * p.bs + ps.row_off;
            if constexpr (KIND == KIND_PAGED) {
              const int isv = r / CH;
              const int ch = r % CH;
              uint8_t* dst = st + (isv ? L.off_v : L.off_k) + ch * (kTile * 128) + j * ps.rows * 128;
              tma_load_3d(dst, isv ? &p.tm_v : &p.tm_k, &full[stage], ch * 64, s.kv, row);
            } else {
              constexpr int CC = D / 128;  // 128-byte slices of an int8 row
              if (r < 2 * CC) {
                const int isv = r / CC;
                const int ch = r % CC;
                uint8_t* dst = st + (isv ? L.off_v : L.off_k) + ch * (kTile * 128) + j * ps.rows * 128;
                tma_load_3d(dst, isv ? &p.tm_v : &p.tm_k, &full[stage], ch * 128, s.kv, row);
              } else {
                const int isv = r - 2 * CC;
                const uint16_t* src = (isv ? p.v_scale : p.k_scale) + (long long)blk * p.bs * p.Hkv;
                uint8_t* dst = st + L.off_sc + isv * (kTile * p.Hkv * 2) + j * p.bs * p.Hkv * 2;
                bulk_load(dst, src, (uint32_t)(p.bs * p.Hkv * 2), &full[stage]);
              }
            }
          }
        }
      } else {
        // ----- hot ring tile: slots [at*64, at*64+64) of sequence b
        if (lane == 0) {
          bytes += (uint32_t)(2 * CH * kTile * 128);
          *reinterpret_cast<uint32_t*>(st + L.off_hdr) = 0u;
          mbar_arrive_expect_tx(&full[stage], bytes);
        }
        __syncwarp();
        if (lane < 2 * CH) {
          const int isv = lane / CH;
          const int ch = lane % CH;
          uint8_t* dst = st + (isv ? L.off_v : L.off_k) + ch * (kTile * 128);
          tma_load_4d(dst, isv ? &p.tm_vh : &p.tm_kh, &full[stage], ch * 64, s.kv, at * kTile,
                      s.b + p.hot_b0);
        }
      }
      if (q_load && lane == 0) {
        const float* src = p.q + ((long long)s.b * p.Hq + s.kv * p.G + s.hg * kHeadTile) * D;
        bulk_load(st + L.off_q, src, (uint32_t)(p.NH * D * 4), &full[stage]);
      }
      if (++stage == p.stages) {
        stage = 0;
        ++round;
      }
    }
  }
  if (flags && lane == 0) atomicOr(&misc->flags, flags);
}

// ============================================================== consumer
template <int D>
struct Acc {
  float o[D / 16][4];  // O^T fragments: (d = 16mt + r (+8), head 2c (+1))
  float m[2], l[2];    // heads 2c, 2c+1 (base-2 units)
};

// Writes the merged result of the four consumer warps for segment s.
template <int KIND, int D>
__device__ void finish_segment(const KParams& p, const Seg& s, Acc<D>& a, float* red_o,
                               float* red_ml, Misc* misc, const int* pre, const SeqPlan* plan) {
  const int tid = threadIdx.x;  // 0..127
  const int warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  const int NH = p.NH;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float l = a.l[j];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    a.l[j] = l;
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int h = 2 * c + j;
    if (h < NH) {
      float* ro = red_o + (warp * NH + h) * D;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        ro[16 * mt + r] = a.o[mt][j];
        ro[16 * mt + r + 8] = a.o[mt][2 + j];
      }
      if (r == 0) {
        red_ml[(warp * NH + h) * 2 + 0] = a.m[j];
        red_ml[(warp * NH + h) * 2 + 1] = a.l[j];
      }
    }
  }
  named_bar_sync(kRedBarrier, kConsumerWarps * 32);
  const int h0 = s.kv * p.G + s.hg * kHeadTile;
  const long long row0 = (long long)s.b * p.Hq + h0;
  for (int idx = tid; idx < NH * D; idx += kConsumerWarps * 32) {
    const int h = idx / D, d = idx % D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_ml[(w * NH + h) * 2]);
    float o = 0.f, lse = kNegInf;
    if (M != kNegInf) {
      float Ls = 0.f, Os = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float f = exp2f(red_ml[(w * NH + h) * 2] - M);
        Ls += f * red_ml[(w * NH + h) * 2 + 1];
        Os += f * red_o[(w * NH + h) * D + d];
      }
      o = Os / Ls;
      lse = (M + log2f(Ls)) * kLn2;
    }
    if (s.dest == DEST_OUT) {
      p.out[(row0 + h) * D + d] = o;
      if (d == 0 && p.lse) p.lse[row0 + h] = lse;
    } else if (s.dest == DEST_SPLIT) {
      const long long pr = (row0 + h) * p.max_splits + s.slot;
      p.o_part[pr * D + d] = o;
      if (d == 0) p.lse_part[pr] = lse;
    } else {
      const long long sl = ((long long)blockIdx.x * 2 + s.slot) * kHeadTile + h;
      p.ws_o[sl * D + d] = o;
      if (d == 0) p.ws_lse[sl] = lse;
    }
  }
  if (s.dest == DEST_PARTIAL) __threadfence();
  named_bar_sync(kRedBarrier, kConsumerWarps * 32);
  if (s.dest != DEST_PARTIAL) return;
  // ---- last-arriver merge of the unit's partial states
  const long long T = pre[p.B];
  const int nt = plan[s.pidx].ntiles;
  const int uib = s.unit - s.b * p.Hkv * p.HG;
  const long long g0 = pre[s.b] + (long long)uib * nt;
  const long long g1 = g0 + nt - 1;
  const int c0 = stream_cta_of(g0, T, p.grid);
  const int c1 = stream_cta_of(g1, T, p.grid);
  if (tid == 0) misc->ticket = atomicAdd(&p.ws_cnt[s.unit], 1);
  named_bar_sync(kRedBarrier, kConsumerWarps * 32);
  const int ticket = misc->ticket;
  if (ticket == c1 - c0) {
    __threadfence();
    for (int idx = tid; idx < NH * D; idx += kConsumerWarps * 32) {
      const int h = idx / D, d = idx % D;
      float M = kNegInf;
      for (int cc = c0; cc <= c1; ++cc) {
        const long long sl = (long long)stream_slot(cc, c0, g0, T, p.grid) * kHeadTile + h;
        M = fmaxf(M, __ldcg(p.ws_lse + sl));
      }
      float o = 0.f, lse = kNegInf;
      if (M != kNegInf) {
        float Ws = 0.f, Os = 0.f;
        for (int cc = c0; cc <= c1; ++cc) {
          const long long sl = (long long)stream_slot(cc, c0, g0, T, p.grid) * kHeadTile + h;
          const float ls = __ldcg(p.ws_lse + sl);
          const float w = (ls == kNegInf) ? 0.f : expf(ls - M);
          Ws += w;
          Os += w * __ldcg(p.ws_o + sl * D + d);
        }
        o = Os / Ws;
        lse = M + logf(Ws);
      }
      p.out[(row0 + h) * D + d] = o;
      if (d == 0 && p.lse) p.lse[row0 + h] = lse;
    }
    if (tid == 0) p.ws_cnt[s.unit] = 0;
  }
  named_bar_sync(kRedBarrier, kConsumerWarps * 32);
}

// Key validity of row k (0..63) of a paged / cold tile.
__device__ __forceinline__ bool key_ok_paged(const KParams& p, int at, int k, int vlo, int vhi,
                                             uint32_t bad_mask) {
  const int t = at * kTile + k;
  if (t < vlo || t >= vhi) return false;
  const int j = p.bs <= kTile ? (k >> p.log2_bs) : 0;
  return ((bad_mask >> j) & 1u) == 0;
}

template <int KIND, int D>
__device__ void consumer_loop(const KParams& p, const SeqPlan* plan, const int* pre,
                              uint8_t* stages, const SmemLayout& L, uint64_t* full,
                              uint64_t* empty, float* red_o, float* red_ml, Misc* misc) {
  constexpr int KS = D / 16;  // k-steps of QK, m-tiles of PV
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  const int k0 = warp * 16;

  // Sequences with no visible key: out = 0, lse = -inf.
  if (p.sched != SCHED_SPLIT) {
    for (int b = blockIdx.x; b < p.B; b += p.grid) {
      if (plan[b].ntiles != 0) continue;
      for (int idx = tid; idx < p.Hq * D; idx += kConsumerWarps * 32)
        p.out[(long long)b * p.Hq * D + idx] = 0.f;
      if (p.lse)
        for (int h = tid; h < p.Hq; h += kConsumerWarps * 32) p.lse[(long long)b * p.Hq + h] = kNegInf;
    }
  }

  SegIter it;
  seg_init(p, pre, it);
  Seg s;
  int stage = 0;
  uint32_t round = 0;
  Acc<D> a;
  uint32_t qhi[KS][2], qlo[KS][2];

  while (seg_next(p, plan, pre, it, s)) {
    if (s.i0 >= s.i1) {
      // SPLIT with no visible key: o = 0, lse = -inf
      const int h0 = s.kv * p.G + s.hg * kHeadTile;
      for (int idx = tid; idx < p.NH * D; idx += kConsumerWarps * 32) {
        const int h = idx / D, d = idx % D;
        const long long pr = ((long long)s.b * p.Hq + h0 + h) * p.max_splits + s.slot;
        p.o_part[pr * D + d] = 0.f;
        if (d == 0) p.lse_part[pr] = kNegInf;
      }
      continue;
    }
    const SeqPlan& e = plan[s.pidx];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) a.o[mt][0] = a.o[mt][1] = a.o[mt][2] = a.o[mt][3] = 0.f;
    a.m[0] = a.m[1] = kNegInf;
    a.l[0] = a.l[1] = 0.f;

    for (int i = s.i0; i < s.i1; ++i) {
      if (!mbar_wait(&full[stage], round & 1)) {
        if (lane == 0) atomicOr(&misc->flags, DEV_TIMEOUT);
        misc->abort = 1;
        return;
      }
      uint8_t* st = stages + (size_t)stage * L.stage_bytes;
      if (i == s.i0) {
        // Q rows of the head group, prescaled by scale*log2(e), as hi/lo f16
        const float* qs = reinterpret_cast<const float*>(st + L.off_q);
        const bool hv = r < p.NH;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int d0 = 16 * ks + 2 * c;
          float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
          if (hv) {
            x0 = qs[r * D + d0] * p.qscale;
            x1 = qs[r * D + d0 + 1] * p.qscale;
            x2 = qs[r * D + d0 + 8] * p.qscale;
            x3 = qs[r * D + d0 + 9] * p.qscale;
          }
          split_half2(x0, x1, qhi[ks][0], qlo[ks][0]);
          split_half2(x2, x3, qhi[ks][1], qlo[ks][1]);
        }
      }
      const uint32_t bad_mask = *reinterpret_cast<const uint32_t*>(st + L.off_hdr);
      const int at = e.t0 + i;
      const bool vA = key_ok_paged(p, at, k0 + r, s.vlo, s.vhi, bad_mask);
      const bool vB = key_ok_paged(p, at, k0 + r + 8, s.vlo, s.vhi, bad_mask);
      const bool any = __any_sync(0xffffffffu, vA || vB);
      if (any) {
        const uint8_t* kst = st + L.off_k;
        uint8_t* vst = st + L.off_v;
        if (!__all_sync(0xffffffffu, vA && vB)) {
          // zero the V rows of masked keys so 0 * (stale or non-finite) cannot leak
          constexpr int UPR = D / 8;  // 16-byte units per row
          for (int u = lane; u < 16 * UPR; u += 32) {
            const int row = u / UPR, ug = u % UPR;
            const int k = k0 + row;
            if (!key_ok_paged(p, at, k, s.vlo, s.vhi, bad_mask)) {
              uint8_t* dst = vst + (ug >> 3) * (kTile * 128) + k * 128 + (((ug & 7) ^ (k & 7)) << 4);
              *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        // ---- S^T = K Q^T (16 keys x 8 heads)
        float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const int mat = lane >> 3;
          const int key = k0 + (lane & 7) + ((mat & 1) << 3);
          const uint32_t rowaddr = smem_u32(kst) + key * 128;
          const int x = lane & 7;
          const int dh = mat >> 1;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const int ug = 2 * ks + dh;
            const uint32_t addr = rowaddr + (ug >> 3) * (kTile * 128) + (((ug & 7) ^ x) << 4);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(addr, a0, a1, a2, a3);
            mma_f16_16816(sh, a0, a1, a2, a3, qhi[ks][0], qhi[ks][1]);
            mma_f16_16816(sl, a0, a1, a2, a3, qlo[ks][0], qlo[ks][1]);
          }
        }
        float sc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float v = sh[j] + sl[j];
          if (p.softcap2 > 0.f) v = p.softcap2 * tanhf(v / p.softcap2);
          sc[j] = v;
        }
        if (!vA) sc[0] = sc[1] = kNegInf;
        if (!vB) sc[2] = sc[3] = kNegInf;
        // ---- online softmax (base 2)
        float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(a.m[0], mx0), mn1 = fmaxf(a.m[1], mx1);
        const float al0 = (mn0 == kNegInf) ? 1.f : exp2f(a.m[0] - mn0);
        const float al1 = (mn1 == kNegInf) ? 1.f : exp2f(a.m[1] - mn1);
        const float mu0 = (mn0 == kNegInf) ? 0.f : mn0;
        const float mu1 = (mn1 == kNegInf) ? 0.f : mn1;
        const float p0 = exp2f(sc[0] - mu0), p1 = exp2f(sc[1] - mu1);
        const float p2 = exp2f(sc[2] - mu0), p3 = exp2f(sc[3] - mu1);
        a.l[0] = a.l[0] * al0 + (p0 + p2);
        a.l[1] = a.l[1] * al1 + (p1 + p3);
        a.m[0] = mn0;
        a.m[1] = mn1;
        if (!__all_sync(0xffffffffu, al0 == 1.f && al1 == 1.f)) {
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            a.o[mt][0] *= al0;
            a.o[mt][1] *= al1;
            a.o[mt][2] *= al0;
            a.o[mt][3] *= al1;
          }
        }
        // ---- P^T as the B operand (hi + lo), via an 8x8 transpose
        uint32_t h01, l01, h23, l23;
        split_half2(p0, p1, h01, l01);
        split_half2(p2, p3, h23, l23);
        const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
        const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);
        // ---- O^T += V^T P^T
        {
          const int mat = lane >> 3;
          const int key = k0 + (lane & 7) + ((mat >> 1) << 3);
          const uint32_t rowaddr = smem_u32(vst) + key * 128;
          const int x = lane & 7;
          const int dh = mat & 1;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            const int ug = 2 * mt + dh;
            const uint32_t addr = rowaddr + (ug >> 3) * (kTile * 128) + (((ug & 7) ^ x) << 4);
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(addr, a0, a1, a2, a3);
            mma_f16_16816(a.o[mt], a0, a1, a2, a3, bh0, bh1);
            mma_f16_16816(a.o[mt], a0, a1, a2, a3, bl0, bl1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == p.stages) {
        stage = 0;
        ++round;
      }
    }
    finish_segment<KIND, D>(p, s, a, red_o, red_ml, misc, pre, plan);
  }
}

// ================================================================ kernel
template <int KIND, int D>
__global__ void __launch_bounds__(kThreads, 1) decode_attn_kernel(const __grid_constant__ KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int nplan = (p.sched == SCHED_SPLIT) ? 1 : p.B;
  const SmemLayout L = make_layout(KIND, D, p.NH, p.Hkv, p.stages, nplan);
  uint8_t* stages = base + L.off_stages;
  float* red_o = reinterpret_cast<float*>(base + L.off_red_o);
  float* red_ml = reinterpret_cast<float*>(base + L.off_red_ml);
  SeqPlan* plan = reinterpret_cast<SeqPlan*>(base + L.off_plan);
  int* pre = reinterpret_cast<int*>(base + L.off_pre);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + L.off_bar);
  uint64_t* empty = full + p.stages;
  Misc* misc = reinterpret_cast<Misc*>(base + L.off_misc);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbarrier_init();
    misc->flags = 0;
    misc->ticket = 0;
    misc->abort = 0;
  }
  if (warp == kConsumerWarps && (tid & 31) == 0) {
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
    if (KIND == KIND_TIERED) {
      prefetch_tensormap(&p.tm_kh);
      prefetch_tensormap(&p.tm_vh);
    }
  }
  // ---- per-sequence plan
  int fl = 0;
  if (p.sched == SCHED_SPLIT) {
    if (tid == 0) {
      const int b = blockIdx.y / (p.Hkv * p.HG);
      fl |= plan_sequence<KIND>(p, b, plan[0]);
      if (blockIdx.x == 0 && plan[0].ntiles > 0 &&
          (long long)plan[0].hi > (long long)p.max_splits * p.split_tokens)
        fl |= DEV_SPLIT_OVERFLOW;
    }
  } else {
    for (int b = tid; b < p.B; b += kThreads) {
      int f = plan_sequence<KIND>(p, b, plan[b]);
      if (b % p.grid == (int)blockIdx.x) fl |= f;  // report once per sequence
    }
  }
  if (fl) atomicOr(&misc->flags, fl);
  __syncthreads();
  if (p.sched != SCHED_SPLIT && warp == 0) plan_prefix(plan, pre, p.B, p.Hkv * p.HG, tid & 31);
  __syncthreads();

  if (warp == kConsumerWarps) {
    producer_loop<KIND, D>(p, plan, pre, stages, L, full, empty, misc);
  } else {
    consumer_loop<KIND, D>(p, plan, pre, stages, L, full, empty, red_o, red_ml, misc);
  }
  __syncthreads();
  if (tid == 0 && misc->flags && p.dev_status) atomicOr(p.dev_status, misc->flags);
}

}  // namespace da
