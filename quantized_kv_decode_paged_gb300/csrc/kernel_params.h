// kernel_params.h — the parameter block the host launcher hands to the
// decode kernels, their per-instantiation geometry, and the shared-memory
// layout both sides compute.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace da {

constexpr int kHeadTile = 8;             // query heads per kv head in a unit (the MMA n dim)
constexpr int kMaxStages = 8;
constexpr int kMaxBatchPerLaunch = 256;  // per-sequence plan lives in shared memory
constexpr int kSmemLimit = 232448;       // 227 KB opt-in per block on sm_100-class parts
constexpr uint32_t kRedBarrier = 1;      // named barrier id for the consumer warps

// PAGED: f16 pages, one query token per sequence.  PAGED_MULTI: f16 pages,
// several query tokens per sequence.  TIERED: int8 cold pages (+ f16
// scales) and an f16 hot ring.  TIERED_F16: f16 cold pages and an f16 hot ring.
// PAGED_SPARSE: f16 pages, one query token, keys selected per query head by
// a block-sparse CSR layout.  PAGED_SPLIT: PAGED under the SPLIT schedule
// (the split-partial entry point); PAGED runs STREAM and UNITS only, so that
// neither kernel carries the other's code.
enum Kind : int {
  KIND_PAGED = 0,
  KIND_TIERED = 1,
  KIND_TIERED_F16 = 2,
  KIND_PAGED_MULTI = 3,
  KIND_PAGED_SPARSE = 4,
  KIND_PAGED_SPLIT = 5
};
__host__ __device__ constexpr bool is_paged(int kind) {
  return kind == KIND_PAGED || kind == KIND_PAGED_MULTI || kind == KIND_PAGED_SPARSE ||
         kind == KIND_PAGED_SPLIT;
}
// one query token, no per-head key selection: the compact per-sequence plan
__host__ __device__ constexpr bool one_token_paged(int kind) {
  return kind == KIND_PAGED || kind == KIND_PAGED_SPLIT;
}
__host__ __device__ constexpr bool is_tiered(int kind) { return !is_paged(kind); }
__host__ __device__ constexpr bool cold_int8(int kind) { return kind == KIND_TIERED; }
// STREAM: every CTA takes an equal share of the concatenated key tiles of all
//         units; units cut between CTAs are merged by the last CTA to finish.
// UNITS:  every CTA takes whole units (no workspace needed).
// SPLIT:  CTA (s, unit) covers keys [s*split_tokens, (s+1)*split_tokens) and
//         writes a partial result.
enum Sched : int { SCHED_STREAM = 0, SCHED_UNITS = 1, SCHED_SPLIT = 2 };

// Device status bits (same values as the public DA_DEV_* enum).
enum : int {
  DEV_BAD_BLOCK = 1,
  DEV_BAD_SEQ_LEN = 2,
  DEV_BAD_QPOS = 4,
  DEV_SPLIT_OVERFLOW = 8,
  DEV_BAD_TIER = 16,
  DEV_TIMEOUT = 32
};

// Geometry of one kernel instantiation.
//   KVB kv heads are processed together, so every token row read from the
//   pool is KVB * (row bytes of one head) contiguous bytes: >= 512 B keeps
//   HBM streaming near its peak, 256-byte pieces at a 2 KB stride do not.
//   W consumer warps; warp w takes kv head w / TG of the block and the
//   16-key groups g of a tile with g % TG == w % TG, TG = W / KVB.
//   A paged tile holds TOK = 16*TG keys of each of the KVB heads (one group
//   per warp); an int8 cold tile 2*16*TG keys (two groups per warp) and a
//   hot-ring tile 16*TG keys, so every tile moves 32*W*D bytes of K and of V.
template <int KIND, int D, int KVB>
struct Geo {
  static constexpr int W = (D >= 256) ? 4 : 8;
  static constexpr int TG = W / KVB;
  static constexpr int ESZ = cold_int8(KIND) ? 1 : 2;  // bytes of a paged / cold element
  static constexpr int ROWB = D * ESZ;                        // bytes of one (token, head) row
  static constexpr int CHN = ROWB / 128;                      // 128-byte slices of such a row
  static constexpr int CHH = D * 2 / 128;                     // slices of an f16 hot row
  static constexpr int GPW = cold_int8(KIND) ? 2 : 1;    // key groups per warp, paged/cold tile
  static constexpr int TOK = 16 * TG * GPW;                   // keys per paged / cold tile
  static constexpr int TOKH = 16 * TG;                        // keys per hot-ring tile
  static constexpr int REGION = 32 * W * D;                   // K (or V) bytes of a stage
  // Eight consumer warps share the SM with a producer warpgroup (the TMA
  // warp and three idle warps) so that registers can move between
  // warpgroups: the producer group gives up registers with setmaxnreg and
  // the consumers take them (REG_PROD / REG_CONS per thread; the launch
  // gives every warp REG_LAUNCH).  Four consumer warps need no such split.
  static constexpr bool REG_SPLIT = (W == 8);
  static constexpr int RED_PARTS = cold_int8(KIND) ? 2 : 1;  // tree-merge parts (red_parts)
  static constexpr int THREADS = REG_SPLIT ? (W + 4) * 32 : (W + 1) * 32;
  static constexpr int REG_LAUNCH = 168, REG_PROD = 72, REG_CONS = 216;
  static_assert(!REG_SPLIT || (W * REG_CONS + 4 * REG_PROD <= (W + 4) * REG_LAUNCH),
                "register split must fit in the launch's registers");
  static_assert(!REG_SPLIT || (W + 4) * 32 * REG_LAUNCH <= 65536, "launch registers");
  static_assert(W % KVB == 0, "warps per head");
  static_assert(TOK * KVB * ROWB == REGION && TOKH * KVB * D * 2 == REGION, "stage fill");
};

struct alignas(128) KParams {
  CUtensorMap tm_k;   // paged: f16 K pool; tiered: int8 cold K words (as bytes)
  CUtensorMap tm_v;
  CUtensorMap tm_kh;  // tiered: f16 hot K ring
  CUtensorMap tm_vh;

  int B, Hq, Hkv, D;
  int G;        // Hq / Hkv
  int q_len;    // query tokens per sequence (T); q, out are [B, T, Hq, D]
  int Gv;       // query rows per kv head: T * G ("virtual heads", token-major)
  int NH;       // Q-slot rows per kv head: min(Gv, kHeadTile)
  int HG;       // head groups per kv head: ceil(Gv / kHeadTile); the last may be partial
  int KVB;      // warp slots per unit (equals the instantiation's KVB)
  // A unit covers KVU kv heads x HGU head groups (KVB = KVU * HGU slots;
  // slot ks: kv head ks >> hgu_shift, head group ks & (HGU - 1)).  HGU > 1
  // lets every head group of a kv head share each K/V byte read.
  int KVU, HGU, hgu_shift;
  int HGN;      // units per kv-head block: HG / HGU
  int bs, log2_bs, max_blocks, num_blocks;
  float qscale;     // scale * log2(e): scores are kept in base-2 units
  float softcap2;   // softcap * log2(e) (0 = off)
  float softcap_inv;  // 1 / softcap2
  int window, causal;
  int stages;
  int sched;
  int grid;         // CTAs of the launch (STREAM / UNITS)
  unsigned long long wait_ns;  // time limit of every wait (abort mode after it)
  int test_skip_arm;  // test knob: CTA 0 never arms its first stage (a wait runs out)

  const float* q;
  const int* block_table;
  const int* seq_lens;
  const int* q_pos;
  float* out;
  float* lse;
  int* dev_status;

  // STREAM workspace
  float* ws_o;      // [grid][2][KVB * kHeadTile][D]
  float* ws_lse;    // [grid][2][KVB * kHeadTile]
  int* ws_cnt;      // [grid] tickets (one per CTA that starts a cut unit), zero between calls

  // SPLIT outputs
  int split_tokens, max_splits;
  float* o_part;    // [B, Hq, max_splits, D]
  float* lse_part;  // [B, Hq, max_splits]

  // tiered
  const uint16_t* k_scale;  // [NB, bs, Hkv] f16
  const uint16_t* v_scale;
  int hot_window, hot_cap;
  int hot_b0;  // sequence index of this launch's first sequence in the hot ring
  int cold_len, hot_len, hot_start;
  const int* cold_lens;
  const int* hot_lens;
  const int* hot_starts;

  // block-sparse layouts (PAGED_SPARSE): head h reads layout h % sp_nl; the
  // query at position qp reads CSR row qp >> sp_log2_block of it
  const int* sp_row_ptr;  // [sp_nl][sp_rows + 1]
  const int* sp_col_idx;  // [sp_nl][sp_nnz]
  int sp_nl;              // layouts
  int sp_nlu;             // layouts some head reads: min(sp_nl, Hq)
  int sp_rows, sp_nnz;
  int sp_log2_block;      // log2 of the keys per sparse block
  int sp_tw;              // words of a sequence's tile bitmask
  int sp_bw;              // words of a (sequence, layout) block bitmask
  int sp_words;           // words of a sequence's sparse area (sparse_words)
  int sp_max_len;         // host bound on the lengths; the bitmasks cover it
};

// Per-sequence shared-memory area of the block-sparse kind, in 32-bit words:
//   [0, tw)                 bitmask of the tiles that hold a selected key
//   [tw, 2 tw)              set bits of the tile bitmask before each word
//   [2 tw, 2 tw + nlu*bw)   per layout: bitmask of its selected key blocks
__host__ __device__ constexpr int sparse_words(int tw, int bw, int nlu) {
  return 2 * tw + nlu * bw;
}

// Per-sequence plan entries kept in shared memory (paged kernels use the
// first four fields only).
struct SeqPlan {
  int lo, hi;    // visible absolute key positions [lo, hi) (union over the query tokens)
  int qp0;       // position of query token 0
  int t0;        // first paged / cold tile
  int ntiles;    // tiles per unit
  // tiered only
  int ncold;     // cold tiles (they come first)
  int hot_start, hot_len;
  int ha0, ha1, hb0, hb1;  // hot slot tiles: [ha0, ha1) then [hb0, hb1)
  int cold_len;
};
struct SeqPlanPaged {
  int lo, hi, t0, ntiles;
};

struct SmemLayout {
  int stage_bytes;
  int off_k, off_v, off_sc;  // inside a stage
  int off_stages;            // from the 1024-aligned base
  int off_hdr;               // per-stage 16-byte headers
  int off_q;                 // one Q slot: [KVB][NH][D] f32
  int off_red;               // tree-merge buffer: [W/2][red_floats(D, RED_PARTS)] f32
  int off_plan, off_pre, off_sparse;
  int off_bar, off_misc;
  int total;  // bytes to request (includes 1 KB of alignment slack)
};

__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Floats one warp stores to hand its merge state to a partner warp: the
// O^T fragments (D/4 per lane) plus m and l of its two heads, per lane.
// Floats of one tree-merge slot: a part of the O fragments plus m and l.
__host__ __device__ constexpr int red_floats(int D, int parts) { return (D / 4 / parts + 4) * 32; }
// The int8 tiered kernels merge in two parts, so that their larger stages
// (K, V and the scale slabs) leave room for the per-sequence plan.
__host__ __device__ constexpr int red_parts(int kind) { return cold_int8(kind) ? 2 : 1; }

__host__ __device__ inline SmemLayout make_layout(int kind, int D, int KVB, int W, int region,
                                                  int tok, int NH, int Hkv, int stages, int B,
                                                  int sp_words = 0) {
  SmemLayout L;
  L.off_k = 0;
  L.off_v = region;
  L.off_sc = 2 * region;
  const int sc_bytes = cold_int8(kind) ? align_up(2 * tok * Hkv * 2, 128) : 0;
  L.stage_bytes = align_up(L.off_sc + sc_bytes, 1024);
  L.off_stages = 0;
  int off = stages * L.stage_bytes;
  L.off_hdr = off;
  off += stages * 16;
  off = align_up(off, 128);
  L.off_q = off;
  off += align_up(KVB * NH * D * 4, 128);
  L.off_red = off;
  off += (W / 2) * red_floats(D, red_parts(kind)) * 4;
  L.off_plan = off;
  off += B * (one_token_paged(kind) ? (int)sizeof(SeqPlanPaged) : (int)sizeof(SeqPlan));
  L.off_pre = off;
  off += (B + 1) * 4;
  L.off_sparse = off;
  off += B * sp_words * 4;
  off = align_up(off, 8);
  L.off_bar = off;
  off += (2 * stages + 2) * 8;  // full[stages], empty[stages], qfull, qempty
  L.off_misc = off;
  off += 64;
  L.total = off + 1024;
  return L;
}

}  // namespace da
