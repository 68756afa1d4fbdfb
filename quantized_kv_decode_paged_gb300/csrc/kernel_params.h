// kernel_params.h — the parameter block the host launcher hands to the
// decode kernels, and the shared-memory layout both sides compute.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace da {

constexpr int kTile = 64;          // keys per pipeline stage
constexpr int kGroupWarps = 4;     // consumer warps of a group; each takes 16 keys of a stage
constexpr int kHeadTile = 8;       // query heads per work unit (the MMA n dimension)
constexpr int kMaxStages = 8;
constexpr int kMaxBatchPerLaunch = 256;  // per-sequence plan lives in shared memory
constexpr int kSmemLimit = 232448;       // 227 KB opt-in per block on sm_100-class parts
constexpr uint32_t kRedBarrier = 1;      // named barrier id for the consumer warps

// Consumer warps and threads of a CTA with `groups` consumer groups (group g
// takes the stages s with s % groups == g) plus one producer warp.
__host__ __device__ constexpr int consumer_warps(int groups) { return kGroupWarps * groups; }
__host__ __device__ constexpr int cta_threads(int groups) {
  return (consumer_warps(groups) + 1) * 32;
}

enum Kind : int { KIND_PAGED = 0, KIND_TIERED = 1 };
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

struct alignas(128) KParams {
  CUtensorMap tm_k;   // paged: f16 K pool; tiered: int8 cold K words (as bytes)
  CUtensorMap tm_v;
  CUtensorMap tm_kh;  // tiered: f16 hot K ring
  CUtensorMap tm_vh;

  int B, Hq, Hkv, D;
  int G;        // Hq / Hkv
  int NH;       // heads per unit: min(G, kHeadTile)
  int HG;       // head groups per kv head: ceil(G / kHeadTile)
  int bs, log2_bs, max_blocks, num_blocks;
  float qscale;     // scale * log2(e): scores are kept in base-2 units
  float softcap2;   // softcap * log2(e) (0 = off)
  int window, causal;
  int stages;
  int sched;
  int grid;         // CTAs of the launch (STREAM / UNITS)

  const float* q;
  const int* block_table;
  const int* seq_lens;
  const int* q_pos;
  float* out;
  float* lse;
  int* dev_status;

  // STREAM workspace
  float* ws_o;      // [grid][2][kHeadTile][D]
  float* ws_lse;    // [grid][2][kHeadTile]
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
};

// Per-sequence plan entries kept in shared memory.
struct SeqPlan {
  int lo, hi;    // visible absolute key positions [lo, hi)
  int t0;        // paged: first absolute tile; tiered: first cold tile
  int ntiles;    // tiles per unit
  // tiered only
  int ncold;     // cold tiles (they come first)
  int hot_start, hot_len;
  int ha0, ha1, hb0, hb1;  // hot slot tiles: [ha0, ha1) then [hb0, hb1)
  int cold_len;
};

struct SmemLayout {
  int stage_bytes;
  int off_k, off_v, off_sc, off_hdr;  // inside a stage
  int off_stages;                     // from the 1024-aligned base
  int q_slot_bytes, off_q;            // two-slot Q ring
  int off_red_o, off_red_ml;
  int off_plan, off_pre;
  int off_bar, off_misc;
  int total;  // bytes to request (includes 1 KB of alignment slack)
};

__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline SmemLayout make_layout(int kind, int D, int NH, int Hkv, int stages,
                                                  int B, int groups) {
  SmemLayout L;
  const int kv_region = kTile * D * 2;  // f16 rows (int8 cold rows use the first half)
  L.off_k = 0;
  L.off_v = kv_region;
  L.off_sc = 2 * kv_region;
  const int sc_bytes = (kind == KIND_TIERED) ? align_up(2 * kTile * Hkv * 2, 128) : 0;
  L.off_hdr = L.off_sc + sc_bytes;
  L.stage_bytes = align_up(L.off_hdr + 16, 1024);
  L.off_stages = 0;
  int off = stages * L.stage_bytes;
  L.q_slot_bytes = align_up(NH * D * 4, 128);
  L.off_q = off;
  off += 2 * L.q_slot_bytes;
  L.off_red_o = off;
  off += consumer_warps(groups) * NH * D * 4;
  L.off_red_ml = off;
  off += consumer_warps(groups) * NH * 2 * 4;
  off = align_up(off, 16);
  L.off_plan = off;
  off += B * (int)sizeof(SeqPlan);
  L.off_pre = off;
  off += (B + 1) * 4;
  off = align_up(off, 8);
  L.off_bar = off;
  off += (2 * stages + 4) * 8;  // full[stages], empty[stages], qfull[2], qempty[2]
  L.off_misc = off;
  off += 64;
  L.total = off + 1024;
  return L;
}

}  // namespace da
