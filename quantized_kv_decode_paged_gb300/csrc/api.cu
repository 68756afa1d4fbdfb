// api.cu — the C ABI of libdecode_attn.so (declared in include/decode_attn.h):
// argument validation, TMA tensor-map encoding, schedule and stage sizing,
// batch chunking, and the kernel launches.  Host code only.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/decode_attn.h"
#include "kernel_params.h"
#include "launch.h"

namespace {

using da::KParams;
using da::SmemLayout;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

constexpr int kMaxDevices = 128;

// SM count of the current device, queried once per device.  Entries are
// atomics: host threads making their first call together each store the same
// value.
int device_sms(int* sms_out) {
  static std::atomic<int> sms[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DA_ERR_CUDA;
  int v = sms[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      return DA_ERR_CUDA;
    sms[dev].store(v, std::memory_order_relaxed);
  }
  *sms_out = v;
  return DA_OK;
}

// Process-wide tuning state.  Its initial values are read from the
// environment once, when the library is loaded (DA_KVB, DA_FUSE_HG, DA_PACK,
// DA_MAX_STAGES, DA_WAIT_LIMIT_MS, DA_UNSPLIT_MAX_LEN; unset or invalid values keep the
// defaults); decode_attn_set_tuning replaces them.  Every launch reads a
// snapshot of the fields.  The test hook that leaves a stage unarmed is set
// only through decode_attn_testing_skip_first_arm, never from the
// environment.
struct Tuning {
  std::atomic<int> kvb{0};         // 0 = automatic, else 1, 2 or 4
  std::atomic<int> fuse_hg{1};     // 0 = one unit per head group
  std::atomic<int> pack{1};        // 0 = two-operand kernels always
  std::atomic<int> max_stages{0};  // 0 = kMaxStages, else 2..kMaxStages
  std::atomic<int> wait_ms{2000};  // 1..10000
  std::atomic<int> unsplit_len{512};  // 0..65536 keys
  std::atomic<int> skip_arm{0};    // test hook
};

bool valid_kvb(int v) { return v == 0 || v == 1 || v == 2 || v == 4; }
bool valid_stages(int v) { return v == 0 || (v >= 2 && v <= da::kMaxStages); }
bool valid_wait(int v) { return v >= 1 && v <= 10000; }
bool valid_unsplit(int v) { return v >= 0 && v <= 65536; }

da_tuning env_tuning() {
  da_tuning t{0, 1, 1, 0, 2000, 512};
  auto env_int = [](const char* name, int* out) {
    const char* e = getenv(name);
    if (!e || !*e) return false;
    char* end = nullptr;
    const long v = strtol(e, &end, 10);
    if (*end != '\0' || v < -1000000 || v > 1000000) return false;
    *out = (int)v;
    return true;
  };
  int v = 0;
  if (env_int("DA_KVB", &v) && valid_kvb(v)) t.kv_heads_per_unit = v;
  if (env_int("DA_FUSE_HG", &v) && (v == 0 || v == 1)) t.fuse_head_groups = v;
  if (env_int("DA_PACK", &v) && (v == 0 || v == 1)) t.packed_operands = v;
  if (env_int("DA_MAX_STAGES", &v) && valid_stages(v)) t.max_stages = v;
  if (env_int("DA_WAIT_LIMIT_MS", &v) && valid_wait(v)) t.wait_limit_ms = v;
  if (env_int("DA_UNSPLIT_MAX_LEN", &v) && valid_unsplit(v)) t.unsplit_max_len = v;
  return t;
}

const da_tuning& load_time_tuning() {
  static const da_tuning t = env_tuning();
  return t;
}

Tuning& tuning() {
  static Tuning* t = [] {
    Tuning* x = new Tuning;
    const da_tuning& e = load_time_tuning();
    x->kvb = e.kv_heads_per_unit;
    x->fuse_hg = e.fuse_head_groups;
    x->pack = e.packed_operands;
    x->max_stages = e.max_stages;
    x->wait_ms = e.wait_limit_ms;
    x->unsplit_len = e.unsplit_max_len;
    return x;
  }();
  return *t;
}

// Reads the environment when the library is loaded, not at the first call.
const bool g_tuning_loaded = (tuning(), true);

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int ilog2(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

// Validation shared by every entry point that takes da_params.
int check_params(const da_params* p, bool tiered) {
  if (!p) return DA_ERR_INVALID;
  if (p->batch < 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0) return DA_ERR_INVALID;
  if (p->num_q_heads % p->num_kv_heads != 0) return DA_ERR_INVALID;
  if (p->head_dim <= 0) return DA_ERR_INVALID;
  if (tiered) {
    if (p->head_dim != 128 && p->head_dim != 256) return DA_ERR_UNSUPPORTED;
  } else {
    if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256) return DA_ERR_UNSUPPORTED;
  }
  if (p->block_size <= 0 || p->max_blocks_per_seq <= 0 || p->num_blocks <= 0)
    return DA_ERR_INVALID;
  if (!pow2(p->block_size) || p->block_size < 8 || p->block_size > 256) return DA_ERR_UNSUPPORTED;
  if ((long long)p->num_blocks * p->block_size > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
  if ((long long)p->max_blocks_per_seq * p->block_size > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
  if (!(p->scale >= 0.f) || isinf(p->scale)) return DA_ERR_INVALID;
  if (!(p->softcap >= 0.f) || isinf(p->softcap)) return DA_ERR_INVALID;
  if (p->sliding_window < 0) return DA_ERR_INVALID;
  if (p->causal != 0 && p->causal != 1) return DA_ERR_INVALID;
  if (p->max_seq_len < 0) return DA_ERR_INVALID;
  return DA_OK;
}

// 1/sqrt(D) rounded to f32 when scale is 0, then times log2(e) (the kernels
// keep scores in base-2 units).
float effective_qscale(const da_params* p) {
  const double s = p->scale > 0.f ? (double)p->scale : (double)(float)(1.0 / sqrt((double)p->head_dim));
  return (float)s * 1.4426950408889634f;
}

// The tuning state's kv heads per unit, when set, replaces the automatic
// choice if an instantiation exists and it divides Hkv.
int kvb_override(int kind, int D, int Hkv, int kvb) {
  const int v = tuning().kvb.load(std::memory_order_relaxed);
  if (v >= 1 && Hkv % v == 0 && da::decode_geo(kind, D, v).W != 0) return v;
  return kvb;
}

// Units of (kv heads x head groups).  With more than one head group per kv
// head (more than kHeadTile query rows per kv head), a unit takes all of a
// kv head's head groups when there are 2 or 4 of them: the four warp slots
// of a KVB = 4 instantiation then split as KVU kv heads x HGU head groups
// (KVU * HGU = 4) and every K/V byte serves all the kv head's query rows
// (read once instead of HG times).  The tuning state's fuse_head_groups = 0
// keeps one head group per unit.
void plan_units(KParams& k, int kind) {
  k.KVU = k.KVB;
  k.HGU = 1;
  k.hgu_shift = 0;
  k.HGN = k.HG;
  if (tuning().fuse_hg.load(std::memory_order_relaxed) == 0) return;
  if (k.HG != 2 && k.HG != 4) return;
  const int kvu = 4 / k.HG;
  if (k.Hkv % kvu != 0 || da::decode_geo(kind, k.D, 4).W == 0) return;
  k.KVB = 4;
  k.KVU = kvu;
  k.HGU = k.HG;
  k.hgu_shift = k.HG == 2 ? 1 : 2;
  k.HGN = 1;
}

// Whether to launch the packed variant: at most four query heads per kv
// head leave half of the MMA's eight columns free for the remainder parts.
// The tuning state's packed_operands = 0 forces the unpacked variant.
bool use_packed(const KParams& k) {
  if (k.NH > 4) return false;
  return tuning().pack.load(std::memory_order_relaxed) != 0;
}

// Time limit of every wait inside the kernels (the tuning state's
// wait_limit_ms), and the test hook that makes CTA 0 leave its first stage
// unarmed, so that its consumers' wait runs out and the kernel ends in abort
// mode with DA_DEV_TIMEOUT (no copy is issued for that stage and nothing
// faults).
unsigned long long wait_limit_ns() {
  return (unsigned long long)tuning().wait_ms.load(std::memory_order_relaxed) * 1000000ull;
}
int test_skip_arm() { return tuning().skip_arm.load(std::memory_order_relaxed); }

// T query tokens per sequence: T*G query rows per kv head, in head groups of
// kHeadTile (the last one may be partial).
void set_query_tokens(KParams& k, int T) {
  k.q_len = T;
  k.Gv = T * k.G;
  k.NH = k.Gv < da::kHeadTile ? k.Gv : da::kHeadTile;
  k.HG = (k.Gv + da::kHeadTile - 1) / da::kHeadTile;
}

void fill_common(KParams& k, const da_params* p) {
  k.B = p->batch;
  k.Hq = p->num_q_heads;
  k.Hkv = p->num_kv_heads;
  k.D = p->head_dim;
  k.G = p->num_q_heads / p->num_kv_heads;
  set_query_tokens(k, 1);
  k.bs = p->block_size;
  k.log2_bs = ilog2(p->block_size);
  k.max_blocks = p->max_blocks_per_seq;
  k.num_blocks = p->num_blocks;
  k.qscale = effective_qscale(p);
  k.softcap2 = p->softcap > 0.f ? p->softcap * 1.4426950408889634f : 0.f;
  k.softcap_inv = k.softcap2 > 0.f ? (float)(1.0 / (double)k.softcap2) : 0.f;
  k.window = p->sliding_window;
  k.causal = p->causal;
  k.KVB = da::decode_kvb(da::KIND_PAGED, p->head_dim, p->num_kv_heads);
  k.KVB = kvb_override(da::KIND_PAGED, p->head_dim, p->num_kv_heads, k.KVB);
  plan_units(k, da::KIND_PAGED);
  k.wait_ns = wait_limit_ns();
  k.test_skip_arm = test_skip_arm();
}

int encode_pool_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize,
                    long long D, long long heads, long long rows, int box_rows, int kvb);

// K/V pool maps of a paged / cold cache (f16, or int8 words): boxes of the
// unit's KVU kv heads.
int encode_paged_maps(KParams& k, int kind, const void* kp, const void* vp, const da_params* p) {
  const da::GeoInfo g = da::decode_geo(kind, p->head_dim, k.KVB);
  if (g.W == 0) return DA_ERR_UNSUPPORTED;
  const int box_rows = p->block_size < g.TOK ? p->block_size : g.TOK;
  const long long rows = (long long)p->num_blocks * p->block_size;
  const CUtensorMapDataType dt =
      da::cold_int8(kind) ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const int esize = da::cold_int8(kind) ? 1 : 2;
  int st = encode_pool_map(&k.tm_k, kp, dt, esize, p->head_dim, p->num_kv_heads, rows, box_rows,
                           k.KVU);
  if (st != DA_OK) return st;
  return encode_pool_map(&k.tm_v, vp, dt, esize, p->head_dim, p->num_kv_heads, rows, box_rows,
                         k.KVU);
}

// 4-D map over a paged pool [rows, Hkv, D] of esize-byte elements with the
// token dimension inside the (128-byte slice, kv head) dimensions:
//   dims {128/esize, rows, D*esize/128, Hkv}, strides {Hkv*D*esize, 128, D*esize},
//   box  {128/esize, box_rows, D*esize/128, kvb},
// so one box holds box_rows keys of kvb heads and all of D, laid out
// [head][slice][key][128 bytes] with the 128-byte swizzle.
int encode_pool_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize,
                    long long D, long long heads, long long rows, int box_rows, int kvb) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return DA_ERR_CUDA;
  const long long row_bytes = D * esize;
  cuuint64_t dims[4] = {(cuuint64_t)(128 / esize), (cuuint64_t)rows, (cuuint64_t)(row_bytes / 128),
                        (cuuint64_t)heads};
  cuuint64_t strides[3] = {(cuuint64_t)(heads * row_bytes), 128, (cuuint64_t)row_bytes};
  cuuint32_t box[4] = {(cuuint32_t)(128 / esize), (cuuint32_t)box_rows,
                       (cuuint32_t)(row_bytes / 128), (cuuint32_t)kvb};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = fn(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_CUDA;
}

// 5-D map over the hot ring [B, cap, Hkv, D] f16, token dimension inside:
//   dims {64, cap, D/64, Hkv, B}, box {64, box_rows, D/64, kvb, 1}.
int encode_ring_map(CUtensorMap* m, const void* base, long long D, long long heads, long long cap,
                    long long B, int box_rows, int kvb) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return DA_ERR_CUDA;
  cuuint64_t dims[5] = {64, (cuuint64_t)cap, (cuuint64_t)(D / 64), (cuuint64_t)heads,
                        (cuuint64_t)B};
  cuuint64_t strides[4] = {(cuuint64_t)(heads * D * 2), 128, (cuuint64_t)(D * 2),
                           (cuuint64_t)(cap * heads * D * 2)};
  cuuint32_t box[5] = {64u, (cuuint32_t)box_rows, (cuuint32_t)(D / 64), (cuuint32_t)kvb, 1u};
  cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_CUDA;
}

// Upper bound on pipeline stages: kMaxStages, or the tuning state's
// max_stages when set.
int max_stages() {
  const int v = tuning().max_stages.load(std::memory_order_relaxed);
  return v >= 2 ? v : da::kMaxStages;
}

// Largest stage count (>= 2) whose layout fits in shared memory, or 0.
// A stage holds the K and V of the unit's KVU kv heads: REGION >> hgu_shift
// bytes each.
int pick_stages(int kind, int D, int KVB, const da::GeoInfo& g, int hgu_shift, int NH, int Hkv,
                int nplan, int* smem_out, int sp_words = 0) {
  for (int s = max_stages(); s >= 2; --s) {
    SmemLayout L = da::make_layout(kind, D, KVB, g.W, g.REGION >> hgu_shift, g.TOK, NH, Hkv, s,
                                   nplan, sp_words);
    if (L.total <= da::kSmemLimit) {
      *smem_out = L.total;
      return s;
    }
  }
  return 0;
}

// Workspace: [tickets: one int per CTA][partial lse][partial o].  The ticket
// region comes first and its size depends only on the device, so a
// workspace can serve calls of any shape: only the tickets must be zero
// between calls, and every call leaves them zero.
struct WsLayout {
  size_t cnt_off, lse_off, o_off, total;
};

WsLayout ws_layout(int grid, int D, int kvb) {
  WsLayout w;
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  w.cnt_off = 0;
  w.lse_off = al((size_t)grid * 4);
  w.o_off = w.lse_off + al((size_t)grid * 2 * kvb * da::kHeadTile * 4);
  w.total = w.o_off + al((size_t)grid * 2 * kvb * da::kHeadTile * D * 4);
  return w;
}

// Warp slots per unit the workspace must serve (any cache kind, any number
// of query tokens): the chosen KVB, or up to 4 when head groups share a unit.
int ws_kvb(const da_params* p) {
  const int D = p->head_dim, H = p->num_kv_heads;
  int m = 0;
  for (int kind : {da::KIND_PAGED, da::KIND_TIERED, da::KIND_TIERED_F16, da::KIND_PAGED_MULTI,
                   da::KIND_PAGED_SPARSE}) {
    int v = kvb_override(kind, D, H, da::decode_kvb(kind, D, H));
    for (int f = 4; f > v; f /= 2)
      if (da::decode_geo(kind, D, f).W != 0) {
        v = f;
        break;
      }
    m = v > m ? v : m;
  }
  return m;
}

// Whether a call with a workspace runs whole units instead of the split
// (stream) schedule.  Splitting a short sequence costs the cross-CTA hand-off
// and merge, more than the parallel keys save while the units fill at most
// two waves of one CTA per SM.  Measured on GB300 (D = 128, 8 kv heads,
// flushed L2), with lim the tuning's unsplit_max_len (512):
// - one token: 256 keys x 64 units 24.1 -> 13.9 us, 512 keys x 16 units
//   20.5 -> 18.5 us, 256 keys x 4 units 18.0 -> 13.9 us; at 1024 keys either
//   schedule can win, at 2048 splitting wins (27.0 against 35.2 us for 16
//   units), and with 1024 units splitting wins at any length: up to lim keys;
// - two or four tokens (more work a tile and a larger merge): whole units
//   win up to 1024 keys (four tokens, 16 units: 51.5 -> 39.2 us), tie at
//   the least: up to 2 lim keys;
// - block-sparse (four local + stride layouts of 64-key blocks): whole
//   units win up to 2048 keys with 64 units (41.2 -> 37.1 us) and lose with
//   256 units (53.5 against 55.6 us) or at 4096 keys: up to 4 lim keys and
//   one unit per SM.
bool run_unsplit(int kind, const da_params* p, int units, int sms) {
  const long long lim = tuning().unsplit_len.load(std::memory_order_relaxed);
  const long long L = p->max_seq_len;
  if (L <= 0) return false;
  if (kind == da::KIND_PAGED) return L <= lim && units <= 2 * sms;
  if (kind == da::KIND_PAGED_MULTI) return L <= 2 * lim && units <= 2 * sms;
  if (kind == da::KIND_PAGED_SPARSE) return L <= 4 * lim && units <= sms;
  return false;
}

struct Launch {
  int kind;
  const da_params* p;
  void* workspace;
  size_t workspace_bytes;
};

// Runs the decode kernel over the batch in chunks of kMaxBatchPerLaunch.
// `base` holds every field except the per-chunk pointers, which
// `offset_chunk` shifts.
template <typename OffsetFn>
int run_batched(KParams& base, const Launch& lc, OffsetFn offset_chunk, cudaStream_t stream) {
  const da_params* p = lc.p;
  int sms = 0;
  int st = device_sms(&sms);
  if (st != DA_OK) return st;
  const bool use_ws = lc.workspace != nullptr;
  if (use_ws) {
    const size_t need = decode_attn_workspace_size(p);
    if (lc.workspace_bytes < need) return DA_ERR_WORKSPACE;
    if (!aligned(lc.workspace, 256)) return DA_ERR_INVALID;
  } else if (lc.workspace_bytes != 0) {
    return DA_ERR_INVALID;
  }
  const int grid_max = sms;
  const WsLayout w = ws_layout(grid_max, p->head_dim, ws_kvb(p));
  // Sequences per launch.  The per-sequence plan sits in shared memory next
  // to the pipeline stages; a launch takes at most as many sequences as
  // leave room for the stages a small batch gets (one stage fewer costs
  // more than another launch), split evenly over the launches.
  int chunk = da::kMaxBatchPerLaunch;
  {
    const da::GeoInfo g = da::decode_geo(lc.kind, base.D, base.KVB);
    if (g.W == 0) return DA_ERR_UNSUPPORTED;
    int sm_small = 0, sm_c = 0;
    int small = p->batch < 16 ? p->batch : 16;
    auto stages_for = [&](int nplan, int* sm) {
      return pick_stages(lc.kind, base.D, base.KVB, g, base.hgu_shift, base.NH, base.Hkv, nplan, sm,
                         base.sp_words);
    };
    int s_small = stages_for(small, &sm_small);
    // a per-sequence area too large for sixteen sequences (block-sparse
    // bitmasks of long sequences): fewer sequences a launch
    while (s_small == 0 && small > 1) {
      small = (small + 1) / 2;
      s_small = stages_for(small, &sm_small);
    }
    if (s_small == 0) return DA_ERR_UNSUPPORTED;
    while (chunk > small && stages_for(chunk, &sm_c) < s_small) chunk -= 8;
    if (chunk < small) chunk = small;
    const int nchunks = (p->batch + chunk - 1) / chunk;
    chunk = (p->batch + nchunks - 1) / nchunks;
  }
  for (int b0 = 0; b0 < p->batch; b0 += chunk) {
    const int nb = (p->batch - b0) < chunk ? (p->batch - b0) : chunk;
    KParams k = base;
    k.B = nb;
    offset_chunk(k, b0);
    const int units = nb * (k.Hkv / k.KVU) * k.HGN;
    const da::GeoInfo g = da::decode_geo(lc.kind, k.D, k.KVB);
    if (g.W == 0) return DA_ERR_UNSUPPORTED;
    int smem = 0;
    k.stages = pick_stages(lc.kind, k.D, k.KVB, g, k.hgu_shift, k.NH, k.Hkv, nb, &smem, k.sp_words);
    if (k.stages == 0) return DA_ERR_UNSUPPORTED;
    int grid;
    if (use_ws && !run_unsplit(lc.kind, p, units, sms)) {
      k.sched = da::SCHED_STREAM;
      grid = grid_max;
      if (p->max_seq_len > 0) {
        // never more CTAs than key tiles
        const long long tiles = (long long)units * ((p->max_seq_len + g.TOK - 1) / g.TOK + 1);
        if (tiles < grid) grid = (int)(tiles > 0 ? tiles : 1);
      }
      k.ws_o = reinterpret_cast<float*>(static_cast<char*>(lc.workspace) + w.o_off);
      k.ws_lse = reinterpret_cast<float*>(static_cast<char*>(lc.workspace) + w.lse_off);
      k.ws_cnt = reinterpret_cast<int*>(static_cast<char*>(lc.workspace) + w.cnt_off);
    } else {
      k.sched = da::SCHED_UNITS;
      grid = units < 8 * sms ? units : 8 * sms;
      if (grid < 1) grid = 1;
    }
    k.grid = grid;
    cudaError_t e = da::launch_decode(lc.kind, k.D, k.KVB, use_packed(k), k, dim3(grid), smem,
                                      stream);
    if (e != cudaSuccess) return DA_ERR_CUDA;
  }
  return DA_OK;
}

// Both tiered caches: int8 cold words with scales (KIND_TIERED) or f16 cold
// rows (KIND_TIERED_F16, k_scale = v_scale = NULL).
int tiered_impl(int kind, const da_params* p, const da_tier_params* t, const float* q,
                const uint16_t* k_hot, const uint16_t* v_hot, const void* k_cold,
                const void* v_cold, const uint16_t* k_scale, const uint16_t* v_scale,
                const int32_t* block_table, const int32_t* q_pos, float* out, float* lse,
                void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  const bool i8 = da::cold_int8(kind);
  int st = check_params(p, i8);
  if (st != DA_OK) return st;
  if (!t || !q || !k_hot || !v_hot || !k_cold || !v_cold || (i8 && (!k_scale || !v_scale)) ||
      !block_table || !out)
    return DA_ERR_INVALID;
  if (!workspace && workspace_bytes) return DA_ERR_INVALID;
  if (t->hot_window < 0 || t->hot_capacity < 1 || t->hot_capacity < t->hot_window)
    return DA_ERR_INVALID;
  if (!t->cold_lens && t->cold_len < 0) return DA_ERR_INVALID;
  if (!t->hot_starts && t->hot_start < 0) return DA_ERR_INVALID;
  if (!t->hot_lens) {
    const int limit = t->hot_window > 0 ? t->hot_window : t->hot_capacity;
    if (t->hot_len < 0 || t->hot_len > limit) return DA_ERR_INVALID;
  }
  if (!t->cold_lens && (long long)t->cold_len > (long long)p->max_blocks_per_seq * p->block_size)
    return DA_ERR_INVALID;
  if (((long long)p->block_size * p->num_kv_heads * 2) % 16 != 0) return DA_ERR_UNSUPPORTED;
  if ((long long)t->hot_capacity * p->batch > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_hot, 16) || !aligned(v_hot, 16) || !aligned(k_cold, 16) ||
      !aligned(v_cold, 16) || (i8 && (!aligned(k_scale, 16) || !aligned(v_scale, 16))) ||
      !aligned(out, 16) || !aligned(block_table, 4) || (q_pos && !aligned(q_pos, 4)) ||
      (lse && !aligned(lse, 4)) || (dev_status && !aligned(dev_status, 4)))
    return DA_ERR_INVALID;
  if (p->batch == 0) return DA_OK;
  KParams k;
  memset(&k, 0, sizeof(k));
  fill_common(k, p);
  k.KVB = kvb_override(kind, p->head_dim, p->num_kv_heads,
                       da::decode_kvb(kind, p->head_dim, p->num_kv_heads));
  plan_units(k, kind);
  st = encode_paged_maps(k, kind, k_cold, v_cold, p);
  if (st != DA_OK) return st;
  {
    const da::GeoInfo g = da::decode_geo(kind, k.D, k.KVB);
    if (g.W == 0) return DA_ERR_UNSUPPORTED;
    st = encode_ring_map(&k.tm_kh, k_hot, p->head_dim, p->num_kv_heads, t->hot_capacity,
                         p->batch, g.TOKH, k.KVU);
    if (st != DA_OK) return st;
    st = encode_ring_map(&k.tm_vh, v_hot, p->head_dim, p->num_kv_heads, t->hot_capacity,
                         p->batch, g.TOKH, k.KVU);
    if (st != DA_OK) return st;
  }
  k.dev_status = dev_status;
  k.k_scale = k_scale;
  k.v_scale = v_scale;
  k.hot_window = t->hot_window;
  k.hot_cap = t->hot_capacity;
  k.cold_len = t->cold_len;
  k.hot_len = t->hot_len;
  k.hot_start = t->hot_start;
  Launch lc{kind, p, workspace, workspace_bytes};
  const long long Hq = p->num_q_heads, D = p->head_dim, mb = p->max_blocks_per_seq;
  // The hot-ring tensor map spans the whole batch; a chunk keeps the global
  // sequence index through `hot_b0`, so the ring map is not re-encoded.
  auto off = [&](KParams& kk, int b0) {
    kk.q = q + (long long)b0 * Hq * D;
    kk.block_table = block_table + (long long)b0 * mb;
    kk.q_pos = q_pos ? q_pos + b0 : nullptr;
    kk.out = out + (long long)b0 * Hq * D;
    kk.lse = lse ? lse + (long long)b0 * Hq : nullptr;
    kk.cold_lens = t->cold_lens ? t->cold_lens + b0 : nullptr;
    kk.hot_lens = t->hot_lens ? t->hot_lens + b0 : nullptr;
    kk.hot_starts = t->hot_starts ? t->hot_starts + b0 : nullptr;
    kk.hot_b0 = b0;
  };
  return run_batched(k, lc, off, static_cast<cudaStream_t>(stream));
}

// Paged decode of T query tokens per sequence (T = 1: one-token decode).
int paged_impl(const da_params* p, int T, const float* q, const uint16_t* k_pool,
               const uint16_t* v_pool, const int32_t* block_table, const int32_t* seq_lens,
               const int32_t* q_pos, float* out, float* lse, void* workspace,
               size_t workspace_bytes, int32_t* dev_status, void* stream) {
  int st = check_params(p, false);
  if (st != DA_OK) return st;
  if (T < 1) return DA_ERR_INVALID;
  if ((long long)T * p->num_q_heads > 0x7fffffffLL / 64) return DA_ERR_UNSUPPORTED;
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out) return DA_ERR_INVALID;
  if (!workspace && workspace_bytes) return DA_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || (q_pos && !aligned(q_pos, 4)) ||
      (lse && !aligned(lse, 4)) || (dev_status && !aligned(dev_status, 4)))
    return DA_ERR_INVALID;
  if (p->batch == 0) return DA_OK;
  KParams k;
  memset(&k, 0, sizeof(k));
  fill_common(k, p);
  set_query_tokens(k, T);
  const int kind = T > 1 ? da::KIND_PAGED_MULTI : da::KIND_PAGED;
  k.KVB = kvb_override(kind, p->head_dim, p->num_kv_heads,
                       da::decode_kvb(kind, p->head_dim, p->num_kv_heads));
  plan_units(k, kind);
  st = encode_paged_maps(k, kind, k_pool, v_pool, p);
  if (st != DA_OK) return st;
  k.dev_status = dev_status;
  Launch lc{kind, p, workspace, workspace_bytes};
  const long long Hq = p->num_q_heads, D = p->head_dim, mb = p->max_blocks_per_seq;
  auto off = [&](KParams& kk, int b0) {
    kk.q = q + (long long)b0 * T * Hq * D;
    kk.block_table = block_table + (long long)b0 * mb;
    kk.seq_lens = seq_lens + b0;
    kk.q_pos = q_pos ? q_pos + b0 : nullptr;
    kk.out = out + (long long)b0 * T * Hq * D;
    kk.lse = lse ? lse + (long long)b0 * T * Hq : nullptr;
  };
  return run_batched(k, lc, off, static_cast<cudaStream_t>(stream));
}

// Block-sparse paged decode (one query token): the paged path with per-head
// key blocks from the CSR layouts.
int sparse_impl(const da_params* p, const da_sparse_layout* sl, const float* q,
                const uint16_t* k_pool, const uint16_t* v_pool, const int32_t* block_table,
                const int32_t* seq_lens, const int32_t* q_pos, float* out, float* lse,
                void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  int st = check_params(p, false);
  if (st != DA_OK) return st;
  if (!sl || !q || !k_pool || !v_pool || !block_table || !seq_lens || !out) return DA_ERR_INVALID;
  if (!sl->row_ptr || (!sl->col_idx && sl->max_nnz > 0)) return DA_ERR_INVALID;
  if (sl->num_layouts < 1 || sl->num_rows < 1 || sl->max_nnz < 0) return DA_ERR_INVALID;
  if (sl->sparse_block < 16 || sl->sparse_block > (1 << 20) || !pow2(sl->sparse_block))
    return DA_ERR_INVALID;
  if ((long long)sl->num_layouts * (sl->num_rows + 1) > 0x7fffffffLL ||
      (long long)sl->num_layouts * sl->max_nnz > 0x7fffffffLL)
    return DA_ERR_UNSUPPORTED;
  if (p->max_seq_len <= 0) return DA_ERR_INVALID;  // sizes the selection bitmasks
  if (!workspace && workspace_bytes) return DA_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || (q_pos && !aligned(q_pos, 4)) ||
      (lse && !aligned(lse, 4)) || (dev_status && !aligned(dev_status, 4)) ||
      !aligned(sl->row_ptr, 4) || (sl->col_idx && !aligned(sl->col_idx, 4)))
    return DA_ERR_INVALID;
  if (p->batch == 0) return DA_OK;
  KParams k;
  memset(&k, 0, sizeof(k));
  fill_common(k, p);
  const int kind = da::KIND_PAGED_SPARSE;
  k.KVB = kvb_override(kind, p->head_dim, p->num_kv_heads,
                       da::decode_kvb(kind, p->head_dim, p->num_kv_heads));
  plan_units(k, kind);
  st = encode_paged_maps(k, kind, k_pool, v_pool, p);
  if (st != DA_OK) return st;
  const da::GeoInfo g = da::decode_geo(kind, p->head_dim, k.KVB);
  if (g.W == 0) return DA_ERR_UNSUPPORTED;
  k.dev_status = dev_status;
  k.sp_row_ptr = sl->row_ptr;
  k.sp_col_idx = sl->col_idx;
  k.sp_nl = sl->num_layouts;
  k.sp_nlu = sl->num_layouts < p->num_q_heads ? sl->num_layouts : p->num_q_heads;
  k.sp_rows = sl->num_rows;
  k.sp_nnz = sl->max_nnz;
  k.sp_log2_block = ilog2(sl->sparse_block);
  k.sp_max_len = p->max_seq_len;
  {
    const long long tiles = ((long long)p->max_seq_len + g.TOK - 1) / g.TOK;
    long long blocks = ((long long)p->max_seq_len + sl->sparse_block - 1) / sl->sparse_block;
    if (blocks > sl->num_rows) blocks = sl->num_rows;
    k.sp_tw = (int)((tiles + 31) / 32);
    k.sp_bw = (int)((blocks + 31) / 32);
    k.sp_words = da::sparse_words(k.sp_tw, k.sp_bw, k.sp_nlu);
  }
  Launch lc{kind, p, workspace, workspace_bytes};
  const long long Hq = p->num_q_heads, D = p->head_dim, mb = p->max_blocks_per_seq;
  auto off = [&](KParams& kk, int b0) {
    kk.q = q + (long long)b0 * Hq * D;
    kk.block_table = block_table + (long long)b0 * mb;
    kk.seq_lens = seq_lens + b0;
    kk.q_pos = q_pos ? q_pos + b0 : nullptr;
    kk.out = out + (long long)b0 * Hq * D;
    kk.lse = lse ? lse + (long long)b0 * Hq : nullptr;
  };
  return run_batched(k, lc, off, static_cast<cudaStream_t>(stream));
}

}  // namespace

namespace da {

size_t workspace_ticket_bytes() {
  int sms = 0;
  if (device_sms(&sms) != DA_OK) return 0;
  return ws_layout(sms, 64, 1).lse_off;
}

}  // namespace da

extern "C" {

const char* decode_attn_status_string(int status) {
  switch (status) {
    case DA_OK: return "ok";
    case DA_ERR_INVALID: return "invalid argument";
    case DA_ERR_UNSUPPORTED: return "unsupported configuration";
    case DA_ERR_WORKSPACE: return "workspace too small";
    case DA_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

size_t decode_attn_workspace_size(const da_params* p) {
  if (check_params(p, false) != DA_OK && check_params(p, true) != DA_OK) return 0;
  int sms = 0;
  if (device_sms(&sms) != DA_OK) return 0;
  return ws_layout(sms, p->head_dim, ws_kvb(p)).total;
}

int decode_attn_get_tuning(da_tuning* t) {
  if (!t) return DA_ERR_INVALID;
  Tuning& s = tuning();
  t->kv_heads_per_unit = s.kvb.load();
  t->fuse_head_groups = s.fuse_hg.load();
  t->packed_operands = s.pack.load();
  t->max_stages = s.max_stages.load();
  t->wait_limit_ms = s.wait_ms.load();
  t->unsplit_max_len = s.unsplit_len.load();
  return DA_OK;
}

int decode_attn_set_tuning(const da_tuning* t) {
  const da_tuning& v = t ? *t : load_time_tuning();
  if (!valid_kvb(v.kv_heads_per_unit) || (v.fuse_head_groups != 0 && v.fuse_head_groups != 1) ||
      (v.packed_operands != 0 && v.packed_operands != 1) || !valid_stages(v.max_stages) ||
      !valid_wait(v.wait_limit_ms) || !valid_unsplit(v.unsplit_max_len))
    return DA_ERR_INVALID;
  Tuning& s = tuning();
  s.kvb = v.kv_heads_per_unit;
  s.fuse_hg = v.fuse_head_groups;
  s.pack = v.packed_operands;
  s.max_stages = v.max_stages;
  s.wait_ms = v.wait_limit_ms;
  s.unsplit_len = v.unsplit_max_len;
  return DA_OK;
}

int decode_attn_testing_skip_first_arm(int32_t on) {
  if (on != 0 && on != 1) return DA_ERR_INVALID;
  tuning().skip_arm = on;
  return DA_OK;
}

int decode_attn_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (!workspace && bytes) return DA_ERR_INVALID;
  if (!bytes) return DA_OK;
  return cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DA_OK
             : DA_ERR_CUDA;
}

int decode_attn_paged(const da_params* p, const float* q, const uint16_t* k_pool,
                      const uint16_t* v_pool, const int32_t* block_table,
                      const int32_t* seq_lens, const int32_t* q_pos, float* out, float* lse,
                      void* workspace, size_t workspace_bytes, int32_t* dev_status,
                      void* stream) {
  return paged_impl(p, 1, q, k_pool, v_pool, block_table, seq_lens, q_pos, out, lse, workspace,
                    workspace_bytes, dev_status, stream);
}

int decode_attn_paged_sparse(const da_params* p, const da_sparse_layout* sl, const float* q,
                             const uint16_t* k_pool, const uint16_t* v_pool,
                             const int32_t* block_table, const int32_t* seq_lens,
                             const int32_t* q_pos, float* out, float* lse, void* workspace,
                             size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return sparse_impl(p, sl, q, k_pool, v_pool, block_table, seq_lens, q_pos, out, lse, workspace,
                     workspace_bytes, dev_status, stream);
}

int decode_attn_paged_multi(const da_params* p, int32_t q_len, const float* q,
                            const uint16_t* k_pool, const uint16_t* v_pool,
                            const int32_t* block_table, const int32_t* seq_lens,
                            const int32_t* q_pos, float* out, float* lse, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return paged_impl(p, q_len, q, k_pool, v_pool, block_table, seq_lens, q_pos, out, lse,
                    workspace, workspace_bytes, dev_status, stream);
}

int decode_attn_split_partial(const da_params* p, int32_t split_tokens, int32_t max_splits,
                              const float* q, const uint16_t* k_pool, const uint16_t* v_pool,
                              const int32_t* block_table, const int32_t* seq_lens,
                              const int32_t* q_pos, float* o_part, float* lse_part,
                              int32_t* dev_status, void* stream) {
  int st = check_params(p, false);
  if (st != DA_OK) return st;
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !o_part || !lse_part)
    return DA_ERR_INVALID;
  if (split_tokens <= 0 || max_splits <= 0 || split_tokens % p->block_size != 0)
    return DA_ERR_INVALID;
  if ((long long)split_tokens * max_splits > 0x7fffffffLL) return DA_ERR_INVALID;
  if (max_splits > 65535) return DA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o_part, 4) ||
      !aligned(lse_part, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      (q_pos && !aligned(q_pos, 4)) || (dev_status && !aligned(dev_status, 4)))
    return DA_ERR_INVALID;
  if (p->batch == 0) return DA_OK;
  KParams k;
  memset(&k, 0, sizeof(k));
  fill_common(k, p);
  st = encode_paged_maps(k, da::KIND_PAGED, k_pool, v_pool, p);
  if (st != DA_OK) return st;
  k.dev_status = dev_status;
  k.sched = da::SCHED_SPLIT;
  k.split_tokens = split_tokens;
  k.max_splits = max_splits;
  const da::GeoInfo g = da::decode_geo(da::KIND_PAGED, k.D, k.KVB);
  if (g.W == 0) return DA_ERR_UNSUPPORTED;
  int smem = 0;
  k.stages = pick_stages(da::KIND_PAGED_SPLIT, k.D, k.KVB, g, k.hgu_shift, k.NH, k.Hkv, 1, &smem);
  if (k.stages == 0) return DA_ERR_UNSUPPORTED;
  const long long units_total = (long long)p->batch * (k.Hkv / k.KVU) * k.HGN;
  const long long Hq = p->num_q_heads, D = p->head_dim, mb = p->max_blocks_per_seq;
  // grid.y is limited to 65535 units per launch: chunk whole sequences
  const int upb = (k.Hkv / k.KVU) * k.HGN;
  const int seqs_per_launch = 65535 / upb > 0 ? 65535 / upb : 1;
  if (upb > 65535) return DA_ERR_UNSUPPORTED;
  (void)units_total;
  for (int b0 = 0; b0 < p->batch; b0 += seqs_per_launch) {
    const int nb = (p->batch - b0) < seqs_per_launch ? (p->batch - b0) : seqs_per_launch;
    KParams kk = k;
    kk.B = nb;
    kk.q = q + (long long)b0 * Hq * D;
    kk.block_table = block_table + (long long)b0 * mb;
    kk.seq_lens = seq_lens + b0;
    kk.q_pos = q_pos ? q_pos + b0 : nullptr;
    kk.o_part = o_part + (long long)b0 * Hq * max_splits * D;
    kk.lse_part = lse_part + (long long)b0 * Hq * max_splits;
    kk.grid = max_splits;
    cudaError_t e = da::launch_decode(da::KIND_PAGED_SPLIT, kk.D, kk.KVB, use_packed(kk), kk,
                                      dim3(max_splits, nb * upb), smem,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return DA_ERR_CUDA;
  }
  return DA_OK;
}

int decode_attn_split_merge(int32_t batch, int32_t num_q_heads, int32_t head_dim,
                            int32_t max_splits, const float* o_part, const float* lse_part,
                            float* out, float* lse, void* stream) {
  if (batch < 0 || num_q_heads <= 0 || head_dim <= 0 || max_splits <= 0) return DA_ERR_INVALID;
  if (!o_part || !lse_part || !out) return DA_ERR_INVALID;
  if ((long long)batch * num_q_heads > 0x7fffffffLL) return DA_ERR_UNSUPPORTED;
  if (batch == 0) return DA_OK;
  cudaError_t e = da::launch_split_merge(batch * num_q_heads, max_splits, head_dim, o_part,
                                         lse_part, out, lse, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

int decode_attn_tiered_int8(const da_params* p, const da_tier_params* t, const float* q,
                            const uint16_t* k_hot, const uint16_t* v_hot,
                            const uint32_t* k_cold, const uint32_t* v_cold,
                            const uint16_t* k_scale, const uint16_t* v_scale,
                            const int32_t* block_table, const int32_t* q_pos, float* out,
                            float* lse, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, void* stream) {
  return tiered_impl(da::KIND_TIERED, p, t, q, k_hot, v_hot, k_cold, v_cold, k_scale, v_scale,
                     block_table, q_pos, out, lse, workspace, workspace_bytes, dev_status, stream);
}

int decode_attn_tiered_f16(const da_params* p, const da_tier_params* t, const float* q,
                           const uint16_t* k_hot, const uint16_t* v_hot,
                           const uint16_t* k_cold, const uint16_t* v_cold,
                           const int32_t* block_table, const int32_t* q_pos, float* out,
                           float* lse, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream) {
  return tiered_impl(da::KIND_TIERED_F16, p, t, q, k_hot, v_hot, k_cold, v_cold, nullptr,
                     nullptr, block_table, q_pos, out, lse, workspace, workspace_bytes,
                     dev_status, stream);
}

}  // extern "C"
