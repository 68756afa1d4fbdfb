/*
 * decode_attn.h — C ABI of the GB300 decode-attention library
 * (libdecode_attn.so, built from quantized_kv_decode_paged_gb300/csrc).
 *
 * The operation: single-token (decode) grouped-query attention over a KV
 * cache whose pages are reached through a per-sequence block table, with an
 * optional int8 cold tier and an f16 hot ring.  For every sequence b and
 * query head h (kv head = h / (Hq/Hkv)) the library computes
 *
 *     s_t   = scale * <Q[b,h,:], K_t>           (optionally  cap*tanh(s_t/cap))
 *     out   = sum_t softmax(s)_t * V_t           over the visible keys t
 *     lse   = max_t s_t + ln sum_t exp(s_t - max_t s_t)     (natural log)
 *
 * Definitions followed:
 *   - paged layout, block_table indirection and the LSE output:
 *       boostr "paged_attention.wgsl", paged_attention_fwd_f32 (both passes
 *       and the lse store);
 *   - GQA head map, causal and sliding-window masks, softcap after scale,
 *     zero-sum guard: @simulatte/doppler 0.1.0 "attention_f16kv.wgsl",
 *     get_kv_head_idx / is_masked / the online-softmax block loop;
 *   - int8 cold tier (4 values per u32, little-endian byte lane d%4, sign
 *     extended, times one f16 scale per (token, kv head)) and the f16 hot
 *     ring (slot = (hot_start + j) % hot_window):
 *       @simulatte/doppler 0.1.0 "attention_decode_tiered_int8_f16kv.wgsl",
 *       read_cold_k / read_cold_v / get_hot_pos / main;
 *   - merge of two partial softmax states (m, d):
 *       com.microsoft.SparseAttention "sparse-attention.wgsl.jinja",
 *       combine_partials.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument that names a tensor is a DEVICE pointer of the
 *     current CUDA device, owned by the caller.  The library never frees or
 *     keeps them.  f16 data is passed as uint16_t (IEEE binary16 bits).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is asynchronous on that stream and never
 *     synchronises the host; the library allocates no device memory.
 *   - Host-detectable errors return a negative da_status before any launch
 *     and leave every output untouched.
 *   - Problems that only the device can see (a block id outside
 *     [0, num_blocks), a length beyond the table, ...) never fault: the
 *     offending keys are treated as masked (a length is clamped) and the
 *     matching DA_DEV_* bit is OR-ed into *dev_status when dev_status is
 *     non-NULL.  The caller zeroes *dev_status before the call.
 *   - Layouts (row-major, innermost last):
 *       q            f32  [B, Hq, D]
 *       k_pool/v_pool f16 [num_blocks, block_size, Hkv, D]
 *       block_table  i32  [B, max_blocks_per_seq]; logical token t of
 *                         sequence b lives in page block_table[b][t/bs] at
 *                         row t % bs
 *       seq_lens     i32  [B]
 *       q_pos        i32  [B] absolute position of the query, or NULL
 *                         (NULL: the last cached token, seq_len-1)
 *       out          f32  [B, Hq, D]
 *       lse          f32  [B, Hq] or NULL (not written)
 *   - A sequence with no visible key (seq_len 0) gets out = 0, lse = -inf.
 *   - Supported sizes: head_dim in {64, 128, 256}; num_q_heads a multiple of
 *     num_kv_heads; block_size a power of two in [8, 256]; tensor pointers
 *     16-byte aligned (index arrays 4-byte aligned).  Other sizes return
 *     DA_ERR_UNSUPPORTED.
 */
#ifndef DECODE_ATTN_H
#define DECODE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DA_OK = 0,
  DA_ERR_INVALID = -1,     /* argument out of range, NULL or misaligned  */
  DA_ERR_UNSUPPORTED = -2, /* valid request this build does not handle   */
  DA_ERR_WORKSPACE = -3,   /* workspace too small for the requested path */
  DA_ERR_CUDA = -4         /* a CUDA runtime or driver call failed       */
} da_status;

/* Bits OR-ed into *dev_status by the kernels. */
enum {
  DA_DEV_BAD_BLOCK = 1,      /* block_table entry outside [0, num_blocks): its keys are masked */
  DA_DEV_BAD_SEQ_LEN = 2,    /* length < 0 or beyond max_blocks_per_seq*block_size: clamped    */
  DA_DEV_BAD_QPOS = 4,       /* q_pos[b] < 0: the row is written as empty (out 0, lse -inf)   */
  DA_DEV_SPLIT_OVERFLOW = 8, /* split_partial: keys past max_splits*split_tokens were dropped  */
  DA_DEV_BAD_TIER = 16,      /* tiered: hot_len > ring capacity or negative tier length        */
  DA_DEV_TIMEOUT = 32        /* an internal pipeline wait ran past its time limit (never      */
                             /* expected; 2 s, or DA_WAIT_LIMIT_MS): the kernel then ends     */
                             /* without waiting further and its outputs are undefined          */
};

typedef struct {
  int32_t batch;              /* B  >= 1                                                     */
  int32_t num_q_heads;        /* Hq >= 1, multiple of num_kv_heads                           */
  int32_t num_kv_heads;       /* Hkv >= 1                                                    */
  int32_t head_dim;           /* D in {64, 128, 256}                                         */
  int32_t block_size;         /* tokens per page, power of two in [8, 256]                   */
  int32_t max_blocks_per_seq; /* columns of block_table                                      */
  int32_t num_blocks;         /* pages in the pool (valid ids are [0, num_blocks))            */
  int32_t max_seq_len;        /* host upper bound of the key lengths (sizes the launch);
                                 0 = unknown.  Larger device lengths are still correct.       */
  float scale;                /* score scale; 0 => 1/sqrt(D) rounded to f32; < 0 invalid      */
  float softcap;              /* 0 => off; > 0 => s = cap*tanh(s/cap) after scaling; < 0 invalid */
  int32_t sliding_window;     /* 0 => off; W > 0 => keys below qpos-W+1 are masked when qpos >= W */
  int32_t causal;             /* 1 => keys after qpos are masked; 0 => not                    */
} da_params;

/*
 * decode_attn_paged — f16 paged decode attention, f32 output and LSE.
 * Operation: boostr "paged_attention.wgsl" paged_attention_fwd_f32 with a
 * single query per (b, h), plus the causal / sliding-window / softcap rules
 * of doppler "attention_f16kv.wgsl" is_masked and its softcap step.
 *
 * workspace: device scratch of at least decode_attn_workspace_size(p)
 * bytes, zero-filled once before its first use (decode_attn_workspace_init
 * or cudaMemsetAsync).  Its leading ticket counters are left at zero by
 * every call, so one buffer serves later calls of any shape that fit in it.
 * With it the keys of long sequences are split across CTAs (flash-decoding)
 * and the partial results are merged inside the same launch.  Short
 * sequences are not split: when 0 < p->max_seq_len <= the tuning's
 * unsplit_max_len (512 keys by default) and the launch has at most two
 * units per SM, whole units run per CTA and the workspace is not touched
 * (da_tuning gives the bounds of the other paged entry points).
 * workspace = NULL and workspace_bytes = 0 selects the unsplit path (whole
 * (b, kv head) units per CTA).  Two calls that share a workspace must be
 * ordered (same stream or synchronised); calls that overlap on the GPU race
 * on it.
 * Returns DA_OK or a negative da_status.
 */
int decode_attn_paged(const da_params* p, const float* q, const uint16_t* k_pool,
                      const uint16_t* v_pool, const int32_t* block_table,
                      const int32_t* seq_lens, const int32_t* q_pos, float* out,
                      float* lse, void* workspace, size_t workspace_bytes,
                      int32_t* dev_status, void* stream);

/*
 * decode_attn_paged_multi — decode attention of q_len query tokens per
 * sequence (speculative or chunked decode) over the paged cache.  Token t of
 * sequence b has position q_pos[b] + t (q_pos NULL: seq_len - q_len + t, the
 * q_len new tokens being the last q_len cached keys) and applies the causal
 * and sliding-window rules at its own position (doppler
 * "attention_f16kv.wgsl" is_masked for a query tile with start_pos).
 *   q   f32 [B, q_len, Hq, D]
 *   out f32 [B, q_len, Hq, D];  lse f32 [B, q_len, Hq] or NULL
 * Everything else as for decode_attn_paged, which is the q_len = 1 case.
 * The q_len*G query rows of a kv head share every K/V byte read from HBM.
 */
int decode_attn_paged_multi(const da_params* p, int32_t q_len, const float* q,
                            const uint16_t* k_pool, const uint16_t* v_pool,
                            const int32_t* block_table, const int32_t* seq_lens,
                            const int32_t* q_pos, float* out, float* lse, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * Block-sparse layouts for decode_attn_paged_sparse, in the CSR form of
 * com.microsoft.SparseAttention "sparse-attention.wgsl.jinja" (the attention
 * pass, main): query head h reads layout h % num_layouts; the query at
 * position qpos reads row qpos / sparse_block of that layout; the row lists
 * col_idx[layout][row_ptr[layout][row] .. row_ptr[layout][row + 1]), and
 * each listed column c selects the sparse_block keys c*sparse_block ..
 * (c+1)*sparse_block - 1.  The CSR is a boolean mask: a repeated column
 * selects nothing more.  Both arrays are DEVICE pointers owned by the
 * caller and are only read.
 */
typedef struct {
  int32_t sparse_block;   /* keys per sparse block: a power of two, >= 16           */
  int32_t num_layouts;    /* >= 1                                                  */
  int32_t num_rows;       /* rows of every layout (row_ptr has num_rows + 1 per layout) */
  int32_t max_nnz;        /* column entries per layout (row offsets lie in [0, max_nnz]) */
  const int32_t* row_ptr; /* i32 [num_layouts, num_rows + 1]                        */
  const int32_t* col_idx; /* i32 [num_layouts, max_nnz]                             */
} da_sparse_layout;

/*
 * decode_attn_paged_sparse — block-sparse decode attention (one query token
 * per sequence) over the f16 paged cache.  Row (b, h) attends to the keys of
 * the blocks its layout's row selects, within the causal and sliding-window
 * bounds of decode_attn_paged at qpos (q_pos[b], or seq_len - 1).  A row
 * that selects no key gets out = 0 and lse = -inf.  Device-side problems
 * never fault: a row index past num_rows, a malformed row (start < 0,
 * end < start or end > max_nnz) and a column outside [0, num_rows) select
 * nothing and set DA_DEV_BAD_BLOCK; a length above p->max_seq_len is
 * clamped to it and sets DA_DEV_BAD_SEQ_LEN.
 * Only the pages of blocks some head selects are read, once for all the
 * query heads of a kv head.  p->max_seq_len must be > 0: it sizes the
 * selection bitmasks each CTA keeps in shared memory, and a batch whose
 * bitmasks do not fit is run in several launches.
 * Everything else (layouts, workspace, q_pos, out, lse, stream) as for
 * decode_attn_paged.  DA_ERR_INVALID for a sparse_block that is not a power
 * of two >= 16 or a layout description out of range.
 */
int decode_attn_paged_sparse(const da_params* p, const da_sparse_layout* sl, const float* q,
                             const uint16_t* k_pool, const uint16_t* v_pool,
                             const int32_t* block_table, const int32_t* seq_lens,
                             const int32_t* q_pos, float* out, float* lse, void* workspace,
                             size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * Tier geometry for decode_attn_tiered_int8 and decode_attn_tiered_f16.
 * Cold keys have absolute positions 0 .. cold_len-1 and are paged through
 * block_table (the f16 "coldPageTable" layout of doppler attention.js
 * executeAttentionTiered, applied to the int8 tier).  Hot key j
 * (0 <= j < hot_len) has absolute position hot_start + j and lives in ring
 * slot (hot_start + j) % hot_window, or slot j when hot_window = 0
 * (doppler "attention_decode_tiered_int8_f16kv.wgsl", get_hot_pos).
 * The scalar lengths apply to every sequence unless the matching device
 * array ([B] i32) is non-NULL.
 */
typedef struct {
  int32_t hot_window;   /* ring size W >= 0                                             */
  int32_t hot_capacity; /* rows per sequence in k_hot / v_hot; >= max(W, 1) and, when
                           W = 0, >= every hot_len                                     */
  int32_t cold_len;     /* used when cold_lens == NULL                                  */
  int32_t hot_len;      /* used when hot_lens == NULL                                   */
  int32_t hot_start;    /* used when hot_starts == NULL                                 */
  const int32_t* cold_lens;  /* [B] device or NULL                                      */
  const int32_t* hot_lens;   /* [B] device or NULL                                      */
  const int32_t* hot_starts; /* [B] device or NULL                                      */
} da_tier_params;

/*
 * decode_attn_tiered_int8 — decode attention over an int8 cold tier and an
 * f16 hot ring.  Operation: doppler "attention_decode_tiered_int8_f16kv.wgsl"
 * main (cold loop, hot loop, softmax, PV) batched over B and with the LSE of
 * boostr paged_attention_fwd_f32.
 *   k_hot, v_hot   f16 [B, hot_capacity, Hkv, D]
 *   k_cold, v_cold u32 [num_blocks, block_size, Hkv, D/4]: value d of a row is
 *                  the signed byte (d % 4) of word d / 4 (little endian)
 *   k_scale, v_scale f16 [num_blocks, block_size, Hkv]: cold value =
 *                  int8 * scale of its (token, kv head)
 *   block_table    i32 [B, max_blocks_per_seq] (cold pages)
 *   q_pos          i32 [B] or NULL (NULL: hot_start+hot_len-1 when hot_len > 0,
 *                  else cold_len-1)
 * p->head_dim must be 128 or 256 here.  p->max_seq_len bounds cold_len +
 * hot_len.  Workspace rules as for decode_attn_paged.
 */
int decode_attn_tiered_int8(const da_params* p, const da_tier_params* t, const float* q,
                            const uint16_t* k_hot, const uint16_t* v_hot,
                            const uint32_t* k_cold, const uint32_t* v_cold,
                            const uint16_t* k_scale, const uint16_t* v_scale,
                            const int32_t* block_table, const int32_t* q_pos, float* out,
                            float* lse, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, void* stream);

/*
 * decode_attn_tiered_f16 — decode attention over an f16 cold tier and an f16
 * hot ring: the f16 tiered layout of doppler attention.js
 * executeAttentionTiered (cold tier paged through "coldPageTable", hot tier a
 * ring), whose kernel body is not on the pages; it computes exactly what
 * decode_attn_tiered_int8 computes with the cold values read as f16.
 *   k_hot, v_hot   f16 [B, hot_capacity, Hkv, D]
 *   k_cold, v_cold f16 [num_blocks, block_size, Hkv, D] (cold pages)
 *   block_table    i32 [B, max_blocks_per_seq] (cold pages)
 * Tier geometry, q_pos, masks, output, workspace and errors as for
 * decode_attn_tiered_int8; p->head_dim may be 64, 128 or 256.
 */
int decode_attn_tiered_f16(const da_params* p, const da_tier_params* t, const float* q,
                           const uint16_t* k_hot, const uint16_t* v_hot,
                           const uint16_t* k_cold, const uint16_t* v_cold,
                           const int32_t* block_table, const int32_t* q_pos, float* out,
                           float* lse, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream);

/*
 * KV append: the step before a decode step (none of the pages prints it; the
 * layouts are the ones the decode entry points read).
 *
 * decode_attn_append_paged — writes the new token of every sequence into the
 * paged pool: k_new / v_new f16 [B, Hkv, D] go to page
 * block_table[b][pos / block_size], row pos % block_size, pos = positions[b]
 * (i32 [B], device; typically the new seq_len - 1).  A position outside
 * [0, max_blocks_per_seq * block_size) sets DA_DEV_BAD_SEQ_LEN, a page id
 * outside [0, num_blocks) DA_DEV_BAD_BLOCK; that sequence writes nothing.
 * Uses batch, num_kv_heads, head_dim, block_size, max_blocks_per_seq and
 * num_blocks of p.  Pointers to rows must be 16-byte aligned.
 */
int decode_attn_append_paged(const da_params* p, const uint16_t* k_new, const uint16_t* v_new,
                             const int32_t* positions, const int32_t* block_table,
                             uint16_t* k_pool, uint16_t* v_pool, int32_t* dev_status,
                             void* stream);

/*
 * decode_attn_append_tiered_int8 — one append step of every sequence of an
 * int8-cold / f16-hot tiered cache whose tier lengths live on the device
 * (cold_lens, hot_lens, hot_starts: i32 [B], read and updated in place).
 * With W = hot_window (> 0):
 *   - when hot_len == W, the oldest hot token (position hot_start, ring
 *     slot hot_start % W) moves to cold position cold_len, which must equal
 *     hot_start: page block_table[b][cold_len / block_size], row
 *     cold_len % block_size.  Each (token, kv head) row is quantized with
 *     scale s = f16(max|x| / 127) (f32 division) and value
 *     clamp(rint(x / s), -127, 127) (ties to even; 0 when s is 0), the
 *     symmetric int8 format the tiered decode reads.  Then cold_len += 1,
 *     hot_start += 1, hot_len -= 1;
 *   - the new token (k_new / v_new f16 [B, Hkv, D]) goes to slot
 *     (hot_start + hot_len) % W and hot_len += 1.
 * A sequence with an inconsistent state (hot_len outside [0, W], negative
 * lengths, or cold_len != hot_start with a full ring) sets DA_DEV_BAD_TIER,
 * a cold position past the table DA_DEV_BAD_SEQ_LEN, a bad page id
 * DA_DEV_BAD_BLOCK; such a sequence is left unchanged.  hot_capacity >= W
 * is the row count per sequence of k_hot / v_hot.  Buffers as for
 * decode_attn_tiered_int8.  Two calls that share the cache must be ordered.
 */
int decode_attn_append_tiered_int8(const da_params* p, int32_t hot_window, int32_t hot_capacity,
                                   const uint16_t* k_new, const uint16_t* v_new,
                                   uint16_t* k_hot, uint16_t* v_hot, uint32_t* k_cold,
                                   uint32_t* v_cold, uint16_t* k_scale, uint16_t* v_scale,
                                   const int32_t* block_table, int32_t* cold_lens,
                                   int32_t* hot_lens, int32_t* hot_starts, int32_t* dev_status,
                                   void* stream);

/*
 * decode_attn_append_tiered_f16 — as decode_attn_append_tiered_int8 for the
 * f16 cold tier (decode_attn_tiered_f16's layout): the token leaving the
 * ring is copied as f16 into its cold row.
 */
int decode_attn_append_tiered_f16(const da_params* p, int32_t hot_window, int32_t hot_capacity,
                                  const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_hot,
                                  uint16_t* v_hot, uint16_t* k_cold, uint16_t* v_cold,
                                  const int32_t* block_table, int32_t* cold_lens,
                                  int32_t* hot_lens, int32_t* hot_starts, int32_t* dev_status,
                                  void* stream);

/*
 * decode_attn_split_partial — first half of flash-decoding: split s covers
 * the visible keys of [s*split_tokens, (s+1)*split_tokens) and writes the
 * normalised partial output and its LSE:
 *   o_part   f32 [B, Hq, max_splits, D]
 *   lse_part f32 [B, Hq, max_splits]
 * A split with no visible key writes o = 0, lse = -inf.  Keys at or beyond
 * max_splits*split_tokens are not read (DA_DEV_SPLIT_OVERFLOW).
 * split_tokens must be a positive multiple of block_size.
 */
int decode_attn_split_partial(const da_params* p, int32_t split_tokens, int32_t max_splits,
                              const float* q, const uint16_t* k_pool, const uint16_t* v_pool,
                              const int32_t* block_table, const int32_t* seq_lens,
                              const int32_t* q_pos, float* o_part, float* lse_part,
                              int32_t* dev_status, void* stream);

/*
 * decode_attn_split_merge — second half: per (b, h), with M = max_s lse_s,
 *   w_s = exp(lse_s - M),  out = sum_s w_s o_s / sum_s w_s,
 *   lse = M + ln sum_s w_s;  all splits at -inf give out = 0, lse = -inf.
 * This is the pairwise (m, d) merge of com.microsoft.SparseAttention
 * combine_partials applied to max_splits states at once.
 * lse may be NULL.
 */
int decode_attn_split_merge(int32_t batch, int32_t num_q_heads, int32_t head_dim,
                            int32_t max_splits, const float* o_part, const float* lse_part,
                            float* out, float* lse, void* stream);

/*
 * decode_attn_paged_static_ws — decode_attn_paged (split path) for callers
 * that cannot allocate device memory: plugins whose host framework owns
 * every allocation, processes held to a fixed device-memory budget, loops
 * that cannot take cudaMalloc's implicit synchronisation.  The pages have no
 * counterpart for this entry point; it only changes where the scratch lives.
 *
 * The scratch is a buffer of DECODE_ATTN_STATIC_WS_BYTES bytes compiled into
 * the library (held by every GPU that loads it, until exit).  The call
 * allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 * The first call on a device looks up the buffer's device address
 * (cudaGetSymbolAddress) once per device and context.  Each
 * call clears the buffer's ticket counters on `stream` (cudaMemsetAsync)
 * and launches on `stream`; calls that overlap on the GPU share the buffer
 * and race.  Arguments, layouts, outputs and device flags are those of
 * decode_attn_paged.  Returns DA_ERR_WORKSPACE when
 * decode_attn_workspace_size(p) exceeds DECODE_ATTN_STATIC_WS_BYTES.
 */
#define DECODE_ATTN_STATIC_WS_BYTES (8u << 20)
int decode_attn_paged_static_ws(const da_params* p, const float* q, const uint16_t* k_pool,
                                const uint16_t* v_pool, const int32_t* block_table,
                                const int32_t* seq_lens, const int32_t* q_pos, float* out,
                                float* lse, int32_t* dev_status, void* stream);

/* Bytes of workspace the split path of decode_attn_paged /
 * decode_attn_tiered_int8 needs for these parameters on the current device;
 * 0 when p is invalid. */
size_t decode_attn_workspace_size(const da_params* p);

/* Zero-fills a workspace (cudaMemsetAsync on stream). */
int decode_attn_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Static text for a da_status value. */
const char* decode_attn_status_string(int status);

/*
 * Tuning of the kernel choice, process-wide.  These settings change which
 * kernel instantiation and schedule a call uses, never what it computes.
 * The pages have no counterpart; they have one kernel per variant.
 *
 * When the library is loaded, the fields are set from the environment
 * variables DA_KVB, DA_FUSE_HG, DA_PACK, DA_MAX_STAGES, DA_WAIT_LIMIT_MS and
 * DA_UNSPLIT_MAX_LEN.
 * The environment is read once, at load; unset or out-of-range values keep
 * the defaults below.  decode_attn_set_tuning replaces every field;
 * decode_attn_set_tuning(NULL) restores the load-time values.  A call that
 * runs while another host thread changes the tuning may see a mix of old and
 * new fields.  Each mix is a valid configuration.
 */
typedef struct {
  int32_t kv_heads_per_unit; /* 0 = automatic (default); 1, 2 or 4 kv heads per
                                work unit, used when a kernel exists and it
                                divides num_kv_heads */
  int32_t fuse_head_groups;  /* 1 (default): 2 or 4 head groups of 8 query rows
                                of one kv head share a unit (each K/V byte is
                                read once); 0: one unit per head group */
  int32_t packed_operands;   /* 1 (default): with at most 4 query rows per kv
                                head, the f16 and remainder parts of Q and P
                                share one MMA operand; 0: two operands */
  int32_t max_stages;        /* 0 (default): as many pipeline stages as fit in
                                shared memory; else a cap in [2, 8] */
  int32_t wait_limit_ms;     /* time limit of every wait inside the kernels,
                                [1, 10000], default 2000; a wait that runs
                                out sets DA_DEV_TIMEOUT (see the device flags) */
  int32_t unsplit_max_len;   /* keys below which a call with a workspace runs
                                whole units per CTA (no split, no merge) when
                                0 < max_seq_len <= the bound and the units fill
                                at most two waves of one CTA per SM:
                                decode_attn_paged this value,
                                decode_attn_paged_multi twice it,
                                decode_attn_paged_sparse four times it (one
                                wave); tiered calls always split.  0 = always
                                split; [0, 65536], default 512 */
} da_tuning;

/* Copies the current tuning into *t.  DA_ERR_INVALID when t is NULL. */
int decode_attn_get_tuning(da_tuning* t);

/* Replaces the tuning (NULL: the load-time values).  DA_ERR_INVALID, with
 * nothing changed, when a field is out of range. */
int decode_attn_set_tuning(const da_tuning* t);

/* Test hook, for tests of the bounded waits only: with on = 1, CTA 0 of
 * every later decode launch leaves its first pipeline stage unarmed.  Its
 * consumers' wait then runs out after wait_limit_ms.  The kernel ends in
 * abort mode with DA_DEV_TIMEOUT set and a wrong output; nothing faults.
 * on = 0 (the state at load) turns it off.  This hook is never set from the
 * environment. */
int decode_attn_testing_skip_first_arm(int32_t on);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H */
