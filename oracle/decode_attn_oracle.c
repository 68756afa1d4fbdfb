/*
 * decode_attn_oracle.c — reference CPU implementation of paged / tiered
 * decode attention in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  The product path
 * (the CUDA library and its Python binding) never calls it, and this file
 * shares no code, header or constant with the CUDA sources: every rule below
 * is restated here from the defining pages.
 *
 * It is deliberately plain and slow: one (sequence, query head) row at a
 * time, the keys visited in logical token order, two passes (the maximum,
 * then the exponentials, the sum and the weighted V), every value widened to
 * double before use.
 *
 * Pages followed
 *   [B] boostr "paged_attention.wgsl", paged_attention_fwd_f32: paged
 *       address ((block*block_size + offset)*Hkv + kv)*D + d, logical token t
 *       in page block_table[b][t/block_size] row t%block_size, the two-pass
 *       max / exp-sum structure and lse = ln(sum) + max.
 *   [F] @simulatte/doppler 0.1.0 "attention_f16kv.wgsl": get_kv_head_idx
 *       (kv = h / (Hq/Hkv)), is_masked (causal: key > query; window W: when
 *       query >= W, key < query - W + 1), score = scale*dot then
 *       cap*tanh(score/cap) when cap > 0, output zero when the sum is zero.
 *   [T] @simulatte/doppler 0.1.0 "attention_decode_tiered_int8_f16kv.wgsl":
 *       read_cold_k / read_cold_v (byte lane d%4 of word d/4, sign extended,
 *       times the f16 scale of (token, kv head)), get_hot_pos (slot =
 *       (hot_start + j) % hot_window, or j when hot_window = 0), absolute
 *       position of hot key j = hot_start + j.
 *   [E] @simulatte/doppler 0.1.0 "attention.js", executeAttentionTiered:
 *       the tiered cache with an f16 cold tier paged through "coldPageTable"
 *       and an f16 hot ring (its kernel body is not on the pages: the cold
 *       values are read as f16 and everything else is as in [T]).
 *   [S] com.microsoft.SparseAttention "sparse-attention.wgsl.jinja",
 *       combine_partials: m = max(m1, m2), d = d1 e^(m1-m) + d2 e^(m2-m),
 *       used here in its log-sum-exp form for the split merge; and the
 *       attention pass (main): head h reads layout h % NUM_LAYOUT, the query
 *       at position q reads CSR row q / SPARSE_BLOCK of that layout, each
 *       listed column c selects the SPARSE_BLOCK keys c*SPARSE_BLOCK .., the
 *       CSR is a boolean block mask (a repeated column selects nothing
 *       more), and causality bounds the keys at the query's position.
 *
 * Readings where the pages are silent (each also listed in the design
 * notes): the query position defaults to the last cached key; a row with no
 * visible key gives out = 0 and lse = -inf; a block id outside
 * [0, num_blocks) masks its keys and raises flag 1; a length beyond the
 * block table is clamped (flag 2); q_pos < 0 empties the row (flag 4); keys
 * past the last split are dropped (flag 8); a bad tier length is clamped
 * (flag 16).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_FLAG_BAD_BLOCK 1
#define ORACLE_FLAG_BAD_SEQ_LEN 2
#define ORACLE_FLAG_BAD_QPOS 4
#define ORACLE_FLAG_SPLIT_OVERFLOW 8
#define ORACLE_FLAG_BAD_TIER 16

/* ------------------------------------------------------------------ */
/* IEEE binary16 -> double, written out from the format definition:   */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.            */
/* ------------------------------------------------------------------ */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
  }
  return sign ? -v : v;
}

/* [T] read_cold_k: byte lane i of a little-endian u32, two's complement. */
void oracle_unpack_int8_word(uint32_t word, int32_t out[4]) {
  for (int lane = 0; lane < 4; ++lane) {
    int32_t raw = (int32_t)((word >> (8 * lane)) & 0xffu);
    out[lane] = raw >= 128 ? raw - 256 : raw;
  }
}

/* Default score scale: 1/sqrt(D) rounded to f32, then widened. */
static double effective_scale(double scale, int64_t head_dim) {
  if (scale > 0.0) return scale;
  float s = (float)(1.0 / sqrt((double)head_dim));
  return (double)s;
}

/* [F] is_masked, with positions as signed 64-bit integers. */
static int key_visible(int64_t key, int64_t qpos, int64_t causal, int64_t window) {
  if (causal && key > qpos) return 0;
  if (window > 0 && qpos >= window && key < qpos - window + 1) return 0;
  return 1;
}

static double apply_softcap(double s, double cap) {
  if (cap > 0.0) return cap * tanh(s / cap);
  return s;
}

/*
 * Two-pass softmax over n scores s[0..n) with value rows fetched through
 * `vrow`; writes out[D] and *lse.  [B] first pass = max, second = exp, sum
 * and weighted V; [F] zero output when nothing is visible.
 */
typedef void (*value_fetch_fn)(const void* ctx, int64_t key_index, double* v);

static void softmax_two_pass(const double* s, int64_t n, int64_t D, value_fetch_fn vrow,
                             const void* ctx, double* vbuf, double* out, double* lse) {
  for (int64_t d = 0; d < D; ++d) out[d] = 0.0;
  if (n == 0) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int64_t i = 0; i < n; ++i)
    if (s[i] > m) m = s[i];
  double l = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double w = exp(s[i] - m);
    l += w;
    vrow(ctx, i, vbuf);
    for (int64_t d = 0; d < D; ++d) out[d] += w * vbuf[d];
  }
  for (int64_t d = 0; d < D; ++d) out[d] /= l;
  *lse = m + log(l);
}

/* ================================================================== */
/* Paged f16 decode                                                   */
/* ================================================================== */
typedef struct {
  int64_t B, Hq, Hkv, D, block_size, max_blocks, num_blocks;
  double scale;   /* the f32 argument widened; 0 => 1/sqrt(D) */
  double softcap; /* 0 => off */
  int64_t window, causal;
  const float* q;            /* [B, Hq, D] */
  const uint16_t* k_pool;    /* [NB, bs, Hkv, D] f16 bits */
  const uint16_t* v_pool;    /* [NB, bs, Hkv, D] f16 bits */
  const int32_t* block_table;/* [B, max_blocks] */
  const int32_t* seq_lens;   /* [B] */
  const int32_t* q_pos;      /* [B] or NULL: position of query token 0 */
  int64_t q_len;             /* query tokens per sequence (q is [B, q_len, Hq, D]); 0 => 1 */
} oracle_paged_args;

typedef struct {
  const oracle_paged_args* a;
  const int64_t* rowaddr; /* element offset of each visible key's V row */
} paged_vctx;

static void paged_fetch_v(const void* ctx, int64_t i, double* v) {
  const paged_vctx* c = (const paged_vctx*)ctx;
  const uint16_t* row = c->a->v_pool + c->rowaddr[i];
  for (int64_t d = 0; d < c->a->D; ++d) v[d] = oracle_half_to_double(row[d]);
}

/* Sequence length after the [B]-style bounds rule; sets flags. */
static int64_t paged_len(const oracle_paged_args* a, int64_t b, int32_t* flags) {
  int64_t L = a->seq_lens[b];
  int64_t cap = a->max_blocks * a->block_size;
  if (L < 0) {
    *flags |= ORACLE_FLAG_BAD_SEQ_LEN;
    L = 0;
  }
  if (L > cap) {
    *flags |= ORACLE_FLAG_BAD_SEQ_LEN;
    L = cap;
  }
  return L;
}

/*
 * One row (b, query token tq, head h) restricted to keys in [t_begin, t_end)
 * (the whole sequence for a plain call, one split's range for a split call).
 * With T query tokens per sequence, token tq has position base + tq, where
 * base is q_pos[b] or, by default, L - T (the T new tokens are the last T
 * cached keys); each token applies the causal and window rules at its own
 * position.
 */
static void paged_row(const oracle_paged_args* a, int64_t b, int64_t tq, int64_t h,
                      int64_t t_begin, int64_t t_end, double* out, double* lse, int32_t* flags) {
  const int64_t D = a->D;
  const int64_t G = a->Hq / a->Hkv;
  const int64_t kv = h / G;
  const int64_t T = a->q_len > 1 ? a->q_len : 1;
  const double scale = effective_scale(a->scale, D);
  int64_t L = paged_len(a, b, flags);
  int64_t qpos = L - T + tq;
  if (a->q_pos) {
    qpos = a->q_pos[b];
    if (qpos < 0) {
      *flags |= ORACLE_FLAG_BAD_QPOS;
      L = 0;
    }
    qpos += tq;
  }
  if (t_end > L) t_end = L;
  if (t_begin < 0) t_begin = 0;
  int64_t n_max = t_end > t_begin ? t_end - t_begin : 0;
  double* s = (double*)malloc(sizeof(double) * (size_t)(n_max + 1));
  int64_t* rowaddr = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_max + 1));
  double* vbuf = (double*)malloc(sizeof(double) * (size_t)D);
  const float* qrow = a->q + ((b * T + tq) * a->Hq + h) * D;
  int64_t n = 0;
  for (int64_t t = t_begin; t < t_end; ++t) {
    if (!key_visible(t, qpos, a->causal, a->window)) continue;
    int64_t blk = a->block_table[b * a->max_blocks + t / a->block_size];
    if (blk < 0 || blk >= a->num_blocks) {
      *flags |= ORACLE_FLAG_BAD_BLOCK;
      continue;
    }
    int64_t addr = ((blk * a->block_size + t % a->block_size) * a->Hkv + kv) * D;
    const uint16_t* krow = a->k_pool + addr;
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += (double)qrow[d] * oracle_half_to_double(krow[d]);
    s[n] = apply_softcap(scale * dot, a->softcap);
    rowaddr[n] = addr;
    ++n;
  }
  paged_vctx ctx = {a, rowaddr};
  softmax_two_pass(s, n, D, paged_fetch_v, &ctx, vbuf, out, lse);
  free(s);
  free(rowaddr);
  free(vbuf);
}

/* ================================================================== */
/* Block-sparse selection of key blocks [S]                            */
/* ================================================================== */
typedef struct {
  int64_t sparse_block; /* keys per sparse block (SPARSE_BLOCK) */
  int64_t num_layouts;  /* NUM_LAYOUT */
  int64_t num_rows;     /* rows of each layout's CSR (row_ptr has num_rows + 1 entries) */
  int64_t max_nnz;      /* column entries of each layout (COL_STRIDE) */
  const int32_t* row_ptr; /* [num_layouts, num_rows + 1] */
  const int32_t* col_idx; /* [num_layouts, max_nnz] */
} oracle_sparse_layout;

/*
 * selected[c] = 1 when key block c is listed in CSR row `row` of layout
 * `layout`, for c in [0, num_rows).  A row index outside the layout, a
 * malformed row (start < 0, end < start or end > max_nnz) and a column id
 * outside [0, num_rows) raise flag 1 and select nothing.
 */
static void sparse_row_blocks(const oracle_sparse_layout* sl, int64_t layout, int64_t row,
                              unsigned char* selected, int32_t* flags) {
  for (int64_t c = 0; c < sl->num_rows; ++c) selected[c] = 0;
  if (row < 0 || row >= sl->num_rows) {
    *flags |= ORACLE_FLAG_BAD_BLOCK;
    return;
  }
  const int32_t* rp = sl->row_ptr + layout * (sl->num_rows + 1);
  int64_t start = rp[row], end = rp[row + 1];
  if (start < 0 || end < start || end > sl->max_nnz) {
    *flags |= ORACLE_FLAG_BAD_BLOCK;
    return;
  }
  const int32_t* cols = sl->col_idx + layout * sl->max_nnz;
  for (int64_t e = start; e < end; ++e) {
    int64_t c = cols[e];
    if (c < 0 || c >= sl->num_rows) {
      *flags |= ORACLE_FLAG_BAD_BLOCK;
      continue;
    }
    selected[c] = 1;
  }
}

/*
 * Block-sparse paged decode, one query token: row (b, h) takes the paged
 * row of paged_row over the keys whose sparse block is selected by CSR row
 * qpos / sparse_block of layout h % num_layouts (qpos: q_pos[b] or
 * seq_len - 1).  A query position that is negative empties the row (flag
 * 4) before any layout row is read.
 */
static void sparse_paged_row(const oracle_paged_args* a, const oracle_sparse_layout* sl,
                             int64_t b, int64_t h, double* out, double* lse, int32_t* flags) {
  const int64_t D = a->D;
  const int64_t G = a->Hq / a->Hkv;
  const int64_t kv = h / G;
  const double scale = effective_scale(a->scale, D);
  int64_t L = paged_len(a, b, flags);
  int64_t qpos = L - 1;
  if (a->q_pos) {
    qpos = a->q_pos[b];
    if (qpos < 0) {
      *flags |= ORACLE_FLAG_BAD_QPOS;
      L = 0;
    }
  }
  unsigned char* selected = (unsigned char*)malloc((size_t)(sl->num_rows + 1));
  if (L > 0) {
    sparse_row_blocks(sl, h % sl->num_layouts, qpos / sl->sparse_block, selected, flags);
  } else {
    for (int64_t c = 0; c < sl->num_rows; ++c) selected[c] = 0;
  }
  double* s = (double*)malloc(sizeof(double) * (size_t)(L + 1));
  int64_t* rowaddr = (int64_t*)malloc(sizeof(int64_t) * (size_t)(L + 1));
  double* vbuf = (double*)malloc(sizeof(double) * (size_t)D);
  const float* qrow = a->q + (b * a->Hq + h) * D;
  int64_t n = 0;
  for (int64_t t = 0; t < L; ++t) {
    if (!key_visible(t, qpos, a->causal, a->window)) continue;
    int64_t c = t / sl->sparse_block;
    if (c >= sl->num_rows || !selected[c]) continue;
    int64_t blk = a->block_table[b * a->max_blocks + t / a->block_size];
    if (blk < 0 || blk >= a->num_blocks) {
      *flags |= ORACLE_FLAG_BAD_BLOCK;
      continue;
    }
    int64_t addr = ((blk * a->block_size + t % a->block_size) * a->Hkv + kv) * D;
    const uint16_t* krow = a->k_pool + addr;
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += (double)qrow[d] * oracle_half_to_double(krow[d]);
    s[n] = apply_softcap(scale * dot, a->softcap);
    rowaddr[n] = addr;
    ++n;
  }
  paged_vctx ctx = {a, rowaddr};
  softmax_two_pass(s, n, D, paged_fetch_v, &ctx, vbuf, out, lse);
  free(selected);
  free(s);
  free(rowaddr);
  free(vbuf);
}

/* rows: flat row ids r = b*Hq + h (NULL => all); out [nrows, D], lse [nrows]. */
int32_t oracle_decode_paged_sparse(const oracle_paged_args* a, const oracle_sparse_layout* sl,
                                   const int64_t* rows, int64_t nrows, double* out,
                                   double* lse) {
  int32_t flags = 0;
  if (!rows) nrows = a->B * a->Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : flags)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t r = rows ? rows[i] : i;
    int32_t f = 0;
    sparse_paged_row(a, sl, r / a->Hq, r % a->Hq, out + i * a->D, lse + i, &f);
    flags |= f;
  }
  return flags;
}

/*
 * rows: flat row ids r = (b*T + tq)*Hq + h (NULL => all B*T*Hq rows in order).
 * out: [nrows, D]; lse: [nrows].  Returns the OR of the flags.
 */
int32_t oracle_decode_paged(const oracle_paged_args* a, const int64_t* rows, int64_t nrows,
                            double* out, double* lse) {
  int32_t flags = 0;
  const int64_t T = a->q_len > 1 ? a->q_len : 1;
  if (!rows) nrows = a->B * T * a->Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : flags)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t r = rows ? rows[i] : i;
    int64_t bt = r / a->Hq, h = r % a->Hq;
    int32_t f = 0;
    paged_row(a, bt / T, bt % T, h, 0, INT64_MAX, out + i * a->D, lse + i, &f);
    flags |= f;
  }
  return flags;
}

/*
 * Split partials: split s of row r covers keys [s*split_tokens,
 * (s+1)*split_tokens).  o_part: [nrows, max_splits, D]; lse_part:
 * [nrows, max_splits].  Visible keys at or past max_splits*split_tokens
 * raise flag 8 and are left out.
 */
int32_t oracle_decode_paged_split(const oracle_paged_args* a, int64_t split_tokens,
                                  int64_t max_splits, const int64_t* rows, int64_t nrows,
                                  double* o_part, double* lse_part) {
  int32_t flags = 0;
  if (!rows) nrows = a->B * a->Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : flags)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t r = rows ? rows[i] : i;
    int64_t b = r / a->Hq, h = r % a->Hq;
    int32_t f = 0;
    for (int64_t sp = 0; sp < max_splits; ++sp) {
      int64_t t0 = sp * split_tokens, t1 = t0 + split_tokens;
      paged_row(a, b, 0, h, t0, t1, o_part + (i * max_splits + sp) * a->D,
                lse_part + i * max_splits + sp, &f);
    }
    /* keys beyond the last split: any visible one raises the flag */
    double tail_lse;
    double* tail = (double*)malloc(sizeof(double) * (size_t)a->D);
    int32_t ftail = 0;
    paged_row(a, b, 0, h, max_splits * split_tokens, INT64_MAX, tail, &tail_lse, &ftail);
    if (tail_lse > -INFINITY) f |= ORACLE_FLAG_SPLIT_OVERFLOW;
    free(tail);
    flags |= f;
  }
  return flags;
}

/*
 * [S] merge of S partial states per row in log-sum-exp form:
 * M = max lse_s, w_s = e^(lse_s - M), out = sum w_s o_s / sum w_s,
 * lse = M + ln sum w_s; all -inf => out 0, lse -inf.
 */
void oracle_split_merge(int64_t nrows, int64_t max_splits, int64_t D, const double* o_part,
                        const double* lse_part, double* out, double* lse) {
  for (int64_t i = 0; i < nrows; ++i) {
    double M = -INFINITY;
    for (int64_t sp = 0; sp < max_splits; ++sp)
      if (lse_part[i * max_splits + sp] > M) M = lse_part[i * max_splits + sp];
    for (int64_t d = 0; d < D; ++d) out[i * D + d] = 0.0;
    if (M == -INFINITY) {
      lse[i] = -INFINITY;
      continue;
    }
    double wsum = 0.0;
    for (int64_t sp = 0; sp < max_splits; ++sp) {
      double ls = lse_part[i * max_splits + sp];
      if (ls == -INFINITY) continue;
      double w = exp(ls - M);
      wsum += w;
      for (int64_t d = 0; d < D; ++d) out[i * D + d] += w * o_part[(i * max_splits + sp) * D + d];
    }
    for (int64_t d = 0; d < D; ++d) out[i * D + d] /= wsum;
    lse[i] = M + log(wsum);
  }
}

/* ================================================================== */
/* Tiered decode: int8 [T] or f16 [E] cold pages + f16 hot ring       */
/* ================================================================== */
typedef struct {
  int64_t B, Hq, Hkv, D, block_size, max_blocks, num_blocks;
  double scale, softcap;
  int64_t window, causal;
  int64_t hot_window, hot_capacity;
  const float* q;             /* [B, Hq, D] */
  const uint16_t* k_hot;      /* [B, cap, Hkv, D] f16 bits */
  const uint16_t* v_hot;
  const uint32_t* k_cold;     /* [NB, bs, Hkv, D/4] */
  const uint32_t* v_cold;
  const uint16_t* k_scale;    /* [NB, bs, Hkv] f16 bits */
  const uint16_t* v_scale;
  const int32_t* block_table; /* [B, max_blocks] (cold pages) */
  const int32_t* cold_lens;   /* [B] */
  const int32_t* hot_lens;    /* [B] */
  const int32_t* hot_starts;  /* [B] */
  const int32_t* q_pos;       /* [B] or NULL */
  /* [E] f16 cold tier instead of the int8 words and scales (NULL for [T]) */
  const uint16_t* k_cold_f16; /* [NB, bs, Hkv, D] f16 bits */
  const uint16_t* v_cold_f16;
} oracle_tiered_args;

/* A visible key of the tiered cache: cold (page row) or hot (ring row). */
typedef struct {
  int is_hot;
  int64_t row; /* cold: blk*bs + off; hot: b*cap + slot */
} tiered_key;

typedef struct {
  const oracle_tiered_args* a;
  const tiered_key* keys;
  int64_t kv;
} tiered_vctx;

/* [T] read_cold_v / hot V read for key i, dequantised to double. */
static void tiered_fetch_v(const void* ctx, int64_t i, double* v) {
  const tiered_vctx* c = (const tiered_vctx*)ctx;
  const oracle_tiered_args* a = c->a;
  const int64_t D = a->D;
  tiered_key k = c->keys[i];
  if (k.is_hot) {
    const uint16_t* row = a->v_hot + (k.row * a->Hkv + c->kv) * D;
    for (int64_t d = 0; d < D; ++d) v[d] = oracle_half_to_double(row[d]);
  } else if (a->v_cold_f16) {
    const uint16_t* row = a->v_cold_f16 + (k.row * a->Hkv + c->kv) * D;
    for (int64_t d = 0; d < D; ++d) v[d] = oracle_half_to_double(row[d]);
  } else {
    const uint32_t* words = a->v_cold + (k.row * a->Hkv + c->kv) * (D / 4);
    double sc = oracle_half_to_double(a->v_scale[k.row * a->Hkv + c->kv]);
    for (int64_t w = 0; w < D / 4; ++w) {
      int32_t vals[4];
      oracle_unpack_int8_word(words[w], vals);
      for (int lane = 0; lane < 4; ++lane) v[4 * w + lane] = (double)vals[lane] * sc;
    }
  }
}

static void tiered_row(const oracle_tiered_args* a, int64_t b, int64_t h, double* out,
                       double* lse, int32_t* flags) {
  const int64_t D = a->D;
  const int64_t G = a->Hq / a->Hkv;
  const int64_t kv = h / G;
  const double scale = effective_scale(a->scale, D);
  int64_t cold_len = a->cold_lens[b];
  int64_t hot_len = a->hot_lens[b];
  int64_t hot_start = a->hot_starts[b];
  if (cold_len < 0) {
    *flags |= ORACLE_FLAG_BAD_TIER;
    cold_len = 0;
  }
  if (cold_len > a->max_blocks * a->block_size) {
    *flags |= ORACLE_FLAG_BAD_SEQ_LEN;
    cold_len = a->max_blocks * a->block_size;
  }
  int64_t hot_limit = a->hot_window > 0 ? a->hot_window : a->hot_capacity;
  if (hot_len < 0) {
    *flags |= ORACLE_FLAG_BAD_TIER;
    hot_len = 0;
  }
  if (hot_len > hot_limit) {
    *flags |= ORACLE_FLAG_BAD_TIER;
    hot_len = hot_limit;
  }
  if (hot_start < 0) {
    *flags |= ORACLE_FLAG_BAD_TIER;
    hot_start = 0;
  }
  int64_t qpos = hot_len > 0 ? hot_start + hot_len - 1 : cold_len - 1;
  int empty = 0;
  if (a->q_pos) {
    qpos = a->q_pos[b];
    if (qpos < 0) {
      *flags |= ORACLE_FLAG_BAD_QPOS;
      empty = 1;
    }
  }
  int64_t n_max = cold_len + hot_len;
  double* s = (double*)malloc(sizeof(double) * (size_t)(n_max + 1));
  tiered_key* keys = (tiered_key*)malloc(sizeof(tiered_key) * (size_t)(n_max + 1));
  double* vbuf = (double*)malloc(sizeof(double) * (size_t)D);
  const float* qrow = a->q + (b * a->Hq + h) * D;
  int64_t n = 0;
  /* cold keys, absolute position t */
  for (int64_t t = 0; t < cold_len && !empty; ++t) {
    if (!key_visible(t, qpos, a->causal, a->window)) continue;
    int64_t blk = a->block_table[b * a->max_blocks + t / a->block_size];
    if (blk < 0 || blk >= a->num_blocks) {
      *flags |= ORACLE_FLAG_BAD_BLOCK;
      continue;
    }
    int64_t row = blk * a->block_size + t % a->block_size;
    double dot = 0.0;
    if (a->k_cold_f16) {
      const uint16_t* krow = a->k_cold_f16 + (row * a->Hkv + kv) * D;
      for (int64_t d = 0; d < D; ++d) dot += (double)qrow[d] * oracle_half_to_double(krow[d]);
    } else {
      const uint32_t* words = a->k_cold + (row * a->Hkv + kv) * (D / 4);
      double sc = oracle_half_to_double(a->k_scale[row * a->Hkv + kv]);
      for (int64_t w = 0; w < D / 4; ++w) {
        int32_t vals[4];
        oracle_unpack_int8_word(words[w], vals);
        for (int lane = 0; lane < 4; ++lane)
          dot += (double)qrow[4 * w + lane] * ((double)vals[lane] * sc);
      }
    }
    s[n] = apply_softcap(scale * dot, a->softcap);
    keys[n].is_hot = 0;
    keys[n].row = row;
    ++n;
  }
  /* hot keys, absolute position hot_start + j, ring slot per get_hot_pos */
  for (int64_t j = 0; j < hot_len && !empty; ++j) {
    int64_t pos = hot_start + j;
    if (!key_visible(pos, qpos, a->causal, a->window)) continue;
    int64_t slot = a->hot_window > 0 ? pos % a->hot_window : j;
    int64_t row = b * a->hot_capacity + slot;
    const uint16_t* krow = a->k_hot + (row * a->Hkv + kv) * D;
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += (double)qrow[d] * oracle_half_to_double(krow[d]);
    s[n] = apply_softcap(scale * dot, a->softcap);
    keys[n].is_hot = 1;
    keys[n].row = row;
    ++n;
  }
  tiered_vctx ctx = {a, keys, kv};
  softmax_two_pass(s, n, D, tiered_fetch_v, &ctx, vbuf, out, lse);
  free(s);
  free(keys);
  free(vbuf);
}

int32_t oracle_decode_tiered(const oracle_tiered_args* a, const int64_t* rows, int64_t nrows,
                             double* out, double* lse) {
  int32_t flags = 0;
  if (!rows) nrows = a->B * a->Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : flags)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t r = rows ? rows[i] : i;
    int64_t b = r / a->Hq, h = r % a->Hq;
    int32_t f = 0;
    tiered_row(a, b, h, out + i * a->D, lse + i, &f);
    flags |= f;
  }
  return flags;
}

/* ================================================================== */
/* KV append and int8 demotion (the steps either side of decode: the  */
/* layouts of [T] and [E]; the demotion quantizer is the one the      */
/* tiered workload's inputs are made with, scale = max|x|/127)         */
/* ================================================================== */

/* binary16 encoding of an f32 value, round to nearest even, written out
 * from the format definition.  Values are handled exactly in double. */
uint16_t oracle_float_to_half(float f) {
  uint32_t bits;
  memcpy(&bits, &f, sizeof bits);
  const uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
  if ((bits & 0x7f800000u) == 0x7f800000u)
    return (uint16_t)(sign | ((bits & 0x007fffffu) ? 0x7e00u : 0x7c00u));
  const double a = fabs((double)f);
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u); /* past max + half an ulp */
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: multiples of 2^-24; 1024 of them is the smallest normal */
    const double r = rint(a / ldexp(1.0, -24));
    return (uint16_t)(sign | (uint16_t)r);
  }
  int e2;
  frexp(a, &e2);
  int e = e2 - 1; /* 2^e <= a < 2^(e+1) */
  double r = rint(a / ldexp(1.0, e - 10)); /* 1024 .. 2048 */
  if (r == 2048.0) {
    r = 1024.0;
    e += 1;
  }
  return (uint16_t)(sign | (uint16_t)(((e + 15) << 10) | ((int)r - 1024)));
}

/* Element-wise oracle_float_to_half over an array. */
void oracle_float_to_half_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_float_to_half(x[i]);
}

/* Quantizer of one (token, kv head) row of n f16 values: s16 = f16(m / 127)
 * with m = max|x| and the division in f32; code = rint(x / f32(s16)) (ties
 * to even, f32 division) clamped to [-127, 127]; code 0 when s16 is 0 or the
 * ratio is not a number.  Codes are written as int8. */
void oracle_quantize_row_int8(const uint16_t* x, int64_t n, int8_t* code, uint16_t* scale) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    const float v = (float)oracle_half_to_double(x[i]);
    const float av = fabsf(v);
    if (av > m) m = av;
  }
  const float sf = m / 127.0f;
  const uint16_t s16 = oracle_float_to_half(sf);
  const float s = (float)oracle_half_to_double(s16);
  for (int64_t i = 0; i < n; ++i) {
    int c = 0;
    if (s != 0.0f) {
      const float r = (float)oracle_half_to_double(x[i]) / s;
      if (r == r) {
        float t = rintf(r);
        if (t > 127.0f) t = 127.0f;
        if (t < -127.0f) t = -127.0f;
        c = (int)t;
      }
    }
    code[i] = (int8_t)c;
  }
  *scale = s16;
}

typedef struct {
  int64_t B, Hkv, D, block_size, max_blocks, num_blocks, hot_window, hot_capacity;
  const uint16_t* k_new;      /* [B, Hkv, D] f16 bits */
  const uint16_t* v_new;
  uint16_t* k_hot;            /* [B, cap, Hkv, D] */
  uint16_t* v_hot;
  uint32_t* k_cold;           /* int8 tier: [NB, bs, Hkv, D/4] words, or NULL */
  uint32_t* v_cold;
  uint16_t* k_scale;          /* int8 tier: [NB, bs, Hkv] */
  uint16_t* v_scale;
  uint16_t* k_cold_f16;       /* f16 tier: [NB, bs, Hkv, D], or NULL */
  uint16_t* v_cold_f16;
  const int32_t* block_table; /* [B, max_blocks] (cold pages) */
  int32_t* cold_lens;         /* [B], updated */
  int32_t* hot_lens;
  int32_t* hot_starts;
} oracle_append_args;

static void demote_row(const oracle_append_args* a, const uint16_t* hot, uint32_t* words,
                       uint16_t* scales, uint16_t* f16rows, int64_t hot_row, int64_t cold_row) {
  const int64_t D = a->D;
  for (int64_t kv = 0; kv < a->Hkv; ++kv) {
    const uint16_t* x = hot + (hot_row * a->Hkv + kv) * D;
    if (f16rows) {
      memcpy(f16rows + (cold_row * a->Hkv + kv) * D, x, sizeof(uint16_t) * (size_t)D);
      continue;
    }
    int8_t code[1024]; /* D <= 1024 (checked by the caller) */
    uint16_t s16;
    oracle_quantize_row_int8(x, D, code, &s16);
    for (int64_t w = 0; w < D / 4; ++w) {
      uint32_t word = 0;
      for (int lane = 0; lane < 4; ++lane)
        word |= (uint32_t)(uint8_t)code[4 * w + lane] << (8 * lane);
      words[(cold_row * a->Hkv + kv) * (D / 4) + w] = word;
    }
    scales[cold_row * a->Hkv + kv] = s16;
  }
}

/* One append step of every sequence of a tiered cache (ring of W slots):
 *  - when the ring holds W tokens, the oldest (position hot_start, slot
 *    hot_start % W) moves to the cold tier at position cold_len, which must
 *    equal hot_start (contiguous tiers): page block_table[b][cold_len/bs],
 *    row cold_len % bs; int8 tier: quantized as above; f16 tier: copied;
 *    cold_len += 1, hot_start += 1, hot_len -= 1;
 *  - the new token goes to slot (hot_start + hot_len) % W; hot_len += 1.
 * A sequence whose state is inconsistent (flag 16), whose cold position is
 * past the block table (flag 2) or whose page id is out of range (flag 1)
 * is left unchanged.  Returns the flags. */
int32_t oracle_append_tiered(const oracle_append_args* a) {
  int32_t flags = 0;
  const int64_t W = a->hot_window;
  for (int64_t b = 0; b < a->B; ++b) {
    int64_t cl = a->cold_lens[b], hl = a->hot_lens[b], hs = a->hot_starts[b];
    if (W <= 0 || hl < 0 || hl > W || cl < 0 || hs < 0) {
      flags |= ORACLE_FLAG_BAD_TIER;
      continue;
    }
    if (hl == W) {
      if (cl != hs) {
        flags |= ORACLE_FLAG_BAD_TIER;
        continue;
      }
      if (cl >= a->max_blocks * a->block_size) {
        flags |= ORACLE_FLAG_BAD_SEQ_LEN;
        continue;
      }
      const int64_t blk = a->block_table[b * a->max_blocks + cl / a->block_size];
      if (blk < 0 || blk >= a->num_blocks) {
        flags |= ORACLE_FLAG_BAD_BLOCK;
        continue;
      }
      const int64_t cold_row = blk * a->block_size + cl % a->block_size;
      const int64_t hot_row = b * a->hot_capacity + hs % W;
      demote_row(a, a->k_hot, a->k_cold, a->k_scale, a->k_cold_f16, hot_row, cold_row);
      demote_row(a, a->v_hot, a->v_cold, a->v_scale, a->v_cold_f16, hot_row, cold_row);
      cl += 1;
      hs += 1;
      hl -= 1;
    }
    const int64_t slot = (hs + hl) % W;
    const size_t row_bytes = sizeof(uint16_t) * (size_t)(a->Hkv * a->D);
    memcpy(a->k_hot + (b * a->hot_capacity + slot) * a->Hkv * a->D, a->k_new + b * a->Hkv * a->D,
           row_bytes);
    memcpy(a->v_hot + (b * a->hot_capacity + slot) * a->Hkv * a->D, a->v_new + b * a->Hkv * a->D,
           row_bytes);
    hl += 1;
    a->cold_lens[b] = (int32_t)cl;
    a->hot_lens[b] = (int32_t)hl;
    a->hot_starts[b] = (int32_t)hs;
  }
  return flags;
}

/* Append to a paged f16 cache (the paged address of [B]): the new
 * token of sequence b at position positions[b] goes to page
 * block_table[b][pos/bs], row pos % bs.  A position past the table (flag 2) or
 * a page id out of range (flag 1) writes nothing. */
int32_t oracle_append_paged(int64_t B, int64_t Hkv, int64_t D, int64_t block_size,
                            int64_t max_blocks, int64_t num_blocks, const uint16_t* k_new,
                            const uint16_t* v_new, const int32_t* positions,
                            const int32_t* block_table, uint16_t* k_pool, uint16_t* v_pool) {
  int32_t flags = 0;
  const size_t row_bytes = sizeof(uint16_t) * (size_t)(Hkv * D);
  for (int64_t b = 0; b < B; ++b) {
    const int64_t pos = positions[b];
    if (pos < 0 || pos >= max_blocks * block_size) {
      flags |= ORACLE_FLAG_BAD_SEQ_LEN;
      continue;
    }
    const int64_t blk = block_table[b * max_blocks + pos / block_size];
    if (blk < 0 || blk >= num_blocks) {
      flags |= ORACLE_FLAG_BAD_BLOCK;
      continue;
    }
    const int64_t row = blk * block_size + pos % block_size;
    memcpy(k_pool + row * Hkv * D, k_new + b * Hkv * D, row_bytes);
    memcpy(v_pool + row * Hkv * D, v_new + b * Hkv * D, row_bytes);
  }
  return flags;
}

/* Threads the OpenMP runtime will use (reported beside timings). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
