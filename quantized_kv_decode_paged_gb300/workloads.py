"""Seeded synthetic inputs for decode attention over a paged / tiered KV cache.

This module only *draws* inputs: sequence lengths, page assignments, K/V/Q
values and the int8 packing of the cold tier.  It holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle can consume its output.

Every random stream is a counter-based Philox generator keyed by
``(seed, sequence, stream-id)``.  A sequence's pages can therefore be
regenerated on their own (the oracle only needs the sampled sequences) and
the values do not depend on the device that later holds them.

Workloads (the shapes of the pages' serving cases):

* ``tiny``      B=1, Hq=8, Hkv=2, D=64, L=256, bs=16, a shuffled 16-page pool
* ``paged``     B=32, Hq=32, Hkv=8, D=128, L ~ U{512..4096}, bs=16, 65536-page pool
* ``tiered``    B=16, Hq=32, Hkv=8, D=128, L=8192: 7168 int8 cold keys (paged, bs=16)
                + a 1024-slot f16 hot ring
* ``window``    B=64, Hq=16, Hkv=8, D=256, L=8192, window 4096, softcap 50, bs=32,
                1% of keys scaled by 8
* ``longctx``   B=128, Hq=64, Hkv=8, D=128, L ~ lognormal(median 8192, sigma 0.8)
                clamped to [128, 32768], bs=16, pool exactly filled and shuffled
* ``tiered_f16`` the ``tiered`` shape with the 7168 cold keys kept as f16 rows
* ``paged_spec2``, ``paged_spec4`` the ``paged`` shape with 2 or 4 query tokens per
                sequence (speculative decode)
* ``paged_sparse`` the ``paged`` shape with four block-sparse layouts (64-key blocks,
                the last four blocks plus every eighth block, a different eighth per
                layout), query head h reading layout h % 4
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
from typing import Optional

import numpy as np

# stream ids inside a (seed, sequence) key
_S_K, _S_V, _S_OUTLIER, _S_Q, _S_META = 0, 1, 2, 3, 4
_GLOBAL = 1 << 30  # "sequence" index used for batch-wide draws

WORKLOADS = ("tiny", "paged", "tiered", "window", "longctx", "tiered_f16", "paged_spec2",
             "paged_spec4", "paged_sparse")
# Smaller or tighter copies of serving workloads for profiler captures that
# replay a launch: the same kernel instantiation on a few GB at most.
# paged_compact: the keys and values of "paged" in a pool of exactly the used
# pages (about 310 MB instead of 4 GiB); window_compact: 16 of the 64
# sequences of "window".
VARIANTS = ("paged_compact", "paged_sparse_compact", "longctx_compact", "window_compact")


def _rng(seed: int, seq: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[int(seed), int(seq) * 8 + int(stream)]))


def _normal_f16(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def _pool_threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


@dataclass
class PagedCase:
    """f16 paged decode inputs.  K/V rows are stored per sequence (the pages
    that sequence owns, in logical order); full pools are materialised on
    demand on the host or the device."""

    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    q: np.ndarray            # f32 [B, Hq, D]
    block_table: np.ndarray  # i32 [B, max_blocks]; unused entries are -1
    seq_lens: np.ndarray     # i32 [B]
    scale: float = 0.0
    softcap: float = 0.0
    sliding_window: int = 0
    causal: bool = True
    q_pos: Optional[np.ndarray] = None
    outlier_rate: float = 0.0   # fraction of (b, t) keys whose K is scaled by 8
    pages_per_seq: Optional[np.ndarray] = None  # pages holding data per sequence
    nonfinite_tail: bool = False  # fill rows past seq_len in the last page with NaN/Inf
    # block-sparse layouts (CSR): keys per block, row_ptr [NL, rows + 1], col_idx [NL, nnz]
    sparse_block: int = 0
    row_ptr: Optional[np.ndarray] = None
    col_idx: Optional[np.ndarray] = None

    @property
    def sparse(self) -> bool:
        return self.sparse_block > 0

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0

    def seq_pages(self, b: int) -> np.ndarray:
        n = int(self.pages_per_seq[b])
        return self.block_table[b, :n].astype(np.int64)

    def seq_kv(self, b: int):
        """(K, V) f16 rows [n_pages, bs, Hkv, D] of sequence b's pages."""
        n = int(self.pages_per_seq[b])
        shape = (n, self.block_size, self.Hkv, self.D)
        k = _normal_f16(_rng(self.seed, b, _S_K), shape)
        v = _normal_f16(_rng(self.seed, b, _S_V), shape)
        if self.outlier_rate > 0.0 and n:
            hit = _rng(self.seed, b, _S_OUTLIER).random(n * self.block_size) < self.outlier_rate
            k.reshape(n * self.block_size, self.Hkv, self.D)[hit] *= np.float16(8.0)
        if self.nonfinite_tail and n:
            L = int(self.seq_lens[b])
            flat_k = k.reshape(n * self.block_size, self.Hkv, self.D)
            flat_v = v.reshape(n * self.block_size, self.Hkv, self.D)
            flat_k[L:] = np.float16(np.nan)
            flat_v[L:] = np.float16(np.inf)
        return k, v

    def _seqs_with_pages(self, seqs):
        if seqs is None:
            seqs = range(self.B)
        return [int(b) for b in seqs if int(self.pages_per_seq[int(b)]) > 0]

    def host_pools(self, seqs=None):
        """Full host pools (zeros except the pages of ``seqs``; default all)."""
        shape = (self.num_blocks, self.block_size, self.Hkv, self.D)
        k_pool = np.zeros(shape, dtype=np.float16)
        v_pool = np.zeros(shape, dtype=np.float16)
        todo = self._seqs_with_pages(seqs)
        with ThreadPoolExecutor(_pool_threads()) as ex:
            for b, (k, v) in zip(todo, ex.map(self.seq_kv, todo)):
                pages = self.seq_pages(b)
                valid = (pages >= 0) & (pages < self.num_blocks)
                k_pool[pages[valid]] = k[valid]
                v_pool[pages[valid]] = v[valid]
        return k_pool, v_pool

    def device_tensors(self, device="cuda"):
        """Torch tensors on ``device``: q, k_pool, v_pool, block_table, seq_lens,
        q_pos (or None).  Pools are filled sequence by sequence."""
        import torch

        shape = (self.num_blocks, self.block_size, self.Hkv, self.D)
        k_pool = torch.zeros(shape, dtype=torch.float16, device=device)
        v_pool = torch.zeros(shape, dtype=torch.float16, device=device)
        todo = self._seqs_with_pages(None)
        with ThreadPoolExecutor(_pool_threads()) as ex:
            for b, (k, v) in zip(todo, ex.map(self.seq_kv, todo)):
                pages = self.seq_pages(b)
                valid = (pages >= 0) & (pages < self.num_blocks)
                idx = torch.from_numpy(pages[valid]).to(device)
                k_pool.index_copy_(0, idx, torch.from_numpy(k[valid]).to(device))
                v_pool.index_copy_(0, idx, torch.from_numpy(v[valid]).to(device))
        t = dict(
            q=torch.from_numpy(self.q).to(device),
            k_pool=k_pool,
            v_pool=v_pool,
            block_table=torch.from_numpy(self.block_table).to(device),
            seq_lens=torch.from_numpy(self.seq_lens).to(device),
            q_pos=None if self.q_pos is None else torch.from_numpy(self.q_pos).to(device),
        )
        if self.sparse:
            t["row_ptr"] = torch.from_numpy(self.row_ptr).to(device)
            t["col_idx"] = torch.from_numpy(self.col_idx).to(device)
        return t


def _assign_pages(rng, B, pages_needed, num_blocks, max_blocks):
    """Non-overlapping random page assignment: sequence b takes the next
    pages_needed[b] ids of one permutation of the pool."""
    if int(np.sum(pages_needed)) > num_blocks:
        raise ValueError("pool too small for the requested lengths")
    if B and int(np.max(pages_needed)) > max_blocks:
        raise ValueError("block table too narrow for the requested lengths")
    perm = rng.permutation(num_blocks).astype(np.int32)
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        n = int(pages_needed[b])
        table[b, :n] = perm[pos:pos + n]
        pos += n
    return table


def make_paged(name, seed, B, Hq, Hkv, D, block_size, seq_lens, num_blocks=None,
               max_blocks=None, scale=0.0, softcap=0.0, sliding_window=0, causal=True,
               q_pos=None, outlier_rate=0.0, nonfinite_tail=False, q_len=1) -> PagedCase:
    """q_len > 1 draws q [B, q_len, Hq, D] (several query tokens per sequence)."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32).reshape(B)
    pages = np.array([(max(int(L), 0) + block_size - 1) // block_size for L in seq_lens],
                     dtype=np.int64)
    if max_blocks is None:
        max_blocks = max(1, int(pages.max()) if B else 1)
    if num_blocks is None:
        num_blocks = max(1, int(pages.sum()))
    meta = _rng(seed, _GLOBAL, _S_META)
    table = _assign_pages(meta, B, pages, num_blocks, max_blocks)
    qshape = (B, Hq, D) if q_len == 1 else (B, q_len, Hq, D)
    q = _rng(seed, _GLOBAL, _S_Q).standard_normal(qshape, dtype=np.float32)
    return PagedCase(name=name, seed=seed, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size,
                     num_blocks=int(num_blocks), q=q, block_table=table, seq_lens=seq_lens,
                     scale=scale, softcap=softcap, sliding_window=sliding_window,
                     causal=causal, q_pos=None if q_pos is None else
                     np.asarray(q_pos, dtype=np.int32).reshape(B),
                     outlier_rate=outlier_rate, pages_per_seq=pages,
                     nonfinite_tail=nonfinite_tail)


def csr_layouts(rows_of_layouts, num_rows, max_nnz=None):
    """CSR arrays (row_ptr [NL, num_rows + 1], col_idx [NL, max_nnz]) from, per
    layout, a list of column lists (one per row; missing rows are empty).
    Unused column entries hold -1."""
    NL = len(rows_of_layouts)
    need = max([sum(len(r) for r in lay) for lay in rows_of_layouts] + [1])
    nnz = need if max_nnz is None else max(int(max_nnz), need)
    row_ptr = np.zeros((NL, num_rows + 1), np.int32)
    col_idx = np.full((NL, nnz), -1, np.int32)
    for l, lay in enumerate(rows_of_layouts):
        pos = 0
        for r in range(num_rows):
            cols = list(lay[r]) if r < len(lay) else []
            row_ptr[l, r] = pos
            col_idx[l, pos:pos + len(cols)] = cols
            pos += len(cols)
        row_ptr[l, num_rows] = pos
    return row_ptr, col_idx


def local_stride_layouts(num_layouts, num_rows, local_blocks, vert_stride):
    """Block-sparse layouts of the local + vertical-stride kind: row r of
    layout l lists the last `local_blocks` blocks up to r and every block
    c <= r with (c + l) % vert_stride == 0 (each layout a different stride
    phase).  Returns the per-layout lists of sorted column lists."""
    lays = []
    for l in range(num_layouts):
        rows = []
        for r in range(num_rows):
            cols = set(range(max(0, r - local_blocks + 1), r + 1))
            cols.update(c for c in range(r + 1) if (c + l) % vert_stride == 0)
            rows.append(sorted(cols))
        lays.append(rows)
    return lays


def make_sparse(name, seed, B, Hq, Hkv, D, block_size, seq_lens, sparse_block, layouts,
                num_rows=None, max_nnz=None, **kw) -> PagedCase:
    """make_paged plus block-sparse CSR layouts (lists of column lists per
    row, one list per layout)."""
    case = make_paged(name, seed, B, Hq, Hkv, D, block_size, seq_lens, **kw)
    if num_rows is None:
        num_rows = max(1, -(-max(int(np.max(case.seq_lens)), 1) // sparse_block))
    case.sparse_block = int(sparse_block)
    case.row_ptr, case.col_idx = csr_layouts(layouts, num_rows, max_nnz)
    return case


def workload(name: str):
    """The named serving workload (see the module docstring)."""
    if name == "tiny":
        return make_paged("tiny", 0, B=1, Hq=8, Hkv=2, D=64, block_size=16, seq_lens=[256],
                          num_blocks=16, max_blocks=16)
    if name == "paged":
        meta = _rng(1, _GLOBAL, _S_META + 1)
        lens = meta.integers(512, 4096, size=32, endpoint=True)
        return make_paged("paged", 1, B=32, Hq=32, Hkv=8, D=128, block_size=16, seq_lens=lens,
                          num_blocks=65536, max_blocks=256)
    if name == "paged_compact":
        meta = _rng(1, _GLOBAL, _S_META + 1)
        lens = meta.integers(512, 4096, size=32, endpoint=True)
        return make_paged("paged_compact", 1, B=32, Hq=32, Hkv=8, D=128, block_size=16,
                          seq_lens=lens, max_blocks=256)
    if name == "tiered":
        return make_tiered("tiered", 2, B=16, Hq=32, Hkv=8, D=128, block_size=16,
                           cold_len=7168, hot_len=1024, hot_window=1024, hot_start=7168)
    if name in ("paged_spec2", "paged_spec4"):
        # the paged workload with 2 or 4 query tokens per sequence (speculative decode)
        meta = _rng(1, _GLOBAL, _S_META + 1)
        lens = meta.integers(512, 4096, size=32, endpoint=True)
        return make_paged(name, 1, B=32, Hq=32, Hkv=8, D=128, block_size=16, seq_lens=lens,
                          num_blocks=65536, max_blocks=256, q_len=int(name[-1]))
    if name == "tiered_f16":
        return make_tiered("tiered_f16", 2, B=16, Hq=32, Hkv=8, D=128, block_size=16,
                           cold_len=7168, hot_len=1024, hot_window=1024, hot_start=7168,
                           cold_f16=True)
    if name in ("window", "window_compact"):
        B = 64 if name == "window" else 16
        return make_paged(name, 3, B=B, Hq=16, Hkv=8, D=256, block_size=32,
                          seq_lens=[8192] * B, num_blocks=B * 256, max_blocks=256,
                          sliding_window=4096, softcap=50.0, outlier_rate=0.01)
    if name in ("paged_sparse", "paged_sparse_compact"):
        # the compact variant keeps only the used pages (for profiler captures)
        meta = _rng(1, _GLOBAL, _S_META + 1)
        lens = meta.integers(512, 4096, size=32, endpoint=True)
        rows = 4096 // 64
        return make_sparse(name, 1, B=32, Hq=32, Hkv=8, D=128, block_size=16,
                           seq_lens=lens, sparse_block=64,
                           layouts=local_stride_layouts(4, rows, 4, 8), num_rows=rows,
                           num_blocks=65536 if name == "paged_sparse" else None, max_blocks=256)
    if name in ("longctx", "longctx_compact"):
        meta = _rng(4, _GLOBAL, _S_META + 1)
        z = meta.standard_normal(128)
        lens = np.clip(np.rint(np.exp(math.log(8192.0) + 0.8 * z)), 128, 32768).astype(np.int32)
        if name == "longctx_compact":
            # the first 32 sequences (about 1.3 GB of pages): the same kernel
            # instantiation for profiler captures that replay the launch
            return make_paged(name, 4, B=32, Hq=64, Hkv=8, D=128, block_size=16,
                              seq_lens=lens[:32], max_blocks=2048)
        return make_paged("longctx", 4, B=128, Hq=64, Hkv=8, D=128, block_size=16,
                          seq_lens=lens, max_blocks=2048)
    raise KeyError(name)


# ---------------------------------------------------------------------------
# Tiered cache: int8 cold pages + f16 hot ring
# ---------------------------------------------------------------------------

def quantize_int8_rows(x: np.ndarray):
    """Symmetric int8 quantisation of f16 rows ``x[..., D]``: one f16 scale
    per row, scale = f16(max|x| / 127), q = clamp(rint(x / scale), -127, 127)
    (rint ties to even, division in f32), q = 0 where the scale is 0.
    Returns (int8 values [..., D], f16 scales [...])."""
    xf = x.astype(np.float32)
    amax = np.abs(xf).max(axis=-1)
    s16 = (amax / np.float32(127.0)).astype(np.float16)
    s32 = s16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        qf = np.rint(xf / s32[..., None])
    qf = np.where(s32[..., None] > 0, qf, 0.0)
    q = np.clip(qf, -127, 127).astype(np.int8)
    return q, s16


def pack_int8_words(q: np.ndarray) -> np.ndarray:
    """Four int8 values per little-endian u32: value d sits in byte d % 4 of
    word d // 4."""
    D = q.shape[-1]
    assert D % 4 == 0
    b = q.astype(np.int8).view(np.uint8).reshape(q.shape[:-1] + (D // 4, 4)).astype(np.uint32)
    return b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24)


@dataclass
class TieredCase:
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    hot_window: int
    hot_capacity: int
    q: np.ndarray            # f32 [B, Hq, D]
    block_table: np.ndarray  # i32 [B, max_blocks] (cold pages)
    cold_lens: np.ndarray    # i32 [B]
    hot_lens: np.ndarray     # i32 [B]
    hot_starts: np.ndarray   # i32 [B]
    scale: float = 0.0
    softcap: float = 0.0
    sliding_window: int = 0
    causal: bool = True
    q_pos: Optional[np.ndarray] = None
    pages_per_seq: Optional[np.ndarray] = None
    uniform: bool = True     # every sequence has the same tier lengths
    cold_f16: bool = False   # cold tier as f16 rows instead of int8 words + scales

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int((self.cold_lens + self.hot_lens).max())

    def seq_source(self, b: int):
        """Source f16 K/V of sequence b: cold rows [n_pages*bs, Hkv, D] and hot
        rows [hot_len, Hkv, D] in logical order."""
        n = int(self.pages_per_seq[b])
        hl = int(self.hot_lens[b])
        k = _normal_f16(_rng(self.seed, b, _S_K), (n * self.block_size + hl, self.Hkv, self.D))
        v = _normal_f16(_rng(self.seed, b, _S_V), (n * self.block_size + hl, self.Hkv, self.D))
        c = n * self.block_size
        return k[:c], v[:c], k[c:], v[c:]

    def seq_encoded(self, b: int):
        kc, vc, kh, vh = self.seq_source(b)
        n = int(self.pages_per_seq[b])
        if self.cold_f16:
            shp = (n, self.block_size, self.Hkv, self.D)
            return kc.reshape(shp), vc.reshape(shp), None, None, kh, vh
        kq, ks = quantize_int8_rows(kc)
        vq, vs = quantize_int8_rows(vc)
        shp = (n, self.block_size, self.Hkv)
        return (pack_int8_words(kq).reshape(shp + (self.D // 4,)),
                pack_int8_words(vq).reshape(shp + (self.D // 4,)),
                ks.reshape(shp), vs.reshape(shp), kh, vh)

    def _hot_slots(self, b: int) -> np.ndarray:
        hl, hs = int(self.hot_lens[b]), int(self.hot_starts[b])
        j = np.arange(hl, dtype=np.int64)
        return (hs + j) % self.hot_window if self.hot_window > 0 else j

    def host_arrays(self, seqs=None):
        """Host buffers: k_hot, v_hot, k_cold, v_cold and (int8 cold tier)
        k_scale, v_scale; zeros except the data of ``seqs`` (default all)."""
        cap, H, D = self.hot_capacity, self.Hkv, self.D
        k_hot = np.zeros((self.B, cap, H, D), dtype=np.float16)
        v_hot = np.zeros_like(k_hot)
        if self.cold_f16:
            k_cold = np.zeros((self.num_blocks, self.block_size, H, D), dtype=np.float16)
        else:
            k_cold = np.zeros((self.num_blocks, self.block_size, H, D // 4), dtype=np.uint32)
        v_cold = np.zeros_like(k_cold)
        k_scale = np.zeros((self.num_blocks, self.block_size, H), dtype=np.float16)
        v_scale = np.zeros_like(k_scale)
        todo = list(range(self.B)) if seqs is None else [int(b) for b in seqs]
        with ThreadPoolExecutor(_pool_threads()) as ex:
            for b, enc in zip(todo, ex.map(self.seq_encoded, todo)):
                kw, vw, ks, vs, kh, vh = enc
                pages = self.block_table[b, :int(self.pages_per_seq[b])].astype(np.int64)
                ok = (pages >= 0) & (pages < self.num_blocks)  # a corrupted entry holds no data
                k_cold[pages[ok]], v_cold[pages[ok]] = kw[ok], vw[ok]
                if not self.cold_f16:
                    k_scale[pages[ok]], v_scale[pages[ok]] = ks[ok], vs[ok]
                slots = self._hot_slots(b)
                k_hot[b, slots] = kh
                v_hot[b, slots] = vh
        out = dict(k_hot=k_hot, v_hot=v_hot, k_cold=k_cold, v_cold=v_cold)
        if not self.cold_f16:
            out.update(k_scale=k_scale, v_scale=v_scale)
        return out

    def device_tensors(self, device="cuda"):
        import torch

        h = self.host_arrays()
        if not self.cold_f16:
            for k in ("k_cold", "v_cold"):
                h[k] = h[k].view(np.int32)  # the same 32-bit words, as a torch-friendly dtype
        t = {k: torch.from_numpy(v).to(device) for k, v in h.items()}
        t["q"] = torch.from_numpy(self.q).to(device)
        t["block_table"] = torch.from_numpy(self.block_table).to(device)
        for k in ("cold_lens", "hot_lens", "hot_starts"):
            t[k] = torch.from_numpy(getattr(self, k)).to(device)
        t["q_pos"] = None if self.q_pos is None else torch.from_numpy(self.q_pos).to(device)
        return t


def make_tiered(name, seed, B, Hq, Hkv, D, block_size, cold_len, hot_len, hot_window,
                hot_start, hot_capacity=None, scale=0.0, softcap=0.0, sliding_window=0,
                causal=True, q_pos=None, num_blocks=None, max_blocks=None,
                cold_f16=False) -> TieredCase:
    cold_lens = np.broadcast_to(np.asarray(cold_len, dtype=np.int32), (B,)).copy()
    hot_lens = np.broadcast_to(np.asarray(hot_len, dtype=np.int32), (B,)).copy()
    hot_starts = np.broadcast_to(np.asarray(hot_start, dtype=np.int32), (B,)).copy()
    uniform = bool((cold_lens == cold_lens[0]).all() and (hot_lens == hot_lens[0]).all()
                   and (hot_starts == hot_starts[0]).all())
    if hot_capacity is None:
        hot_capacity = max(hot_window, int(hot_lens.max()), 1)
    pages = np.array([(int(c) + block_size - 1) // block_size for c in cold_lens], dtype=np.int64)
    if max_blocks is None:
        max_blocks = max(1, int(pages.max()))
    if num_blocks is None:
        num_blocks = max(1, int(pages.sum()))
    meta = _rng(seed, _GLOBAL, _S_META)
    table = _assign_pages(meta, B, pages, num_blocks, max_blocks)
    q = _rng(seed, _GLOBAL, _S_Q).standard_normal((B, Hq, D), dtype=np.float32)
    return TieredCase(name=name, seed=seed, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size,
                      num_blocks=int(num_blocks), hot_window=int(hot_window),
                      hot_capacity=int(hot_capacity), q=q, block_table=table,
                      cold_lens=cold_lens, hot_lens=hot_lens, hot_starts=hot_starts,
                      scale=scale, softcap=softcap, sliding_window=sliding_window,
                      causal=causal, q_pos=None if q_pos is None else
                      np.asarray(q_pos, dtype=np.int32).reshape(B),
                      pages_per_seq=pages, uniform=uniform, cold_f16=bool(cold_f16))
