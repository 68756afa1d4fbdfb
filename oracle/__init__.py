"""CPU oracle for paged / tiered decode attention (double precision).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers; the product package
never imports this module.  It wraps ``decode_attn_oracle.c`` (plain C,
double precision, two passes over the logical key order) through ctypes and
shares no code with the CUDA library.

Every function takes numpy arrays on the host:

* ``q``            float32 [B, Hq, D]
* ``k_pool/v_pool`` float16 [NB, bs, Hkv, D]
* ``block_table``  int32   [B, max_blocks]
* ``seq_lens``     int32   [B]
* ``q_pos``        int32   [B] or None

and returns float64 outputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "decode_attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

FLAG_BAD_BLOCK = 1
FLAG_BAD_SEQ_LEN = 2
FLAG_BAD_QPOS = 4
FLAG_SPLIT_OVERFLOW = 8
FLAG_BAD_TIER = 16


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP).  Returns the library path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _PagedArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("Hq", ctypes.c_int64), ("Hkv", ctypes.c_int64),
        ("D", ctypes.c_int64), ("block_size", ctypes.c_int64),
        ("max_blocks", ctypes.c_int64), ("num_blocks", ctypes.c_int64),
        ("scale", ctypes.c_double), ("softcap", ctypes.c_double),
        ("window", ctypes.c_int64), ("causal", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("q_pos", ctypes.c_void_p), ("q_len", ctypes.c_int64),
    ]


class _TieredArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("Hq", ctypes.c_int64), ("Hkv", ctypes.c_int64),
        ("D", ctypes.c_int64), ("block_size", ctypes.c_int64),
        ("max_blocks", ctypes.c_int64), ("num_blocks", ctypes.c_int64),
        ("scale", ctypes.c_double), ("softcap", ctypes.c_double),
        ("window", ctypes.c_int64), ("causal", ctypes.c_int64),
        ("hot_window", ctypes.c_int64), ("hot_capacity", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k_hot", ctypes.c_void_p), ("v_hot", ctypes.c_void_p),
        ("k_cold", ctypes.c_void_p), ("v_cold", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("cold_lens", ctypes.c_void_p),
        ("hot_lens", ctypes.c_void_p), ("hot_starts", ctypes.c_void_p),
        ("q_pos", ctypes.c_void_p),
        ("k_cold_f16", ctypes.c_void_p), ("v_cold_f16", ctypes.c_void_p),
    ]


class _AppendArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "Hkv", "D", "block_size", "max_blocks",
                                              "num_blocks", "hot_window", "hot_capacity")] + [
        (n, ctypes.c_void_p) for n in ("k_new", "v_new", "k_hot", "v_hot", "k_cold", "v_cold",
                                       "k_scale", "v_scale", "k_cold_f16", "v_cold_f16",
                                       "block_table", "cold_lens", "hot_lens", "hot_starts")]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_unpack_int8_word.restype = None
            lib.oracle_unpack_int8_word.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
            lib.oracle_decode_paged.restype = ctypes.c_int32
            lib.oracle_decode_paged.argtypes = [ctypes.POINTER(_PagedArgs), ctypes.c_void_p,
                                                ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_decode_paged_sparse.restype = ctypes.c_int32
            lib.oracle_decode_paged_sparse.argtypes = [
                ctypes.POINTER(_PagedArgs), ctypes.POINTER(_SparseLayout), ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_decode_paged_split.restype = ctypes.c_int32
            lib.oracle_decode_paged_split.argtypes = [
                ctypes.POINTER(_PagedArgs), ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_split_merge.restype = None
            lib.oracle_split_merge.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_decode_tiered.restype = ctypes.c_int32
            lib.oracle_decode_tiered.argtypes = [ctypes.POINTER(_TieredArgs), ctypes.c_void_p,
                                                 ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_float_to_half_array.restype = None
            lib.oracle_float_to_half_array.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                                       ctypes.c_void_p]
            lib.oracle_quantize_row_int8.restype = None
            lib.oracle_quantize_row_int8.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                                     ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_append_tiered.restype = ctypes.c_int32
            lib.oracle_append_tiered.argtypes = [ctypes.POINTER(_AppendArgs)]
            lib.oracle_append_paged.restype = ctypes.c_int32
            lib.oracle_append_paged.argtypes = [ctypes.c_int64] * 6 + [ctypes.c_void_p] * 6
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def half_to_double(bits: int) -> float:
    """Decode one IEEE binary16 bit pattern with the oracle's own decoder."""
    return float(_load().oracle_half_to_double(int(bits) & 0xFFFF))


def unpack_int8_word(word: int) -> list[int]:
    """The four signed bytes of a packed cold word, lane 0 first."""
    out = np.zeros(4, dtype=np.int32)
    _load().oracle_unpack_int8_word(int(word) & 0xFFFFFFFF, out.ctypes.data)
    return [int(x) for x in out]


def _rows_arg(rows):
    if rows is None:
        return None
    return np.ascontiguousarray(rows, dtype=np.int64)


class _Keep:
    """Holds the contiguous copies alive for the duration of a call."""

    def __init__(self):
        self.items = []

    def __call__(self, a, dtype):
        c = _c(a, dtype)
        self.items.append(c)
        return c


def _paged_struct(keep, q, k_pool, v_pool, block_table, seq_lens, q_pos, scale, softcap,
                  sliding_window, causal):
    q = keep(q, np.float32)
    k_pool = keep(k_pool, np.float16)
    v_pool = keep(v_pool, np.float16)
    block_table = keep(block_table, np.int32)
    seq_lens = keep(seq_lens, np.int32)
    q_pos = keep(q_pos, np.int32)
    # q is [B, Hq, D], or [B, T, Hq, D] for T query tokens per sequence
    T = q.shape[1] if q.ndim == 4 else 1
    B, Hq, D = q.shape[0], q.shape[-2], q.shape[-1]
    NB, bs, Hkv, D2 = k_pool.shape
    assert D2 == D and v_pool.shape == k_pool.shape
    assert block_table.shape[0] == B and seq_lens.shape == (B,)
    args = _PagedArgs(B, Hq, Hkv, D, bs, block_table.shape[1], NB,
                      float(np.float32(scale)), float(np.float32(softcap)),
                      int(sliding_window), int(bool(causal)),
                      _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                      _ptr(seq_lens), _ptr(q_pos), T)
    return args, B, Hq, D, T


def decode_paged(q, k_pool, v_pool, block_table, seq_lens, q_pos=None, *, scale=0.0,
                 softcap=0.0, sliding_window=0, causal=True, rows=None):
    """Paged f16 decode attention.  Returns (out [n, D], lse [n], flags).

    ``q`` is [B, Hq, D] (one query token per sequence) or [B, T, Hq, D] (T
    tokens at positions q_pos[b] + t, by default seq_len - T + t).  ``rows``
    selects flat rows (b*T + t)*Hq + h (default: every row, in order)."""
    keep = _Keep()
    args, B, Hq, D, T = _paged_struct(keep, q, k_pool, v_pool, block_table, seq_lens, q_pos,
                                      scale, softcap, sliding_window, causal)
    rows_a = _rows_arg(rows)
    n = B * T * Hq if rows_a is None else len(rows_a)
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    flags = _load().oracle_decode_paged(ctypes.byref(args), _ptr(rows_a), n, _ptr(out), _ptr(lse))
    return out, lse, int(flags)


class _SparseLayout(ctypes.Structure):
    _fields_ = [("sparse_block", ctypes.c_int64), ("num_layouts", ctypes.c_int64),
                ("num_rows", ctypes.c_int64), ("max_nnz", ctypes.c_int64),
                ("row_ptr", ctypes.c_void_p), ("col_idx", ctypes.c_void_p)]


def decode_paged_sparse(q, k_pool, v_pool, block_table, seq_lens, row_ptr, col_idx,
                        sparse_block, q_pos=None, *, scale=0.0, softcap=0.0, sliding_window=0,
                        causal=True, rows=None):
    """Block-sparse paged decode (one query token): head h keeps the keys of
    the sparse blocks that CSR row q_pos / sparse_block of layout
    h % num_layouts lists.  row_ptr int32 [num_layouts, num_rows + 1],
    col_idx int32 [num_layouts, max_nnz].  Returns (out [n, D], lse [n], flags)."""
    keep = _Keep()
    args, B, Hq, D, T = _paged_struct(keep, q, k_pool, v_pool, block_table, seq_lens, q_pos,
                                      scale, softcap, sliding_window, causal)
    assert T == 1
    row_ptr = keep(row_ptr, np.int32)
    col_idx = keep(col_idx, np.int32)
    assert row_ptr.ndim == 2 and col_idx.ndim == 2 and row_ptr.shape[0] == col_idx.shape[0]
    sl = _SparseLayout(int(sparse_block), row_ptr.shape[0], row_ptr.shape[1] - 1,
                       col_idx.shape[1], _ptr(row_ptr), _ptr(col_idx))
    rows_a = _rows_arg(rows)
    n = B * Hq if rows_a is None else len(rows_a)
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    flags = _load().oracle_decode_paged_sparse(ctypes.byref(args), ctypes.byref(sl),
                                               _ptr(rows_a), n, _ptr(out), _ptr(lse))
    return out, lse, int(flags)


def decode_paged_split(q, k_pool, v_pool, block_table, seq_lens, q_pos=None, *, split_tokens,
                       max_splits, scale=0.0, softcap=0.0, sliding_window=0, causal=True,
                       rows=None):
    """Split partials (one query token).  Returns (o_part [n, S, D], lse_part [n, S], flags)."""
    keep = _Keep()
    args, B, Hq, D, T = _paged_struct(keep, q, k_pool, v_pool, block_table, seq_lens, q_pos,
                                      scale, softcap, sliding_window, causal)
    assert T == 1
    rows_a = _rows_arg(rows)
    n = B * Hq if rows_a is None else len(rows_a)
    o_part = np.zeros((n, max_splits, D), dtype=np.float64)
    lse_part = np.zeros((n, max_splits), dtype=np.float64)
    flags = _load().oracle_decode_paged_split(ctypes.byref(args), int(split_tokens),
                                              int(max_splits), _ptr(rows_a), n,
                                              _ptr(o_part), _ptr(lse_part))
    return o_part, lse_part, int(flags)


def split_merge(o_part, lse_part):
    """Merge of split partials.  o_part [n, S, D], lse_part [n, S]."""
    o_part = np.ascontiguousarray(o_part, dtype=np.float64)
    lse_part = np.ascontiguousarray(lse_part, dtype=np.float64)
    n, S, D = o_part.shape
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    _load().oracle_split_merge(n, S, D, _ptr(o_part), _ptr(lse_part), _ptr(out), _ptr(lse))
    return out, lse


def decode_tiered(q, k_hot, v_hot, k_cold, v_cold, k_scale, v_scale, block_table, cold_lens,
                  hot_lens, hot_starts, *, hot_window, q_pos=None, scale=0.0, softcap=0.0,
                  sliding_window=0, causal=True, rows=None):
    """Tiered int8-cold / f16-hot decode attention.

    k_hot/v_hot float16 [B, cap, Hkv, D]; k_cold/v_cold uint32 [NB, bs, Hkv, D/4];
    k_scale/v_scale float16 [NB, bs, Hkv]; cold_lens/hot_lens/hot_starts int32 [B].
    Returns (out [n, D], lse [n], flags)."""
    keep = _Keep()
    q = keep(q, np.float32)
    k_hot = keep(k_hot, np.float16)
    v_hot = keep(v_hot, np.float16)
    k_cold = keep(k_cold, np.uint32)
    v_cold = keep(v_cold, np.uint32)
    k_scale = keep(k_scale, np.float16)
    v_scale = keep(v_scale, np.float16)
    block_table = keep(block_table, np.int32)
    B, Hq, D = q.shape
    cold_lens = keep(np.broadcast_to(np.asarray(cold_lens, dtype=np.int32), (B,)), np.int32)
    hot_lens = keep(np.broadcast_to(np.asarray(hot_lens, dtype=np.int32), (B,)), np.int32)
    hot_starts = keep(np.broadcast_to(np.asarray(hot_starts, dtype=np.int32), (B,)), np.int32)
    q_pos = keep(q_pos, np.int32)
    Bh, cap, Hkv, D2 = k_hot.shape
    NB, bs, Hkv2, W4 = k_cold.shape
    assert Bh == B and D2 == D and Hkv2 == Hkv and W4 * 4 == D
    assert k_scale.shape == (NB, bs, Hkv)
    args = _TieredArgs(B, Hq, Hkv, D, bs, block_table.shape[1], NB,
                       float(np.float32(scale)), float(np.float32(softcap)),
                       int(sliding_window), int(bool(causal)), int(hot_window), cap,
                       _ptr(q), _ptr(k_hot), _ptr(v_hot), _ptr(k_cold), _ptr(v_cold),
                       _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(cold_lens),
                       _ptr(hot_lens), _ptr(hot_starts), _ptr(q_pos), None, None)
    rows_a = _rows_arg(rows)
    n = B * Hq if rows_a is None else len(rows_a)
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    flags = _load().oracle_decode_tiered(ctypes.byref(args), _ptr(rows_a), n, _ptr(out), _ptr(lse))
    return out, lse, int(flags)


def decode_tiered_f16(q, k_hot, v_hot, k_cold, v_cold, block_table, cold_lens, hot_lens,
                      hot_starts, *, hot_window, q_pos=None, scale=0.0, softcap=0.0,
                      sliding_window=0, causal=True, rows=None):
    """Tiered f16-cold / f16-hot decode attention (the f16 tiered layout of
    doppler attention.js executeAttentionTiered).

    k_hot/v_hot float16 [B, cap, Hkv, D]; k_cold/v_cold float16 [NB, bs, Hkv, D];
    cold_lens/hot_lens/hot_starts int32 [B].  Returns (out [n, D], lse [n], flags)."""
    keep = _Keep()
    q = keep(q, np.float32)
    k_hot = keep(k_hot, np.float16)
    v_hot = keep(v_hot, np.float16)
    k_cold = keep(k_cold, np.float16)
    v_cold = keep(v_cold, np.float16)
    block_table = keep(block_table, np.int32)
    B, Hq, D = q.shape
    cold_lens = keep(np.broadcast_to(np.asarray(cold_lens, dtype=np.int32), (B,)), np.int32)
    hot_lens = keep(np.broadcast_to(np.asarray(hot_lens, dtype=np.int32), (B,)), np.int32)
    hot_starts = keep(np.broadcast_to(np.asarray(hot_starts, dtype=np.int32), (B,)), np.int32)
    q_pos = keep(q_pos, np.int32)
    Bh, cap, Hkv, D2 = k_hot.shape
    NB, bs, Hkv2, D3 = k_cold.shape
    assert Bh == B and D2 == D and Hkv2 == Hkv and D3 == D and v_cold.shape == k_cold.shape
    args = _TieredArgs(B, Hq, Hkv, D, bs, block_table.shape[1], NB,
                       float(np.float32(scale)), float(np.float32(softcap)),
                       int(sliding_window), int(bool(causal)), int(hot_window), cap,
                       _ptr(q), _ptr(k_hot), _ptr(v_hot), None, None, None, None,
                       _ptr(block_table), _ptr(cold_lens), _ptr(hot_lens), _ptr(hot_starts),
                       _ptr(q_pos), _ptr(k_cold), _ptr(v_cold))
    rows_a = _rows_arg(rows)
    n = B * Hq if rows_a is None else len(rows_a)
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    flags = _load().oracle_decode_tiered(ctypes.byref(args), _ptr(rows_a), n, _ptr(out), _ptr(lse))
    return out, lse, int(flags)


# ---------------------------------------------------------------------------
# KV append and int8 demotion
# ---------------------------------------------------------------------------

def float_to_half(x) -> np.ndarray:
    """binary16 bit patterns (uint16) of float32 values, round to nearest even,
    with the oracle's own encoder."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.zeros(x.shape, dtype=np.uint16)
    _load().oracle_float_to_half_array(_ptr(x), x.size, _ptr(out))
    return out


def quantize_row_int8(x):
    """Demotion quantizer of one row of f16 values: (int8 codes, f16 scale bits)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float16))
    assert x.ndim == 1 and x.size <= 1024
    code = np.zeros(x.size, dtype=np.int8)
    scale = np.zeros(1, dtype=np.uint16)
    _load().oracle_quantize_row_int8(_ptr(x.view(np.uint16)), x.size, _ptr(code), _ptr(scale))
    return code, int(scale[0])


def append_tiered(k_new, v_new, k_hot, v_hot, k_cold, v_cold, k_scale, v_scale, block_table,
                  cold_lens, hot_lens, hot_starts, *, hot_window):
    """One append step of a tiered cache, on copies.  int8 tier: k_cold/v_cold
    uint32 words [NB, bs, Hkv, D/4] with k_scale/v_scale f16 [NB, bs, Hkv];
    f16 tier: k_cold/v_cold float16 [NB, bs, Hkv, D] and k_scale = v_scale =
    None.  Returns (dict of the updated arrays, flags)."""
    k_new = np.ascontiguousarray(k_new, dtype=np.float16)
    v_new = np.ascontiguousarray(v_new, dtype=np.float16)
    st = {n: np.array(a, copy=True) for n, a in (("k_hot", k_hot), ("v_hot", v_hot),
                                                  ("k_cold", k_cold), ("v_cold", v_cold))}
    f16 = st["k_cold"].dtype == np.float16
    if not f16:
        st["k_scale"] = np.array(k_scale, dtype=np.float16, copy=True)
        st["v_scale"] = np.array(v_scale, dtype=np.float16, copy=True)
    for n, a in (("cold_lens", cold_lens), ("hot_lens", hot_lens), ("hot_starts", hot_starts)):
        st[n] = np.array(a, dtype=np.int32, copy=True)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    B, cap, Hkv, D = st["k_hot"].shape
    NB, bs = st["k_cold"].shape[:2]
    assert D <= 1024 and k_new.shape == (B, Hkv, D)
    args = _AppendArgs(B, Hkv, D, bs, bt.shape[1], NB, int(hot_window), cap,
                       _ptr(k_new), _ptr(v_new), _ptr(st["k_hot"]), _ptr(st["v_hot"]),
                       None if f16 else _ptr(st["k_cold"]), None if f16 else _ptr(st["v_cold"]),
                       None if f16 else _ptr(st["k_scale"]), None if f16 else _ptr(st["v_scale"]),
                       _ptr(st["k_cold"]) if f16 else None, _ptr(st["v_cold"]) if f16 else None,
                       _ptr(bt), _ptr(st["cold_lens"]), _ptr(st["hot_lens"]),
                       _ptr(st["hot_starts"]))
    flags = _load().oracle_append_tiered(ctypes.byref(args))
    return st, int(flags)


def append_paged(k_new, v_new, positions, block_table, k_pool, v_pool):
    """Writes each sequence's new K/V row [B, Hkv, D] at its position, on
    copies of the pools.  Returns (k_pool, v_pool, flags)."""
    k_new = np.ascontiguousarray(k_new, dtype=np.float16)
    v_new = np.ascontiguousarray(v_new, dtype=np.float16)
    kp = np.array(k_pool, dtype=np.float16, copy=True)
    vp = np.array(v_pool, dtype=np.float16, copy=True)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    NB, bs, Hkv, D = kp.shape
    B = k_new.shape[0]
    flags = _load().oracle_append_paged(B, Hkv, D, bs, bt.shape[1], NB, _ptr(k_new), _ptr(v_new),
                                        _ptr(pos), _ptr(bt), _ptr(kp), _ptr(vp))
    return kp, vp, int(flags)
