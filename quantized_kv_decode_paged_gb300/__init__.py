"""GB300 decode attention over a paged / tiered (int8 or f16 cold tier) KV cache.

Thin Python binding of ``libdecode_attn.so`` (C ABI in ``include/decode_attn.h``).
The functions below only marshal torch tensors into the C calls: every step
of the computation runs in the library's CUDA kernels.  Nothing falls back
to another implementation: if the library is missing or the device is not a
CUDA device, the call raises.

Layouts (row-major, innermost last): q f32 [B, Hq, D]; K/V pools f16
[num_blocks, block_size, Hkv, D]; block_table i32 [B, max_blocks];
seq_lens i32 [B]; out f32 [B, Hq, D]; lse f32 [B, Hq].
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import _build

__all__ = [
    "load_library", "library_path", "build",
    "decode_attn_paged", "decode_attn_paged_multi", "decode_attn_paged_sparse",
    "decode_attn_tiered_int8", "decode_attn_tiered_f16", "decode_attn_split_partial",
    "decode_attn_split_merge", "decode_attn_workspace_size", "decode_attn_status_string",
    "decode_attn_paged_static_ws", "decode_attn_append_paged", "decode_attn_append_tiered_int8",
    "decode_attn_append_tiered_f16", "DecodeAttnError", "DaTuning", "get_tuning", "set_tuning",
    "tuning", "DEV_BAD_BLOCK", "DEV_BAD_SEQ_LEN",
    "DEV_BAD_QPOS", "DEV_SPLIT_OVERFLOW", "DEV_BAD_TIER", "DEV_TIMEOUT",
]

DEV_BAD_BLOCK = 1
DEV_BAD_SEQ_LEN = 2
DEV_BAD_QPOS = 4
DEV_SPLIT_OVERFLOW = 8
DEV_BAD_TIER = 16
DEV_TIMEOUT = 32

DA_OK = 0
DA_ERR_INVALID = -1
DA_ERR_UNSUPPORTED = -2
DA_ERR_WORKSPACE = -3
DA_ERR_CUDA = -4

_EXPORTS = (
    "decode_attn_paged", "decode_attn_paged_multi", "decode_attn_paged_sparse", "decode_attn_tiered_int8", "decode_attn_tiered_f16",
    "decode_attn_split_partial",
    "decode_attn_split_merge", "decode_attn_workspace_size", "decode_attn_workspace_init",
    "decode_attn_status_string", "decode_attn_paged_static_ws", "decode_attn_append_paged",
    "decode_attn_append_tiered_int8", "decode_attn_append_tiered_f16", "decode_attn_get_tuning",
    "decode_attn_set_tuning", "decode_attn_testing_skip_first_arm",
)


class DecodeAttnError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


class DaParams(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
        ("scale", ctypes.c_float), ("softcap", ctypes.c_float),
        ("sliding_window", ctypes.c_int32), ("causal", ctypes.c_int32),
    ]


class DaTierParams(ctypes.Structure):
    _fields_ = [
        ("hot_window", ctypes.c_int32), ("hot_capacity", ctypes.c_int32),
        ("cold_len", ctypes.c_int32), ("hot_len", ctypes.c_int32),
        ("hot_start", ctypes.c_int32),
        ("cold_lens", ctypes.c_void_p), ("hot_lens", ctypes.c_void_p),
        ("hot_starts", ctypes.c_void_p),
    ]


class DaSparseLayout(ctypes.Structure):
    _fields_ = [
        ("sparse_block", ctypes.c_int32), ("num_layouts", ctypes.c_int32),
        ("num_rows", ctypes.c_int32), ("max_nnz", ctypes.c_int32),
        ("row_ptr", ctypes.c_void_p), ("col_idx", ctypes.c_void_p),
    ]


class DaTuning(ctypes.Structure):
    _fields_ = [
        ("kv_heads_per_unit", ctypes.c_int32), ("fuse_head_groups", ctypes.c_int32),
        ("packed_operands", ctypes.c_int32), ("max_stages", ctypes.c_int32),
        ("wait_limit_ms", ctypes.c_int32), ("unsplit_max_len", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    return _build.build(force=force)


def load_library():
    """Load libdecode_attn.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing: build it first "
                "(quantized_kv_decode_paged_gb300.build() or __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        lib.decode_attn_paged.restype = ctypes.c_int
        lib.decode_attn_paged.argtypes = [ctypes.POINTER(DaParams), P, P, P, P, P, P, P, P, P,
                                          ctypes.c_size_t, P, P]
        lib.decode_attn_paged_multi.restype = ctypes.c_int
        lib.decode_attn_paged_multi.argtypes = [ctypes.POINTER(DaParams), i32, P, P, P, P, P, P,
                                                P, P, P, ctypes.c_size_t, P, P]
        lib.decode_attn_paged_sparse.restype = ctypes.c_int
        lib.decode_attn_paged_sparse.argtypes = [ctypes.POINTER(DaParams),
                                                 ctypes.POINTER(DaSparseLayout), P, P, P, P, P,
                                                 P, P, P, P, ctypes.c_size_t, P, P]
        lib.decode_attn_tiered_int8.restype = ctypes.c_int
        lib.decode_attn_tiered_int8.argtypes = [ctypes.POINTER(DaParams),
                                                ctypes.POINTER(DaTierParams), P, P, P, P, P, P,
                                                P, P, P, P, P, P, ctypes.c_size_t, P, P]
        lib.decode_attn_tiered_f16.restype = ctypes.c_int
        lib.decode_attn_tiered_f16.argtypes = [ctypes.POINTER(DaParams),
                                               ctypes.POINTER(DaTierParams), P, P, P, P, P, P,
                                               P, P, P, P, ctypes.c_size_t, P, P]
        lib.decode_attn_split_partial.restype = ctypes.c_int
        lib.decode_attn_split_partial.argtypes = [ctypes.POINTER(DaParams), i32, i32, P, P, P,
                                                  P, P, P, P, P, P, P]
        lib.decode_attn_split_merge.restype = ctypes.c_int
        lib.decode_attn_split_merge.argtypes = [i32, i32, i32, i32, P, P, P, P, P]
        lib.decode_attn_workspace_size.restype = ctypes.c_size_t
        lib.decode_attn_workspace_size.argtypes = [ctypes.POINTER(DaParams)]
        lib.decode_attn_workspace_init.restype = ctypes.c_int
        lib.decode_attn_workspace_init.argtypes = [P, ctypes.c_size_t, P]
        lib.decode_attn_paged_static_ws.restype = ctypes.c_int
        lib.decode_attn_paged_static_ws.argtypes = [ctypes.POINTER(DaParams), P, P, P, P, P,
                                                    P, P, P, P, P]
        lib.decode_attn_append_paged.restype = ctypes.c_int
        lib.decode_attn_append_paged.argtypes = [ctypes.POINTER(DaParams)] + [P] * 8
        lib.decode_attn_append_tiered_int8.restype = ctypes.c_int
        lib.decode_attn_append_tiered_int8.argtypes = ([ctypes.POINTER(DaParams), i32, i32]
                                                       + [P] * 14)
        lib.decode_attn_append_tiered_f16.restype = ctypes.c_int
        lib.decode_attn_append_tiered_f16.argtypes = ([ctypes.POINTER(DaParams), i32, i32]
                                                      + [P] * 12)
        lib.decode_attn_get_tuning.restype = ctypes.c_int
        lib.decode_attn_get_tuning.argtypes = [ctypes.POINTER(DaTuning)]
        lib.decode_attn_set_tuning.restype = ctypes.c_int
        lib.decode_attn_set_tuning.argtypes = [ctypes.POINTER(DaTuning)]
        lib.decode_attn_testing_skip_first_arm.restype = ctypes.c_int
        lib.decode_attn_testing_skip_first_arm.argtypes = [ctypes.c_int32]
        lib.decode_attn_status_string.restype = ctypes.c_char_p
        lib.decode_attn_status_string.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def decode_attn_status_string(status: int) -> str:
    return load_library().decode_attn_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != DA_OK:
        raise DecodeAttnError(fn, status, decode_attn_status_string(status))


# ---------------------------------------------------------------- tuning
def get_tuning() -> dict:
    """The library's current tuning (decode_attn_get_tuning) as a dict."""
    t = DaTuning()
    _check("decode_attn_get_tuning", load_library().decode_attn_get_tuning(ctypes.byref(t)))
    return {name: int(getattr(t, name)) for name, _ in DaTuning._fields_}


def set_tuning(**fields) -> None:
    """Replaces the named tuning fields, keeping the others
    (decode_attn_set_tuning).  With no fields: the load-time values."""
    lib = load_library()
    if not fields:
        _check("decode_attn_set_tuning", lib.decode_attn_set_tuning(None))
        return
    cur = get_tuning()
    unknown = set(fields) - set(cur)
    if unknown:
        raise TypeError(f"unknown tuning fields: {sorted(unknown)}")
    cur.update(fields)
    t = DaTuning(**{k: int(v) for k, v in cur.items()})
    _check("decode_attn_set_tuning", lib.decode_attn_set_tuning(ctypes.byref(t)))


class tuning:
    """Context manager: ``with tuning(packed_operands=0): ...`` sets the named
    fields for the block and puts the previous tuning back afterwards."""

    def __init__(self, **fields):
        self.fields = fields
        self.saved = None

    def __enter__(self):
        self.saved = get_tuning()
        set_tuning(**self.fields)
        return self

    def __exit__(self, *exc):
        set_tuning(**self.saved)
        return False


# ---------------------------------------------------------------- marshalling
def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _req(t, name, dtype, device, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t


def _stream(device, stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def make_params(q, block_size, num_kv_heads, max_blocks_per_seq, num_blocks, *, scale=0.0,
                softcap=0.0, sliding_window=0, causal=True, max_seq_len=0) -> DaParams:
    B, Hq, D = q.shape
    return DaParams(int(B), int(Hq), int(num_kv_heads), int(D), int(block_size),
                    int(max_blocks_per_seq), int(num_blocks), int(max_seq_len),
                    float(scale), float(softcap), int(sliding_window), int(bool(causal)))


_ws_cache: dict = {}


def decode_attn_workspace_size(params: DaParams) -> int:
    return int(load_library().decode_attn_workspace_size(ctypes.byref(params)))


def _auto_workspace(params: DaParams, device):
    """A zero-filled workspace cached per (device, size); kept zero between
    calls by the kernels."""
    torch = _torch()
    nbytes = decode_attn_workspace_size(params)
    if nbytes == 0:
        raise DecodeAttnError("decode_attn_workspace_size", DA_ERR_INVALID, "invalid parameters")
    key = (str(device), torch.cuda.current_stream(device).cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def _workspace_args(workspace, params, device):
    torch = _torch()
    if isinstance(workspace, str) and workspace == "auto":
        ws = _auto_workspace(params, device)
        return ws.data_ptr(), ws.numel()
    if workspace is None:
        return None, 0
    _req(workspace, "workspace", torch.uint8, device)
    return workspace.data_ptr(), workspace.numel()


def decode_attn_paged(q, k_pool, v_pool, block_table, seq_lens, q_pos=None, *, scale=0.0,
                      softcap=0.0, sliding_window=0, causal=True, max_seq_len=0, out=None,
                      lse=None, workspace="auto", dev_status=None, stream=None):
    """f16 paged decode attention.  Returns (out [B, Hq, D] f32, lse [B, Hq] f32).

    ``workspace``: "auto" (a cached zero-filled buffer), None (unsplit path),
    or a caller-owned zero-filled uint8 tensor of at least
    ``decode_attn_workspace_size`` bytes."""
    torch = _torch()
    lib = load_library()
    dev = q.device
    _req(q, "q", torch.float32, dev, 3)
    _req(k_pool, "k_pool", torch.float16, dev, 4)
    _req(v_pool, "v_pool", torch.float16, dev, 4)
    _req(block_table, "block_table", torch.int32, dev, 2)
    _req(seq_lens, "seq_lens", torch.int32, dev, 1)
    if q_pos is not None:
        _req(q_pos, "q_pos", torch.int32, dev, 1)
    if k_pool.shape != v_pool.shape:
        raise ValueError("k_pool and v_pool shapes differ")
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_pool.shape
    if D2 != D or block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    _req(out, "out", torch.float32, dev, 3)
    _req(lse, "lse", torch.float32, dev, 2)
    if dev_status is not None:
        _req(dev_status, "dev_status", torch.int32, dev)
    params = make_params(q, bs, Hkv, block_table.shape[1], NB, scale=scale, softcap=softcap,
                         sliding_window=sliding_window, causal=causal, max_seq_len=max_seq_len)
    ws_ptr, ws_bytes = _workspace_args(workspace, params, dev)
    st = lib.decode_attn_paged(ctypes.byref(params), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                               _ptr(block_table), _ptr(seq_lens), _ptr(q_pos), _ptr(out),
                               _ptr(lse), ws_ptr, ws_bytes, _ptr(dev_status),
                               _stream(dev, stream))
    _check("decode_attn_paged", st)
    return out, lse


def decode_attn_paged_multi(q, k_pool, v_pool, block_table, seq_lens, q_pos=None, *, scale=0.0,
                            softcap=0.0, sliding_window=0, causal=True, max_seq_len=0, out=None,
                            lse=None, workspace="auto", dev_status=None, stream=None):
    """Decode of T query tokens per sequence: q f32 [B, T, Hq, D]; token t sits
    at q_pos[b] + t (default seq_len - T + t).  Returns (out [B, T, Hq, D],
    lse [B, T, Hq])."""
    torch = _torch()
    lib = load_library()
    dev = q.device
    _req(q, "q", torch.float32, dev, 4)
    _req(k_pool, "k_pool", torch.float16, dev, 4)
    _req(v_pool, "v_pool", torch.float16, dev, 4)
    _req(block_table, "block_table", torch.int32, dev, 2)
    _req(seq_lens, "seq_lens", torch.int32, dev, 1)
    if q_pos is not None:
        _req(q_pos, "q_pos", torch.int32, dev, 1)
    if k_pool.shape != v_pool.shape:
        raise ValueError("k_pool and v_pool shapes differ")
    B, T, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_pool.shape
    if D2 != D or block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((B, T, Hq, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=dev)
    _req(out, "out", torch.float32, dev, 4)
    _req(lse, "lse", torch.float32, dev, 3)
    if dev_status is not None:
        _req(dev_status, "dev_status", torch.int32, dev)
    params = make_params(q[:, 0], bs, Hkv, block_table.shape[1], NB, scale=scale,
                         softcap=softcap, sliding_window=sliding_window, causal=causal,
                         max_seq_len=max_seq_len)
    ws_ptr, ws_bytes = _workspace_args(workspace, params, dev)
    st = lib.decode_attn_paged_multi(ctypes.byref(params), int(T), _ptr(q), _ptr(k_pool),
                                     _ptr(v_pool), _ptr(block_table), _ptr(seq_lens),
                                     _ptr(q_pos), _ptr(out), _ptr(lse), ws_ptr, ws_bytes,
                                     _ptr(dev_status), _stream(dev, stream))
    _check("decode_attn_paged_multi", st)
    return out, lse


def decode_attn_paged_static_ws(q, k_pool, v_pool, block_table, seq_lens, q_pos=None, *,
                                scale=0.0, softcap=0.0, sliding_window=0, causal=True,
                                max_seq_len=0, out=None, lse=None, dev_status=None, stream=None):
    """decode_attn_paged with its split-KV scratch in the library's own fixed
    buffer: for callers that must not allocate device memory.  The output
    tensors are still the caller's (allocated here only when not given)."""
    torch = _torch()
    lib = load_library()
    dev = q.device
    _req(q, "q", torch.float32, dev, 3)
    _req(k_pool, "k_pool", torch.float16, dev, 4)
    _req(v_pool, "v_pool", torch.float16, dev, 4)
    _req(block_table, "block_table", torch.int32, dev, 2)
    _req(seq_lens, "seq_lens", torch.int32, dev, 1)
    if q_pos is not None:
        _req(q_pos, "q_pos", torch.int32, dev, 1)
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_pool.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    params = make_params(q, bs, Hkv, block_table.shape[1], NB, scale=scale, softcap=softcap,
                         sliding_window=sliding_window, causal=causal, max_seq_len=max_seq_len)
    st = lib.decode_attn_paged_static_ws(ctypes.byref(params), _ptr(q), _ptr(k_pool),
                                         _ptr(v_pool), _ptr(block_table), _ptr(seq_lens),
                                         _ptr(q_pos), _ptr(out), _ptr(lse), _ptr(dev_status),
                                         _stream(dev, stream))
    _check("decode_attn_paged_static_ws", st)
    return out, lse


def decode_attn_paged_sparse(q, k_pool, v_pool, block_table, seq_lens, row_ptr, col_idx,
                             sparse_block, q_pos=None, *, max_seq_len, scale=0.0, softcap=0.0,
                             sliding_window=0, causal=True, out=None, lse=None, workspace="auto",
                             dev_status=None, stream=None):
    """Block-sparse paged decode attention (one query token per sequence).
    Head h keeps the keys of the blocks that CSR row q_pos / sparse_block of
    layout h % num_layouts lists.  row_ptr int32 [num_layouts, num_rows + 1]
    and col_idx int32 [num_layouts, max_nnz] on the device; max_seq_len (> 0)
    bounds seq_lens.  Returns (out [B, Hq, D] f32, lse [B, Hq] f32)."""
    torch = _torch()
    lib = load_library()
    dev = q.device
    _req(q, "q", torch.float32, dev, 3)
    _req(k_pool, "k_pool", torch.float16, dev, 4)
    _req(v_pool, "v_pool", torch.float16, dev, 4)
    _req(block_table, "block_table", torch.int32, dev, 2)
    _req(seq_lens, "seq_lens", torch.int32, dev, 1)
    _req(row_ptr, "row_ptr", torch.int32, dev, 2)
    _req(col_idx, "col_idx", torch.int32, dev, 2)
    if q_pos is not None:
        _req(q_pos, "q_pos", torch.int32, dev, 1)
    if k_pool.shape != v_pool.shape:
        raise ValueError("k_pool and v_pool shapes differ")
    if row_ptr.shape[0] != col_idx.shape[0]:
        raise ValueError("row_ptr and col_idx describe different numbers of layouts")
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_pool.shape
    if D2 != D or block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    _req(out, "out", torch.float32, dev, 3)
    _req(lse, "lse", torch.float32, dev, 2)
    if dev_status is not None:
        _req(dev_status, "dev_status", torch.int32, dev)
    params = make_params(q, bs, Hkv, block_table.shape[1], NB, scale=scale, softcap=softcap,
                         sliding_window=sliding_window, causal=causal, max_seq_len=max_seq_len)
    sl = DaSparseLayout(int(sparse_block), int(row_ptr.shape[0]), int(row_ptr.shape[1] - 1),
                        int(col_idx.shape[1]), _ptr(row_ptr), _ptr(col_idx))
    ws_ptr, ws_bytes = _workspace_args(workspace, params, dev)
    st = lib.decode_attn_paged_sparse(ctypes.byref(params), ctypes.byref(sl), _ptr(q),
                                      _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                      _ptr(seq_lens), _ptr(q_pos), _ptr(out), _ptr(lse), ws_ptr,
                                      ws_bytes, _ptr(dev_status), _stream(dev, stream))
    _check("decode_attn_paged_sparse", st)
    return out, lse


def decode_attn_tiered_int8(q, k_hot, v_hot, k_cold, v_cold, k_scale, v_scale, block_table, *,
                            hot_window, cold_len=0, hot_len=0, hot_start=0, cold_lens=None,
                            hot_lens=None, hot_starts=None, q_pos=None, scale=0.0, softcap=0.0,
                            sliding_window=0, causal=True, max_seq_len=0, out=None, lse=None,
                            workspace="auto", dev_status=None, stream=None):
    """Decode attention over an int8 cold tier (paged) and an f16 hot ring.

    k_hot/v_hot f16 [B, hot_capacity, Hkv, D]; k_cold/v_cold int32 or uint32
    words [NB, bs, Hkv, D/4]; k_scale/v_scale f16 [NB, bs, Hkv].
    Returns (out, lse)."""
    torch = _torch()
    lib = load_library()
    dev = q.device
    _req(q, "q", torch.float32, dev, 3)
    _req(k_hot, "k_hot", torch.float16, dev, 4)
    _req(v_hot, "v_hot", torch.float16, dev, 4)
    for name, t in (("k_cold", k_cold), ("v_cold", v_cold)):
        if t.dtype not in (torch.int32, torch.uint32):
            raise TypeError(f"{name} must hold 32-bit words")
        _req(t, name, t.dtype, dev, 4)
    _req(k_scale, "k_scale", torch.float16, dev, 3)
    _req(v_scale, "v_scale", torch.float16, dev, 3)
    _req(block_table, "block_table", torch.int32, dev, 2)
    for name, t in (("cold_lens", cold_lens), ("hot_lens", hot_lens), ("hot_starts", hot_starts),
                    ("q_pos", q_pos)):
        if t is not None:
            _req(t, name, torch.int32, dev, 1)
    B, Hq, D = q.shape
    NB, bs, Hkv, W4 = k_cold.shape
    cap = k_hot.shape[1]
    if W4 * 4 != D or k_hot.shape != (B, cap, Hkv, D) or v_hot.shape != k_hot.shape:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    params = make_params(q, bs, Hkv, block_table.shape[1], NB, scale=scale, softcap=softcap,
                         sliding_window=sliding_window, causal=causal, max_seq_len=max_seq_len)
    tier = DaTierParams(int(hot_window), int(cap), int(cold_len), int(hot_len), int(hot_start),
                        _ptr(cold_lens), _ptr(hot_lens), _ptr(hot_starts))
    ws_ptr, ws_bytes = _workspace_args(workspace, params, dev)
    st = lib.decode_attn_tiered_int8(ctypes.byref(params), ctypes.byref(tier), _ptr(q),
                                     _ptr(k_hot), _ptr(v_hot), _ptr(k_cold), _ptr(v_cold),
                                     _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(q_pos),
                                     _ptr(out), _ptr(lse), ws_ptr, ws_bytes, _ptr(dev_status),
                                     _stream(dev, stream))
    _check("decode_attn_tiered_int8", st)
    return out, lse


def decode_attn_tiered_f16(q, k_hot, v_hot, k_cold, v_cold, block_table, *, hot_window,
                           cold_len=0, hot_len=0, hot_start=0, cold_lens=None, hot_lens=None,
                           hot_starts=None, q_pos=None, scale=0.0, softcap=0.0,
                           sliding_window=0, causal=True, max_seq_len=0, out=None, lse=None,
                           workspace="auto", dev_status=None, stream=None):
    """Decode attention over an f16 cold tier (paged) and an f16 hot ring.

    k_hot/v_hot f16 [B, hot_capacity, Hkv, D]; k_cold/v_cold f16 [NB, bs, Hkv, D].
    Tier arguments as for decode_attn_tiered_int8.  Returns (out, lse)."""
    torch = _torch()
    lib = load_library()
    dev = q.device
    _req(q, "q", torch.float32, dev, 3)
    _req(k_hot, "k_hot", torch.float16, dev, 4)
    _req(v_hot, "v_hot", torch.float16, dev, 4)
    _req(k_cold, "k_cold", torch.float16, dev, 4)
    _req(v_cold, "v_cold", torch.float16, dev, 4)
    _req(block_table, "block_table", torch.int32, dev, 2)
    for name, t in (("cold_lens", cold_lens), ("hot_lens", hot_lens), ("hot_starts", hot_starts),
                    ("q_pos", q_pos)):
        if t is not None:
            _req(t, name, torch.int32, dev, 1)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cold.shape
    cap = k_hot.shape[1]
    if (D2 != D or v_cold.shape != k_cold.shape or k_hot.shape != (B, cap, Hkv, D)
            or v_hot.shape != k_hot.shape):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    params = make_params(q, bs, Hkv, block_table.shape[1], NB, scale=scale, softcap=softcap,
                         sliding_window=sliding_window, causal=causal, max_seq_len=max_seq_len)
    tier = DaTierParams(int(hot_window), int(cap), int(cold_len), int(hot_len), int(hot_start),
                        _ptr(cold_lens), _ptr(hot_lens), _ptr(hot_starts))
    ws_ptr, ws_bytes = _workspace_args(workspace, params, dev)
    st = lib.decode_attn_tiered_f16(ctypes.byref(params), ctypes.byref(tier), _ptr(q),
                                    _ptr(k_hot), _ptr(v_hot), _ptr(k_cold), _ptr(v_cold),
                                    _ptr(block_table), _ptr(q_pos), _ptr(out), _ptr(lse), ws_ptr,
                                    ws_bytes, _ptr(dev_status), _stream(dev, stream))
    _check("decode_attn_tiered_f16", st)
    return out, lse


def decode_attn_split_partial(q, k_pool, v_pool, block_table, seq_lens, q_pos=None, *,
                              split_tokens, max_splits, scale=0.0, softcap=0.0,
                              sliding_window=0, causal=True, o_part=None, lse_part=None,
                              dev_status=None, stream=None):
    """Per-split partial states: (o_part [B, Hq, S, D], lse_part [B, Hq, S])."""
    torch = _torch()
    lib = load_library()
    dev = q.device
    _req(q, "q", torch.float32, dev, 3)
    _req(k_pool, "k_pool", torch.float16, dev, 4)
    _req(v_pool, "v_pool", torch.float16, dev, 4)
    _req(block_table, "block_table", torch.int32, dev, 2)
    _req(seq_lens, "seq_lens", torch.int32, dev, 1)
    if q_pos is not None:
        _req(q_pos, "q_pos", torch.int32, dev, 1)
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_pool.shape
    if o_part is None:
        o_part = torch.empty((B, Hq, max_splits, D), dtype=torch.float32, device=dev)
    if lse_part is None:
        lse_part = torch.empty((B, Hq, max_splits), dtype=torch.float32, device=dev)
    params = make_params(q, bs, Hkv, block_table.shape[1], NB, scale=scale, softcap=softcap,
                         sliding_window=sliding_window, causal=causal)
    st = lib.decode_attn_split_partial(ctypes.byref(params), int(split_tokens), int(max_splits),
                                       _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                       _ptr(seq_lens), _ptr(q_pos), _ptr(o_part), _ptr(lse_part),
                                       _ptr(dev_status), _stream(dev, stream))
    _check("decode_attn_split_partial", st)
    return o_part, lse_part


def decode_attn_split_merge(o_part, lse_part, *, out=None, lse=None, stream=None):
    """Merge split partial states into (out [B, Hq, D], lse [B, Hq])."""
    torch = _torch()
    lib = load_library()
    dev = o_part.device
    _req(o_part, "o_part", torch.float32, dev, 4)
    _req(lse_part, "lse_part", torch.float32, dev, 3)
    B, Hq, S, D = o_part.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    st = lib.decode_attn_split_merge(B, Hq, D, S, _ptr(o_part), _ptr(lse_part), _ptr(out),
                                     _ptr(lse), _stream(dev, stream))
    _check("decode_attn_split_merge", st)
    return out, lse


# ---------------------------------------------------------------------------
# KV append
# ---------------------------------------------------------------------------

def _append_params(k_new, block_table, pool_shape):
    B, Hkv, D = k_new.shape
    NB, bs = pool_shape[0], pool_shape[1]
    return DaParams(B, Hkv, Hkv, D, bs, block_table.shape[1], NB, 0, 0.0, 0.0, 0, 1)


def decode_attn_append_paged(k_new, v_new, positions, block_table, k_pool, v_pool, *,
                             dev_status=None, stream=None):
    """Writes k_new/v_new f16 [B, Hkv, D] into the paged pools [NB, bs, Hkv, D]
    at positions i32 [B] (in place)."""
    torch = _torch()
    lib = load_library()
    dev = k_new.device
    _req(k_new, "k_new", torch.float16, dev, 3)
    _req(v_new, "v_new", torch.float16, dev, 3)
    _req(positions, "positions", torch.int32, dev, 1)
    _req(block_table, "block_table", torch.int32, dev, 2)
    _req(k_pool, "k_pool", torch.float16, dev, 4)
    _req(v_pool, "v_pool", torch.float16, dev, 4)
    if (v_new.shape != k_new.shape or v_pool.shape != k_pool.shape
            or k_pool.shape[2:] != k_new.shape[1:] or positions.shape[0] != k_new.shape[0]):
        raise ValueError("inconsistent shapes")
    params = _append_params(k_new, block_table, k_pool.shape)
    st = lib.decode_attn_append_paged(ctypes.byref(params), _ptr(k_new), _ptr(v_new),
                                      _ptr(positions), _ptr(block_table), _ptr(k_pool),
                                      _ptr(v_pool), _ptr(dev_status), _stream(dev, stream))
    _check("decode_attn_append_paged", st)


def _tier_state_checks(torch, dev, k_new, v_new, k_hot, v_hot, block_table, cold_lens, hot_lens,
                       hot_starts):
    _req(k_new, "k_new", torch.float16, dev, 3)
    _req(v_new, "v_new", torch.float16, dev, 3)
    _req(k_hot, "k_hot", torch.float16, dev, 4)
    _req(v_hot, "v_hot", torch.float16, dev, 4)
    _req(block_table, "block_table", torch.int32, dev, 2)
    for name, t in (("cold_lens", cold_lens), ("hot_lens", hot_lens), ("hot_starts", hot_starts)):
        _req(t, name, torch.int32, dev, 1)
    B, Hkv, D = k_new.shape
    if (v_new.shape != k_new.shape or k_hot.shape[0] != B or k_hot.shape[2:] != (Hkv, D)
            or v_hot.shape != k_hot.shape):
        raise ValueError("inconsistent shapes")


def decode_attn_append_tiered_int8(k_new, v_new, k_hot, v_hot, k_cold, v_cold, k_scale, v_scale,
                                   block_table, cold_lens, hot_lens, hot_starts, *, hot_window,
                                   dev_status=None, stream=None):
    """One append step of an int8-cold / f16-hot tiered cache (in place): the
    oldest hot token of a full ring is quantized into the cold tier, then the
    new token enters the ring; cold_lens/hot_lens/hot_starts are updated."""
    torch = _torch()
    lib = load_library()
    dev = k_new.device
    _tier_state_checks(torch, dev, k_new, v_new, k_hot, v_hot, block_table, cold_lens, hot_lens,
                       hot_starts)
    for name, t in (("k_cold", k_cold), ("v_cold", v_cold)):
        if t.dtype not in (torch.int32, torch.uint32):
            raise TypeError(f"{name} must hold 32-bit words")
        _req(t, name, t.dtype, dev, 4)
    _req(k_scale, "k_scale", torch.float16, dev, 3)
    _req(v_scale, "v_scale", torch.float16, dev, 3)
    if k_cold.shape[3] * 4 != k_new.shape[2] or v_cold.shape != k_cold.shape:
        raise ValueError("inconsistent shapes")
    params = _append_params(k_new, block_table, k_cold.shape)
    st = lib.decode_attn_append_tiered_int8(
        ctypes.byref(params), int(hot_window), int(k_hot.shape[1]), _ptr(k_new), _ptr(v_new),
        _ptr(k_hot), _ptr(v_hot), _ptr(k_cold), _ptr(v_cold), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_table), _ptr(cold_lens), _ptr(hot_lens), _ptr(hot_starts), _ptr(dev_status),
        _stream(dev, stream))
    _check("decode_attn_append_tiered_int8", st)


def decode_attn_append_tiered_f16(k_new, v_new, k_hot, v_hot, k_cold, v_cold, block_table,
                                  cold_lens, hot_lens, hot_starts, *, hot_window,
                                  dev_status=None, stream=None):
    """As decode_attn_append_tiered_int8 for an f16 cold tier [NB, bs, Hkv, D]."""
    torch = _torch()
    lib = load_library()
    dev = k_new.device
    _tier_state_checks(torch, dev, k_new, v_new, k_hot, v_hot, block_table, cold_lens, hot_lens,
                       hot_starts)
    _req(k_cold, "k_cold", torch.float16, dev, 4)
    _req(v_cold, "v_cold", torch.float16, dev, 4)
    if k_cold.shape[2:] != k_new.shape[1:] or v_cold.shape != k_cold.shape:
        raise ValueError("inconsistent shapes")
    params = _append_params(k_new, block_table, k_cold.shape)
    st = lib.decode_attn_append_tiered_f16(
        ctypes.byref(params), int(hot_window), int(k_hot.shape[1]), _ptr(k_new), _ptr(v_new),
        _ptr(k_hot), _ptr(v_hot), _ptr(k_cold), _ptr(v_cold), _ptr(block_table),
        _ptr(cold_lens), _ptr(hot_lens), _ptr(hot_starts), _ptr(dev_status), _stream(dev, stream))
    _check("decode_attn_append_tiered_f16", st)
