"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function the header declares, and rejects bad arguments before any
CUDA call."""
import ctypes
import os
import re

import pytest

import quantized_kv_decode_paged_gb300 as qk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "decode_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(decode_attn_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    qk.build()
    return qk.load_library()


def test_header_declares_the_boundary():
    fns = _header_functions()
    for name in ("decode_attn_paged", "decode_attn_tiered_int8", "decode_attn_split_partial",
                 "decode_attn_split_merge", "decode_attn_workspace_size"):
        assert name in fns


def test_library_exports_every_declared_function(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name


def _header_arity():
    src = open(os.path.join(ROOT, "include", "decode_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(decode_attn_\w+)\s*\(([^)]*)\)\s*;", src):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_argument_counts_match_the_header(lib):
    """Every ctypes prototype the binding sets has as many arguments as the
    header declares (a mismatch would misplace every later argument)."""
    arity = _header_arity()
    assert set(arity) == set(_header_functions())
    for name, n in arity.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None and len(fn.argtypes) == n, (name, n, fn.argtypes)


def test_status_strings(lib):
    assert qk.decode_attn_status_string(0) == "ok"
    assert "invalid" in qk.decode_attn_status_string(-1)
    assert "unsupported" in qk.decode_attn_status_string(-2)
    assert "workspace" in qk.decode_attn_status_string(-3)


def _params(**kw):
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                max_blocks_per_seq=4, num_blocks=8, max_seq_len=64, scale=0.0, softcap=0.0,
                sliding_window=0, causal=1)
    base.update(kw)
    return qk.DaParams(**base)


FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: validation fails first


@pytest.mark.parametrize("kw,status", [
    (dict(num_q_heads=7), qk.DA_ERR_INVALID),
    (dict(head_dim=96), qk.DA_ERR_UNSUPPORTED),
    (dict(block_size=12), qk.DA_ERR_UNSUPPORTED),
    (dict(block_size=4), qk.DA_ERR_UNSUPPORTED),
    (dict(scale=-1.0), qk.DA_ERR_INVALID),
    (dict(softcap=-2.0), qk.DA_ERR_INVALID),
    (dict(sliding_window=-1), qk.DA_ERR_INVALID),
    (dict(causal=2), qk.DA_ERR_INVALID),
    (dict(num_blocks=0), qk.DA_ERR_INVALID),
])
def test_paged_rejects_bad_params(lib, kw, status):
    p = _params(**kw)
    st = lib.decode_attn_paged(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None,
                               None, 0, None, None)
    assert st == status


def test_paged_rejects_null_and_misaligned(lib):
    p = _params()
    st = lib.decode_attn_paged(ctypes.byref(p), None, FAKE, FAKE, FAKE, FAKE, None, FAKE, None,
                               None, 0, None, None)
    assert st == qk.DA_ERR_INVALID
    odd = ctypes.c_void_p(0x10004)
    st = lib.decode_attn_paged(ctypes.byref(p), odd, FAKE, FAKE, FAKE, FAKE, None, FAKE, None,
                               None, 0, None, None)
    assert st == qk.DA_ERR_INVALID
    # a byte count without a workspace pointer
    st = lib.decode_attn_paged(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None,
                               None, 64, None, None)
    assert st == qk.DA_ERR_INVALID


def test_split_rejects_bad_split_sizes(lib):
    p = _params()
    for st_tokens, splits in ((0, 4), (24, 4), (16, 0)):
        st = lib.decode_attn_split_partial(ctypes.byref(p), st_tokens, splits, FAKE, FAKE, FAKE,
                                           FAKE, FAKE, None, FAKE, FAKE, None, None)
        assert st == qk.DA_ERR_INVALID


def test_merge_rejects_bad_sizes(lib):
    assert lib.decode_attn_split_merge(2, 0, 128, 4, FAKE, FAKE, FAKE, None, None) == qk.DA_ERR_INVALID
    assert lib.decode_attn_split_merge(2, 4, 128, 0, FAKE, FAKE, FAKE, None, None) == qk.DA_ERR_INVALID


def test_tiered_rejects_bad_tier(lib):
    p = _params(head_dim=128)
    def call(t, pp=p):
        return lib.decode_attn_tiered_int8(ctypes.byref(pp), ctypes.byref(t), FAKE, FAKE, FAKE,
                                           FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, None,
                                           0, None, None)
    good = dict(hot_window=16, hot_capacity=16, cold_len=32, hot_len=8, hot_start=32,
                cold_lens=None, hot_lens=None, hot_starts=None)
    for bad in (dict(hot_len=17), dict(hot_capacity=8), dict(hot_window=-1), dict(cold_len=-1),
                dict(cold_len=65), dict(hot_start=-3)):
        t = qk.DaTierParams(**{**good, **bad})
        assert call(t) == qk.DA_ERR_INVALID, bad
    assert call(qk.DaTierParams(**good), _params(head_dim=64)) == qk.DA_ERR_UNSUPPORTED


def test_tiered_f16_rejects_bad_tier(lib):
    p = _params(head_dim=128)
    def call(t, pp=p, k_cold=FAKE):
        return lib.decode_attn_tiered_f16(ctypes.byref(pp), ctypes.byref(t), FAKE, FAKE, FAKE,
                                          k_cold, FAKE, FAKE, None, FAKE, None, None, 0, None,
                                          None)
    good = dict(hot_window=16, hot_capacity=16, cold_len=32, hot_len=8, hot_start=32,
                cold_lens=None, hot_lens=None, hot_starts=None)
    for bad in (dict(hot_len=17), dict(hot_capacity=8), dict(hot_window=-1), dict(cold_len=-1),
                dict(cold_len=65), dict(hot_start=-3)):
        t = qk.DaTierParams(**{**good, **bad})
        assert call(t) == qk.DA_ERR_INVALID, bad
    assert call(qk.DaTierParams(**good), k_cold=None) == qk.DA_ERR_INVALID
    assert call(qk.DaTierParams(**good), _params(head_dim=96)) == qk.DA_ERR_UNSUPPORTED


def test_batch_zero_is_a_no_op(lib):
    p = _params(batch=0)
    st = lib.decode_attn_paged(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None,
                               None, 0, None, None)
    assert st == qk.DA_OK


def test_product_package_does_not_import_the_oracle():
    import pathlib
    pkg = pathlib.Path(ROOT) / "quantized_kv_decode_paged_gb300"
    for f in pkg.rglob("*.py"):
        src = f.read_text()
        assert "import oracle" not in src and "from oracle" not in src, f
    for f in list(pkg.rglob("*.cu")) + list(pkg.rglob("*.cuh")) + list(pkg.rglob("*.h")):
        assert "oracle" not in f.read_text().lower(), f
