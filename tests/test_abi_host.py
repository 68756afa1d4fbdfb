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


# ---------------------------------------------------------------------------
# tuning state
# ---------------------------------------------------------------------------

DEFAULT_TUNING = dict(kv_heads_per_unit=0, fuse_head_groups=1, packed_operands=1, max_stages=0,
                      wait_limit_ms=2000, unsplit_max_len=512)


def test_tuning_defaults_set_validate_and_restore(lib):
    qk.set_tuning()
    assert qk.get_tuning() == DEFAULT_TUNING or os.environ.get("DA_KVB") is not None
    with qk.tuning(packed_operands=0, max_stages=3):
        t = qk.get_tuning()
        assert t["packed_operands"] == 0 and t["max_stages"] == 3
        assert t["fuse_head_groups"] == 1
    assert qk.get_tuning()["packed_operands"] == 1
    for bad in (dict(kv_heads_per_unit=3), dict(fuse_head_groups=2), dict(packed_operands=-1),
                dict(max_stages=1), dict(max_stages=9), dict(wait_limit_ms=0),
                dict(wait_limit_ms=10001), dict(unsplit_max_len=-1),
                dict(unsplit_max_len=65537)):
        before = qk.get_tuning()
        with pytest.raises(qk.DecodeAttnError):
            qk.set_tuning(**bad)
        assert qk.get_tuning() == before, bad
    assert lib.decode_attn_get_tuning(None) == qk.DA_ERR_INVALID
    assert lib.decode_attn_testing_skip_first_arm(2) == qk.DA_ERR_INVALID


_LOAD_TIME_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import quantized_kv_decode_paged_gb300 as qk
qk.load_library()
first = qk.get_tuning()
# the environment is read at load only: later changes have no effect
os.environ["DA_PACK"] = "1"
os.environ["DA_MAX_STAGES"] = "2"
qk.set_tuning()
print(json.dumps([first, qk.get_tuning()]))
"""


def test_environment_is_read_once_at_load(lib):
    import json
    import subprocess
    import sys
    env = dict(os.environ, DA_PACK="0", DA_KVB="4", DA_FUSE_HG="0", DA_MAX_STAGES="5",
               DA_WAIT_LIMIT_MS="750", DA_UNSPLIT_MAX_LEN="0", DA_TEST_SKIP_ARM="1")
    r = subprocess.run([sys.executable, "-c", _LOAD_TIME_SCRIPT, ROOT], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    first, restored = json.loads(r.stdout.strip().splitlines()[-1])
    want = dict(kv_heads_per_unit=4, fuse_head_groups=0, packed_operands=0, max_stages=5,
                wait_limit_ms=750, unsplit_max_len=0)
    assert first == want and restored == want
    # out-of-range values keep the defaults
    env = dict(os.environ, DA_PACK="7", DA_KVB="3", DA_MAX_STAGES="1", DA_WAIT_LIMIT_MS="x",
               DA_UNSPLIT_MAX_LEN="70000")
    r = subprocess.run([sys.executable, "-c", _LOAD_TIME_SCRIPT, ROOT], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    first, _ = json.loads(r.stdout.strip().splitlines()[-1])
    assert first == DEFAULT_TUNING


def test_no_environment_read_per_call():
    """The library source reads the environment in one place: the load-time
    tuning reader."""
    import pathlib
    csrc = pathlib.Path(ROOT) / "quantized_kv_decode_paged_gb300" / "csrc"
    hits = [(f.name, ln) for f in sorted(csrc.iterdir()) if f.suffix in (".cu", ".cuh", ".h")
            for ln in f.read_text().splitlines() if "getenv" in ln]
    assert len(hits) == 1 and hits[0][0] == "api.cu", hits
    assert not any("DA_TEST" in f.read_text() for f in csrc.iterdir() if f.is_file())


def test_tuning_from_many_threads(lib):
    """Host threads setting and reading the tuning at once always see valid
    values, and the calls return OK."""
    import threading
    errors = []

    def worker(i):
        try:
            for j in range(300):
                t = qk.DaTuning(kv_heads_per_unit=(0, 1, 2, 4)[(i + j) % 4],
                                fuse_head_groups=j % 2, packed_operands=(j // 2) % 2,
                                max_stages=(0, 2, 3, 8)[j % 4], wait_limit_ms=1 + j,
                                unsplit_max_len=(0, 512, 65536)[j % 3])
                assert lib.decode_attn_set_tuning(ctypes.byref(t)) == qk.DA_OK
                g = qk.DaTuning()
                assert lib.decode_attn_get_tuning(ctypes.byref(g)) == qk.DA_OK
                assert g.kv_heads_per_unit in (0, 1, 2, 4) and g.max_stages in (0, 2, 3, 8)
                assert 1 <= g.wait_limit_ms <= 300 and g.unsplit_max_len in (0, 512, 65536)
        except Exception as e:  # pragma: no cover
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    qk.set_tuning()
    assert not errors, errors


def test_sparse_rejects_bad_layouts(lib):
    p = _params()
    good = dict(sparse_block=64, num_layouts=2, num_rows=4, max_nnz=8, row_ptr=FAKE.value,
                col_idx=FAKE.value)

    def call(pp=p, **kw):
        sl = qk.DaSparseLayout(**{**good, **kw})
        return lib.decode_attn_paged_sparse(ctypes.byref(pp), ctypes.byref(sl), FAKE, FAKE, FAKE,
                                            FAKE, FAKE, None, FAKE, None, None, 0, None, None)

    for bad in (dict(sparse_block=48), dict(sparse_block=8), dict(num_layouts=0),
                dict(num_rows=0), dict(max_nnz=-1), dict(row_ptr=None)):
        assert call(**bad) == qk.DA_ERR_INVALID, bad
    assert call(pp=_params(max_seq_len=0)) == qk.DA_ERR_INVALID
    assert call(pp=_params(head_dim=96)) == qk.DA_ERR_UNSUPPORTED
    assert lib.decode_attn_paged_sparse(ctypes.byref(p), None, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                        FAKE, None, None, 0, None, None) == qk.DA_ERR_INVALID
    assert call(pp=_params(batch=0)) == qk.DA_OK
