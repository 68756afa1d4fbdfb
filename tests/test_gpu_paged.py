"""GPU parity of the f16 paged decode path against the double-precision
oracle, through the C ABI (via the ctypes binding)."""
import math

import numpy as np
import pytest

import oracle
import quantized_kv_decode_paged_gb300 as qk
from quantized_kv_decode_paged_gb300 import workloads as wl
from parity import assert_parity, oracle_paged, run_paged

pytestmark = pytest.mark.gpu

MODES = ("stream", "auto", "units", "split")


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    import torch
    torch.cuda.empty_cache()


def _case(seed, D, Hq, Hkv, bs, lens, **kw):
    B = len(lens)
    pages = sum((max(L, 0) + bs - 1) // bs for L in lens)
    return wl.make_paged(f"edge{seed}", seed, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                         seq_lens=lens, num_blocks=pages + 3, **kw)


def _check_all_rows(case, mode, **run_kw):
    t = case.device_tensors("cuda")
    out, lse = run_paged(case, t, mode, **run_kw)
    ref_out, ref_lse, _ = oracle_paged(case)
    assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse,
                  f"{case.name}/{mode}")


def test_tiny_workload_all_modes():
    case = wl.workload("tiny")
    t = case.device_tensors("cuda")
    ref_out, ref_lse, flags = oracle_paged(case)
    assert flags == 0
    for mode in MODES:
        out, lse = run_paged(case, t, mode, split_tokens=64)
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse, f"tiny/{mode}")


EDGE_LENS = [1, 7, 8, 9, 15, 16, 17, 63, 64, 65, 127, 128, 129, 200, 511, 777]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 8, 16])
def test_head_dims_and_group_sizes(D, G):
    Hkv = 2
    case = _case(100 + D + G, D, G * Hkv, Hkv, 16, EDGE_LENS[:: 2 if D == 256 else 1])
    for mode in MODES:
        _check_all_rows(case, mode)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 3, 4])
def test_unpacked_variant_for_small_groups(D, G):
    """Groups of at most four heads normally pack the f16 and remainder parts
    of Q and P into one MMA operand; the tuning's packed_operands=0 selects
    the two-operand variant, which must agree with the oracle as well."""
    with qk.tuning(packed_operands=0):
        Hkv = 2
        case = _case(150 + D + G, D, G * Hkv, Hkv, 16, EDGE_LENS[:: 2 if D == 256 else 1])
        for mode in MODES:
            _check_all_rows(case, mode)


@pytest.mark.parametrize("fuse", ["1", "0"])
@pytest.mark.parametrize("D,G,Hkv", [(64, 16, 4), (128, 12, 2), (128, 16, 2), (128, 16, 4),
                                     (128, 32, 2), (256, 16, 2)])
def test_head_groups_sharing_a_unit(D, G, Hkv, fuse):
    """More than eight query heads per kv head: two or four head groups of
    a kv head share one unit (each K/V byte read once); the tuning's
    fuse_head_groups=0 keeps a unit per head group.  Both must agree with the oracle, including a
    partial last group (G = 12)."""
    with qk.tuning(fuse_head_groups=int(fuse)):
        case = _case(700 + D + G + Hkv, D, G * Hkv, Hkv, 16, EDGE_LENS[::2])
        for mode in MODES:
            _check_all_rows(case, mode)


@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128, 256])
def test_block_sizes(bs):
    case = _case(200 + bs, 128, 8, 2, bs, [1, bs - 1, bs, bs + 1, 3 * bs + 5, 700])
    for mode in MODES:
        _check_all_rows(case, mode, split_tokens=max(bs, 128))


@pytest.mark.parametrize("window,softcap", [(1, 0.0), (7, 0.0), (100, 5.0), (300, 50.0),
                                            (0, 2.0)])
def test_window_and_softcap(window, softcap):
    case = _case(300 + window, 128, 8, 2, 16, [1, 5, 64, 99, 150, 400, 1000],
                 sliding_window=window, softcap=softcap)
    for mode in MODES:
        _check_all_rows(case, mode)


def test_non_causal_and_explicit_query_positions():
    lens = [10, 100, 300, 64, 1]
    q_pos = [3, 99, 500, 0, 0]
    for causal in (True, False):
        case = _case(400 + causal, 128, 8, 2, 16, lens, q_pos=q_pos, causal=causal,
                     sliding_window=37)
        for mode in MODES:
            _check_all_rows(case, mode)


def test_empty_sequences():
    case = _case(500, 128, 8, 2, 16, [0, 5, 0, 300, 0])
    for mode in MODES:
        _check_all_rows(case, mode)
    out, lse = run_paged(case, case.device_tensors("cuda"), "stream")
    assert not out[0].any() and np.isneginf(lse[0]).all()


def test_non_finite_rows_past_the_end_do_not_leak():
    case = _case(600, 128, 8, 2, 16, [3, 17, 50, 129], nonfinite_tail=True)
    for mode in MODES:
        _check_all_rows(case, mode)


def test_bad_block_ids_are_masked_and_flagged():
    import torch
    case = _case(700, 128, 8, 2, 16, [100, 300, 64])
    bt = case.block_table.copy()
    bt[0, 2] = case.num_blocks + 5
    bt[1, 7] = -9
    case.block_table = bt
    ref_out, ref_lse, flags = oracle_paged(case)
    assert flags & oracle.FLAG_BAD_BLOCK
    t = case.device_tensors("cuda")
    for mode in MODES:
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, lse = run_paged(case, t, mode, dev_status=st)
        assert int(st.item()) & qk.DEV_BAD_BLOCK, mode
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse, f"badblock/{mode}")


def test_length_beyond_table_is_clamped_and_flagged():
    import torch
    case = _case(800, 128, 8, 2, 16, [64, 100])
    case.seq_lens = np.array([64, 100 + 10_000], np.int32)  # table holds 7 pages
    ref_out, ref_lse, flags = oracle_paged(case)
    assert flags & oracle.FLAG_BAD_SEQ_LEN
    t = case.device_tensors("cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_paged(case, t, "stream", dev_status=st)
    assert int(st.item()) & qk.DEV_BAD_SEQ_LEN
    assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse, "clamp")


def test_negative_query_position_flags_and_empties():
    import torch
    case = _case(900, 128, 8, 2, 16, [64, 100], q_pos=[-1, 50])
    ref_out, ref_lse, _ = oracle_paged(case)
    t = case.device_tensors("cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_paged(case, t, "stream", dev_status=st)
    assert int(st.item()) & qk.DEV_BAD_QPOS
    assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse, "qpos")


def test_large_batch_is_chunked():
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 300, size=300).tolist()
    case = _case(1000, 64, 4, 2, 16, lens)
    for mode in MODES:
        _check_all_rows(case, mode)


def test_repeated_calls_are_stable():
    """The stream schedule leaves its ticket counters at zero: calling again
    (same workspace) must give the same bits."""
    case = _case(1100, 128, 32, 8, 16, [4096, 3000, 17, 2500])
    t = case.device_tensors("cuda")
    a = run_paged(case, t, "stream")
    for _ in range(3):
        b = run_paged(case, t, "stream")
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_workspace_reuse_across_shapes():
    """One zero-filled workspace serves calls of different head dims and
    batch shapes: only its leading ticket counters must stay zero."""
    import torch
    big = _case(1200, 256, 8, 2, 16, [777, 511, 129, 64, 3])
    cases = [big, _case(1201, 64, 8, 2, 16, EDGE_LENS), _case(1202, 128, 8, 4, 32, [900, 5, 300]),
             big]
    nbytes = max(qk.decode_attn_workspace_size(
        qk.make_params(torch.empty(c.B, c.Hq, c.D), c.block_size, c.Hkv, c.max_blocks,
                       c.num_blocks, max_seq_len=c.max_seq_len)) for c in cases)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for case in cases:
        t = case.device_tensors("cuda")
        out, lse = qk.decode_attn_paged(t["q"], t["k_pool"], t["v_pool"], t["block_table"],
                                        t["seq_lens"], max_seq_len=case.max_seq_len, workspace=ws)
        ref_out, ref_lse, _ = oracle_paged(case)
        assert_parity(out.cpu().numpy().reshape(-1, case.D), lse.cpu().numpy().reshape(-1),
                      ref_out, ref_lse, f"reuse/{case.name}")


@pytest.mark.parametrize("kind", ["paged", "multi", "sparse"])
def test_short_sequences_leave_the_workspace_untouched(kind):
    """With a workspace, short sequences run whole units: the call writes no
    partial state, so a zero workspace stays all zero, and the result equals
    the oracle.  Forced to split (unsplit_max_len = 0) the same call cuts
    every unit and writes partial states.  Both schedules give the oracle's
    result."""
    import torch
    lens = [300, 17, 512, 64]
    if kind == "sparse":
        rows = -(-512 // 64)
        lays = [[list(range(r + 1)) for r in range(rows)], [[r] for r in range(rows)]]
        case = wl.make_sparse("short_sparse", 43, B=4, Hq=32, Hkv=8, D=128, block_size=16,
                              seq_lens=lens, sparse_block=64, layouts=lays, num_rows=rows)
    else:
        case = _case(42, 128, 32, 8, 16, lens, q_len=2 if kind == "multi" else 1)
    t = case.device_tensors("cuda")
    q2 = t["q"][:, 0] if kind == "multi" else t["q"]
    params = qk.make_params(q2, case.block_size, case.Hkv, case.max_blocks, case.num_blocks,
                            max_seq_len=case.max_seq_len)
    from parity import oracle_sparse
    ref_out, ref_lse, _ = oracle_sparse(case) if kind == "sparse" else oracle_paged(case)

    def call(ws):
        kw = dict(max_seq_len=case.max_seq_len, workspace=ws)
        if kind == "sparse":
            return qk.decode_attn_paged_sparse(t["q"], t["k_pool"], t["v_pool"], t["block_table"],
                                               t["seq_lens"], t["row_ptr"], t["col_idx"],
                                               case.sparse_block, **kw)
        fn = qk.decode_attn_paged_multi if kind == "multi" else qk.decode_attn_paged
        return fn(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], **kw)

    for forced_split in (False, True):
        ws = torch.zeros(qk.decode_attn_workspace_size(params), dtype=torch.uint8, device="cuda")
        with qk.tuning(**({"unsplit_max_len": 0} if forced_split else {})):
            out, lse = call(ws)
        torch.cuda.synchronize()
        touched = bool(ws.any().item())
        assert touched == forced_split, (kind, forced_split)
        assert_parity(out.cpu().numpy().reshape(-1, case.D), lse.cpu().numpy().reshape(-1),
                      ref_out, ref_lse, f"{kind} split={forced_split}")


@pytest.mark.parametrize("softcap", [0.5, 30.0, 70.0, 200.0, 1e3, 1e6, 1e12])
def test_softcap_from_small_to_huge(softcap):
    """The softcap over its whole range, with outlier keys (K scaled by 8)
    so that scores reach both the saturated and the linear part of tanh:
    small caps saturate nearly every score; large caps leave the scores
    almost unchanged, which the kernels compute with the series branch of
    tanh; 1e12 equals no softcap."""
    case = _case(900 + int(math.log10(softcap) * 10), 128, 16, 4, 16, [1, 77, 1000, 3000],
                 softcap=softcap, outlier_rate=0.05)
    for mode in ("stream", "units"):
        _check_all_rows(case, mode)
