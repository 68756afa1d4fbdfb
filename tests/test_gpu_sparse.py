"""GPU parity of the block-sparse paged decode (decode_attn_paged_sparse)
against the double-precision oracle, through the C ABI.

Layouts follow com.microsoft.SparseAttention: head h reads layout
h % num_layouts, the query reads CSR row qpos / sparse_block, and each listed
column selects one block of keys.  The cases cover head dimensions, group
sizes, layout counts, block sizes, unsorted and repeated columns, columns
past the query's row, windows, softcaps, explicit query positions, the
non-causal case, invalid CSR entries, empty selections, both schedules, both
operand packings, head groups sharing a unit, and batches split over
several launches.
"""
import numpy as np
import pytest

import oracle
import quantized_kv_decode_paged_gb300 as qk
from quantized_kv_decode_paged_gb300 import workloads as wl
from parity import assert_parity, oracle_sparse, run_paged, run_sparse

pytestmark = pytest.mark.gpu

MODES = ("stream", "units")


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    import torch
    torch.cuda.empty_cache()


def random_layouts(rng, NL, rows, density=0.35, extra_past_row=True, dup=True):
    lays = []
    for _ in range(NL):
        lay = []
        for r in range(rows):
            cols = [c for c in range(r + 1) if rng.random() < density]
            if extra_past_row and r + 1 < rows and rng.random() < 0.3:
                cols.append(int(rng.integers(r + 1, rows)))  # past the query's row
            if dup and cols and rng.random() < 0.3:
                cols.append(cols[0])                          # a repeated column
            rng.shuffle(cols)
            lay.append(cols)
        lays.append(lay)
    return lays


def _case(seed, D, Hq, Hkv, bs, lens, SB, NL, lays=None, **kw):
    rng = np.random.default_rng(seed)
    B = len(lens)
    L = max(max(lens), 1)
    rows = -(-L // SB)
    if lays is None:
        lays = random_layouts(rng, NL, rows)
    pages = sum((max(x, 0) + bs - 1) // bs for x in lens)
    return wl.make_sparse(f"sparse{seed}", seed, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                          seq_lens=lens, sparse_block=SB, layouts=lays, num_rows=rows,
                          num_blocks=pages + 3, **kw)


def _check(case, modes=MODES, flags=0):
    import torch
    ref_out, ref_lse, f = oracle_sparse(case)
    assert f == flags
    t = case.device_tensors("cuda")
    for mode in modes:
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, lse = run_sparse(case, t, mode, dev_status=st)
        assert int(st.item()) == flags, (mode, int(st.item()))
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse,
                      f"{case.name}/{mode}")


LENS = [1, 15, 16, 17, 64, 65, 200, 511, 777, 1500]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("NL", [1, 3, 4])
def test_head_dims_groups_and_layout_counts(D, G, NL):
    Hkv = 2
    case = _case(10 * D + G + 100 * NL, D, G * Hkv, Hkv, 16, LENS[:: 2 if D == 256 else 1],
                 SB=64, NL=NL)
    _check(case)


@pytest.mark.parametrize("SB", [16, 32, 64, 128, 256])
def test_sparse_block_sizes(SB):
    case = _case(300 + SB, 128, 8, 2, 16, [SB - 1, SB, 3 * SB + 5, 900, 1234], SB=SB, NL=4)
    _check(case)


@pytest.mark.parametrize("bs", [8, 32, 128])
def test_page_sizes(bs):
    case = _case(400 + bs, 128, 16, 4, bs, [bs + 3, 700, 1024, 2000], SB=64, NL=2)
    _check(case)


def test_every_causal_block_equals_plain_paged():
    rows = -(-1500 // 64)
    full = [[list(range(r + 1)) for r in range(rows)] for _ in range(3)]
    case = _case(500, 128, 12, 4, 16, LENS, SB=64, NL=3, lays=full)
    _check(case)
    dense = wl.make_paged("dense500", 500, B=case.B, Hq=12, Hkv=4, D=128, block_size=16,
                          seq_lens=case.seq_lens, num_blocks=case.num_blocks)
    t = case.device_tensors("cuda")
    for mode in MODES:
        a = run_sparse(case, t, mode)
        b = run_paged(dense, t, mode)
        assert_parity(a[0].reshape(-1, 128), a[1].reshape(-1), b[0].reshape(-1, 128).astype(
            np.float64), b[1].reshape(-1).astype(np.float64), f"full/{mode}")


@pytest.mark.parametrize("causal", [True, False])
def test_window_softcap_and_query_positions(causal):
    lens = [300, 1000, 2048, 77]
    case = _case(600 + causal, 128, 32, 8, 16, lens, SB=32, NL=4, sliding_window=300,
                 softcap=30.0, causal=causal, q_pos=[299, 640, 2047, 10])
    _check(case)


def test_invalid_rows_and_columns_flag_and_select_nothing():
    rng = np.random.default_rng(700)
    lens = [400, 250, 130]
    rows = -(-400 // 64)
    lays = random_layouts(rng, 2, rows)
    lays[0][rows - 1] = lays[0][rows - 1] + [-3, rows + 5]   # invalid columns
    case = _case(700, 128, 8, 2, 16, lens, SB=64, NL=2, lays=lays)
    _check(case, flags=oracle.FLAG_BAD_BLOCK)
    # a malformed row (end < start) in layout 1
    r = 250 // 64
    case.row_ptr = case.row_ptr.copy()
    case.row_ptr[1, r], case.row_ptr[1, r + 1] = case.row_ptr[1, r + 1] + 1, case.row_ptr[1, r]
    _check(case, flags=oracle.FLAG_BAD_BLOCK)


def test_empty_selections_give_zero_and_minus_infinity():
    rows = 8
    lays = [[[] for _ in range(rows)], [[r] for r in range(rows)]]
    case = _case(800, 128, 8, 2, 16, [500, 64, 300], SB=64, NL=2, lays=lays)
    _check(case)
    out, lse, _ = oracle_sparse(case)
    assert np.isneginf(lse.reshape(3, 8)[:, 0::2]).all()


def test_unpacked_variant_and_head_groups_sharing_a_unit():
    case = _case(900, 128, 8, 2, 16, LENS, SB=64, NL=4)
    with qk.tuning(packed_operands=0):
        _check(case)
    case = _case(901, 128, 32, 2, 16, LENS, SB=64, NL=5)  # G = 16: two head groups a kv head
    for fuse in (1, 0):
        with qk.tuning(fuse_head_groups=fuse):
            _check(case)


def test_long_sequences_many_bitmask_words():
    case = _case(1000, 128, 16, 4, 16, [20000, 9000, 17, 12345], SB=16, NL=4)
    _check(case)


def test_large_batch_is_split_over_launches():
    rng = np.random.default_rng(1100)
    lens = rng.integers(1, 3000, size=260).tolist()
    case = _case(1100, 64, 8, 2, 16, lens, SB=32, NL=3)
    _check(case)
