"""GPU parity of the block-sparse paged decode (decode_attn_paged_sparse)
against the double-precision oracle, through the C ABI.

Layouts follow com.microsoft.SparseAttention: head h reads layout
h % num_layouts, the query reads CSR row qpos / sparse_block, and each listed
column selects one block of keys.  The cases cover head dimensions, group
sizes, layout counts, block sizes, unsorted and repeated columns, columns
past the query's row, windows, softcaps, explicit query positions, the
non-causal case, invalid CSR entries, empty selections, every schedule, both
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

MODES = ("stream", "auto", "units")


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


@pytest.mark.parametrize("i", range(12))
def test_sparse_random_shapes(i):
    """Every knob drawn from a fixed seed: head dim, kv heads, group size,
    page size, sparse block size, layout count and density, lengths (0 and
    1 included), window, softcap, causal, explicit query positions."""
    rng = np.random.default_rng(9000 + i)
    D = int(rng.choice([64, 128, 256]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 8, 16]))
    bs = int(rng.choice([8, 16, 32, 64]))
    SB = int(rng.choice([16, 32, 64, 128]))
    NL = int(rng.integers(1, 9))
    B = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.choice([0, 1, 2, SB - 1, SB, SB + 1, 97, 300, 1200], size=B)]
    lens[0] = max(lens[0], 1)
    L = max(lens)
    rows = -(-L // SB)
    lays = random_layouts(rng, NL, rows, density=float(rng.choice([0.1, 0.4, 0.9])))
    q_pos = None
    if rng.integers(0, 3) == 0:
        q_pos = [int(rng.integers(0, max(x, 1))) for x in lens]
    pages = sum((x + bs - 1) // bs for x in lens)
    case = wl.make_sparse(f"sfz{i}", 9100 + i, B=B, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs,
                          seq_lens=lens, sparse_block=SB, layouts=lays, num_rows=rows,
                          num_blocks=pages + 2, sliding_window=int(rng.choice([0, 0, 5, 100])),
                          softcap=float(rng.choice([0.0, 0.0, 20.0])),
                          causal=bool(rng.integers(0, 2)), q_pos=q_pos)
    _check(case)


def test_sparse_decode_step_in_a_cuda_graph():
    """One block-sparse step captured into a CUDA graph (the call allocates
    nothing and never synchronises) and replayed over new queries and a new
    layout written into the same buffers."""
    import torch
    rng = np.random.default_rng(9500)
    rows = -(-2200 // 64)
    # room for any layout of these rows: every causal block, one block past
    # the row and one repeat per row
    nnz = rows * (rows + 1) // 2 + 2 * rows
    case = _case(9500, 128, 16, 4, 16, [1000, 17, 640, 2200, 1], SB=64, NL=3, max_nnz=nnz)
    t = case.device_tensors("cuda")
    out = torch.empty((case.B, case.Hq, case.D), dtype=torch.float32, device="cuda")
    lse = torch.empty((case.B, case.Hq), dtype=torch.float32, device="cuda")
    params = qk.make_params(t["q"], case.block_size, case.Hkv, case.max_blocks, case.num_blocks,
                            max_seq_len=case.max_seq_len)
    ws = torch.zeros(qk.decode_attn_workspace_size(params), dtype=torch.uint8, device="cuda")

    def step():
        qk.decode_attn_paged_sparse(t["q"], t["k_pool"], t["v_pool"], t["block_table"],
                                    t["seq_lens"], t["row_ptr"], t["col_idx"], case.sparse_block,
                                    max_seq_len=case.max_seq_len, out=out, lse=lse, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for rep in range(3):
        q_new = rng.standard_normal(case.q.shape).astype(np.float32)
        t["q"].copy_(torch.from_numpy(q_new))
        case.q = q_new
        # a new layout with arrays of the captured shapes
        rp, ci_full = wl.csr_layouts(random_layouts(rng, 3, rows, density=0.3), rows, nnz)
        case.row_ptr, case.col_idx = rp, ci_full
        t["row_ptr"].copy_(torch.from_numpy(rp))
        t["col_idx"].copy_(torch.from_numpy(ci_full))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse, _ = oracle_sparse(case)
        assert_parity(out.cpu().numpy().reshape(-1, case.D), lse.cpu().numpy().reshape(-1),
                      ref_out, ref_lse, f"sparse graph replay {rep}")
