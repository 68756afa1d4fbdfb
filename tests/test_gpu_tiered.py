"""GPU parity of the int8-cold / f16-hot tiered decode path against the
double-precision oracle."""
import numpy as np
import pytest

import oracle
import quantized_kv_decode_paged_gb300 as qk
from quantized_kv_decode_paged_gb300 import workloads as wl
from parity import assert_parity, oracle_tiered, run_tiered

pytestmark = pytest.mark.gpu

MODES = ("stream", "units")


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    import torch
    torch.cuda.empty_cache()


def _check(case, modes=MODES, per_seq=None):
    t = case.device_tensors("cuda")
    ref_out, ref_lse, flags = oracle_tiered(case)
    for mode in modes:
        out, lse = run_tiered(case, t, mode, per_seq=per_seq)
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse,
                      f"{case.name}/{mode}")
    return flags


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("cold_len,hot_len,hot_window,hot_start", [
    (0, 5, 8, 0),          # hot only
    (37, 0, 16, 37),       # cold only
    (100, 64, 64, 100),    # ring phase 100 % 64 = 36: the visible slots wrap
    (128, 64, 64, 128),    # aligned ring
    (64, 10, 0, 64),       # no ring: slot = j
    (300, 100, 128, 300),  # ring not a multiple of the tile, partial fill
    (5, 200, 200, 5),
])
def test_tier_shapes(D, cold_len, hot_len, hot_window, hot_start):
    case = wl.make_tiered(f"t{D}_{cold_len}_{hot_len}", 20 + D, B=3, Hq=8, Hkv=2, D=D,
                          block_size=16, cold_len=cold_len, hot_len=hot_len,
                          hot_window=hot_window, hot_start=hot_start)
    _check(case)


@pytest.mark.parametrize("bs", [8, 32, 128])
def test_tier_block_sizes(bs):
    case = wl.make_tiered(f"bs{bs}", 30 + bs, B=2, Hq=16, Hkv=4, D=128, block_size=bs,
                          cold_len=3 * bs + 7, hot_len=33, hot_window=48, hot_start=3 * bs + 7)
    _check(case)


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 8, 16])
def test_tier_group_sizes(G):
    case = wl.make_tiered(f"g{G}", 40 + G, B=2, Hq=2 * G, Hkv=2, D=128, block_size=16,
                          cold_len=200, hot_len=70, hot_window=96, hot_start=200)
    _check(case)


@pytest.mark.parametrize("fuse", ["1", "0"])
@pytest.mark.parametrize("D,G,Hkv", [(128, 16, 2), (128, 16, 4), (128, 32, 2), (256, 16, 2)])
def test_tier_head_groups_sharing_a_unit(D, G, Hkv, fuse):
    """Two or four head groups per kv head in one unit (fuse_head_groups=1, the
    default) or one unit each (fuse_head_groups=0)."""
    with qk.tuning(fuse_head_groups=int(fuse)):
        case = wl.make_tiered(f"hg{D}_{G}_{Hkv}", 70 + G + D + Hkv, B=2, Hq=G * Hkv, Hkv=Hkv, D=D,
                              block_size=16, cold_len=200, hot_len=70, hot_window=96, hot_start=200)
        _check(case)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("G", [1, 3, 4])
def test_tier_unpacked_variant_for_small_groups(D, G):
    """packed_operands=0 in the tuning: the two-operand variant for groups of at most four heads."""
    with qk.tuning(packed_operands=0):
        case = wl.make_tiered(f"u{D}_{G}", 60 + G + D, B=2, Hq=2 * G, Hkv=2, D=D, block_size=16,
                              cold_len=200, hot_len=70, hot_window=96, hot_start=200)
        _check(case)


def test_tier_window_softcap_and_query_position():
    for causal in (True, False):
        case = wl.make_tiered("wsq", 50 + causal, B=3, Hq=8, Hkv=2, D=128, block_size=16,
                              cold_len=400, hot_len=90, hot_window=128, hot_start=400,
                              sliding_window=150, softcap=20.0, causal=causal,
                              q_pos=[480, 430, 100])
        _check(case)


def test_tier_per_sequence_lengths():
    case = wl.make_tiered("perseq", 60, B=4, Hq=8, Hkv=2, D=128, block_size=16,
                          cold_len=[0, 100, 257, 31], hot_len=[5, 0, 64, 40],
                          hot_window=64, hot_start=[0, 100, 257, 31])
    _check(case, per_seq=True)


def test_tier_bad_block_is_masked_and_flagged():
    import torch
    case = wl.make_tiered("bad", 70, B=2, Hq=8, Hkv=2, D=128, block_size=16, cold_len=100,
                          hot_len=20, hot_window=32, hot_start=100)
    bt = case.block_table.copy()
    bt[1, 3] = 10_000
    case.block_table = bt
    ref_out, ref_lse, flags = oracle_tiered(case)
    assert flags & oracle.FLAG_BAD_BLOCK
    t = case.device_tensors("cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_tiered(case, t, "stream", dev_status=st)
    assert int(st.item()) & qk.DEV_BAD_BLOCK
    assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse, "tiered-bad")


def test_tier_large_batch_is_split_over_launches():
    """240 sequences of the int8 tiered cache: more than one launch keeps
    the pipeline depth of a small batch (the per-sequence plan shares
    shared memory with the stages); every row against the oracle."""
    rng = np.random.default_rng(1240)
    B = 240
    cold = rng.integers(0, 120, size=B).tolist()
    hot = rng.integers(0, 40, size=B).tolist()
    case = wl.make_tiered("bigB", 1240, B=B, Hq=32, Hkv=8, D=128, block_size=16,
                          cold_len=cold, hot_len=hot, hot_window=48, hot_start=cold)
    _check(case, per_seq=True)
