"""GPU parity of the f16-cold / f16-hot tiered decode path (the f16 tiered
layout of doppler attention.js executeAttentionTiered) against the
double-precision oracle."""
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


def _tiered(name, seed, **kw):
    return wl.make_tiered(name, seed, cold_f16=True, **kw)


def _check(case, modes=MODES, per_seq=None, t=None):
    t = case.device_tensors("cuda") if t is None else t
    ref_out, ref_lse, flags = oracle_tiered(case)
    for mode in modes:
        out, lse = run_tiered(case, t, mode, per_seq=per_seq)
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse,
                      f"{case.name}/{mode}")
    return flags


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("cold_len,hot_len,hot_window,hot_start", [
    (0, 5, 8, 0),          # hot only
    (37, 0, 16, 37),       # cold only
    (100, 64, 64, 100),    # ring phase 100 % 64 = 36: the visible slots wrap
    (64, 10, 0, 64),       # no ring: slot = j
    (300, 100, 128, 300),  # ring not a multiple of the tile, partial fill
])
def test_f16_tier_shapes(D, cold_len, hot_len, hot_window, hot_start):
    case = _tiered(f"f{D}_{cold_len}_{hot_len}", 120 + D, B=3, Hq=8, Hkv=2, D=D, block_size=16,
                   cold_len=cold_len, hot_len=hot_len, hot_window=hot_window,
                   hot_start=hot_start)
    _check(case)


@pytest.mark.parametrize("bs", [8, 32, 128])
def test_f16_tier_block_sizes(bs):
    case = _tiered(f"fbs{bs}", 130 + bs, B=2, Hq=16, Hkv=4, D=128, block_size=bs,
                   cold_len=3 * bs + 7, hot_len=33, hot_window=48, hot_start=3 * bs + 7)
    _check(case)


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 8, 16])
def test_f16_tier_group_sizes(G):
    case = _tiered(f"fg{G}", 140 + G, B=2, Hq=2 * G, Hkv=2, D=128, block_size=16,
                   cold_len=200, hot_len=70, hot_window=96, hot_start=200)
    _check(case)


@pytest.mark.parametrize("fuse", ["1", "0"])
@pytest.mark.parametrize("G", [16, 32])
def test_f16_tier_head_groups_sharing_a_unit(G, fuse):
    with qk.tuning(fuse_head_groups=int(fuse)):
        case = _tiered(f"fhg{G}", 155 + G, B=2, Hq=2 * G, Hkv=2, D=128, block_size=16,
                       cold_len=200, hot_len=70, hot_window=96, hot_start=200)
        _check(case)


@pytest.mark.parametrize("G", [1, 4])
def test_f16_tier_unpacked_variant(G):
    with qk.tuning(packed_operands=0):
        case = _tiered(f"fu{G}", 150 + G, B=2, Hq=2 * G, Hkv=2, D=128, block_size=16,
                       cold_len=200, hot_len=70, hot_window=96, hot_start=200)
        _check(case)


def test_f16_tier_window_softcap_and_query_position():
    for causal in (True, False):
        case = _tiered("fwsq", 160 + causal, B=3, Hq=8, Hkv=2, D=128, block_size=16,
                       cold_len=400, hot_len=90, hot_window=128, hot_start=400,
                       sliding_window=150, softcap=20.0, causal=causal, q_pos=[480, 430, 100])
        _check(case)


def test_f16_tier_per_sequence_lengths():
    case = _tiered("fperseq", 170, B=4, Hq=8, Hkv=2, D=128, block_size=16,
                   cold_len=[0, 100, 257, 31], hot_len=[5, 0, 64, 40],
                   hot_window=64, hot_start=[0, 100, 257, 31])
    _check(case, per_seq=True)


def test_f16_tier_nonfinite_rows_past_the_cold_length_do_not_leak():
    """f16 cold pages can hold anything past cold_len (a page being filled);
    NaN and inf there must not reach the output."""
    import torch
    case = _tiered("fnan", 180, B=2, Hq=8, Hkv=2, D=128, block_size=16, cold_len=[45, 70],
                   hot_len=[9, 12], hot_window=32, hot_start=[45, 70])
    t = case.device_tensors("cuda")
    for b in range(case.B):
        cl = int(case.cold_lens[b])
        page = int(case.block_table[b, cl // case.block_size])
        t["k_cold"][page, cl % case.block_size:] = float("nan")
        t["v_cold"][page, cl % case.block_size:] = float("inf")
    torch.cuda.synchronize()
    _check(case, per_seq=True, t=t)


def test_f16_tier_bad_block_is_masked_and_flagged():
    import torch
    case = _tiered("fbad", 190, B=2, Hq=8, Hkv=2, D=128, block_size=16, cold_len=100,
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
    assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse, "tiered-f16-bad")
