"""GPU parity of the multi-token query decode (T query tokens per sequence,
each at its own position with its own causal / window bounds) against the
double-precision oracle, plus the partial head groups it relies on."""
import pytest

import quantized_kv_decode_paged_gb300 as qk
from quantized_kv_decode_paged_gb300 import workloads as wl
from parity import assert_parity, oracle_paged, run_paged

pytestmark = pytest.mark.gpu

MODES = ("stream", "auto", "units")


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    import torch
    torch.cuda.empty_cache()


def _case(seed, D, Hq, Hkv, bs, lens, T, **kw):
    B = len(lens)
    pages = sum((max(L, 0) + bs - 1) // bs for L in lens)
    return wl.make_paged(f"multi{seed}", seed, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                         seq_lens=lens, num_blocks=pages + 3, q_len=T, **kw)


def _check(case, modes=MODES):
    t = case.device_tensors("cuda")
    ref_out, ref_lse, _ = oracle_paged(case)
    for mode in modes:
        out, lse = run_paged(case, t, mode)
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse,
                      f"{case.name}/{mode}")


LENS = [1, 7, 16, 17, 64, 65, 200, 513, 1000]


@pytest.mark.parametrize("T", [2, 3, 4, 8])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_multi_token_group_sizes(T, G):
    case = _case(500 + 10 * T + G, 128, 2 * G, 2, 16, LENS, T)
    _check(case)


@pytest.mark.parametrize("T,G", [(2, 8), (4, 4), (8, 4), (3, 4)])
def test_multi_token_head_groups_one_unit_per_group(T, G):
    """fuse_head_groups=0: one unit per head group of T*G query rows (the default
    puts 2 or 4 head groups of a kv head in one unit)."""
    with qk.tuning(fuse_head_groups=0):
        case = _case(520 + 10 * T + G, 128, 2 * G, 2, 16, LENS, T)
        _check(case)


@pytest.mark.parametrize("D", [64, 256])
def test_multi_token_head_dims(D):
    case = _case(540 + D, D, 8, 2, 16, LENS[::2], 3)
    _check(case)


@pytest.mark.parametrize("window,softcap,causal", [(50, 0.0, True), (7, 20.0, True),
                                                   (0, 0.0, False), (100, 30.0, False)])
def test_multi_token_window_softcap_causal(window, softcap, causal):
    case = _case(560 + window, 128, 8, 2, 16, [5, 90, 300, 777], 4, sliding_window=window,
                 softcap=softcap, causal=causal)
    _check(case)


def test_multi_token_explicit_positions():
    # sequence 1's tokens sit well before the end of the cache; sequence 3's
    # sit past its two keys (they all see both)
    case = _case(580, 128, 8, 2, 16, [300, 300, 64, 2], 4, q_pos=[296, 100, 0, 5])
    _check(case)


def test_multi_token_default_positions_shorter_than_the_tokens():
    case = _case(590, 128, 8, 2, 16, [2, 40], 4)  # sequence 0: tokens 0, 1 at -2, -1
    _check(case)


@pytest.mark.parametrize("G", [12, 24])
def test_single_token_partial_head_groups(G):
    """G = 12 or 24 query heads per kv head: head groups of 8 with a partial
    last one (also the multi-token path's layout)."""
    case = _case(600 + G, 128, 2 * G, 2, 16, LENS[::2], 1)
    for mode in ("stream", "units", "split"):
        t = case.device_tensors("cuda")
        ref_out, ref_lse, _ = oracle_paged(case)
        out, lse = run_paged(case, t, mode)
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse, f"G{G}/{mode}")
