"""The entry point for callers that cannot allocate device memory.

decode_attn_paged_static_ws runs the split-KV paged decode with its scratch
in a buffer compiled into the library.  Callers that need it: a plugin whose
host framework owns every allocation, a process held to a fixed
device-memory budget, or a loop that cannot afford cudaMalloc's implicit
synchronisation.

This test calls it through the C ABI twice in a row.  Both calls are checked
against decode_attn_paged with a caller-provided workspace, and against the
oracle, within the parity tolerance of the other GPU tests.  A second case
has more sequences than one launch takes, so one call makes several launches
that reuse the buffer's ticket counters.

The file is collected last, and the test works both on its own in a fresh
process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest

import quantized_kv_decode_paged_gb300 as qk
from quantized_kv_decode_paged_gb300 import workloads as wl
from parity import assert_parity, oracle_paged

pytestmark = pytest.mark.gpu

OUT_ATOL = 1e-3
OUT_RTOL = 1e-3
LSE_ATOL = 1e-4


def _lens(rng, B):
    # mostly short rows plus some long ones, so that units are cut between
    # CTAs and the scratch is used
    lens = rng.integers(1, 400, size=B)
    lens[rng.random(B) < 0.05] = 3000
    return lens.tolist()


CASES = [
    ("six_sequences", dict(B=6, Hq=16, Hkv=4, D=128, block_size=16,
                           seq_lens=[3000, 17, 1024, 4096, 511, 2222], num_blocks=1200)),
    ("many_sequences", dict(B=300, Hq=8, Hkv=2, D=128, block_size=16,
                            seq_lens=_lens(np.random.default_rng(5), 300), num_blocks=12000)),
]


@pytest.mark.parametrize("name,shape", CASES, ids=[c[0] for c in CASES])
def test_static_scratch_entry_point_matches_workspace_entry_point(cuda_lib, name, shape):
    import torch

    lib = qk.load_library()
    case = wl.make_paged("noalloc_" + name, 77, **shape)
    t = case.device_tensors("cuda")
    params = qk.make_params(t["q"], case.block_size, case.Hkv, case.max_blocks, case.num_blocks,
                            max_seq_len=case.max_seq_len)
    assert qk.decode_attn_workspace_size(params) <= 8 << 20
    ws = torch.zeros(qk.decode_attn_workspace_size(params), dtype=torch.uint8, device="cuda")
    ref_out, ref_lse = qk.decode_attn_paged(t["q"], t["k_pool"], t["v_pool"], t["block_table"],
                                            t["seq_lens"], max_seq_len=case.max_seq_len,
                                            workspace=ws)
    torch.cuda.synchronize()
    ref_out = ref_out.cpu().numpy().astype(np.float64)
    ref_lse = ref_lse.cpu().numpy().astype(np.float64)
    orc_out, orc_lse, flags = oracle_paged(case)
    assert flags == 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full((case.B, case.Hq, case.D), float("nan"), device="cuda")
        lse = torch.full((case.B, case.Hq), float("nan"), device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = lib.decode_attn_paged_static_ws(
            ctypes.byref(params), t["q"].data_ptr(), t["k_pool"].data_ptr(),
            t["v_pool"].data_ptr(), t["block_table"].data_ptr(), t["seq_lens"].data_ptr(), None,
            out.data_ptr(), lse.data_ptr(), status.data_ptr(), stream)
        assert st == qk.DA_OK, qk.decode_attn_status_string(st)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.cpu().numpy().astype(np.float64)
        got_lse = lse.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        assert (np.abs(got - ref_out) <= OUT_ATOL + OUT_RTOL * np.abs(ref_out)).all(), call
        assert np.abs(got_lse - ref_lse).max() <= LSE_ATOL, call
        assert_parity(got.reshape(-1, case.D), got_lse.reshape(-1), orc_out, orc_lse,
                      f"{name} call {call} vs oracle")
