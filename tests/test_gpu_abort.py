"""Bounded waits on the GPU: a wait inside the decode kernel that runs out
ends the kernel in abort mode with DA_DEV_TIMEOUT in dev_status, leaves no
copy in flight and the workspace tickets at zero, and the next call on the
same context and workspace is correct again.  The wait is made to run out
with the library's test hook (decode_attn_testing_skip_first_arm: CTA 0
never arms its first stage, a barrier that nothing completes) and a short
wait limit (the tuning's wait_limit_ms); no fault, trap or endless loop is
involved."""
import contextlib
import pytest

import quantized_kv_decode_paged_gb300 as qk
from quantized_kv_decode_paged_gb300 import workloads as wl
from parity import assert_parity, oracle_paged, oracle_tiered, run_paged, run_tiered

pytestmark = pytest.mark.gpu


@contextlib.contextmanager
def _waits_run_out():
    lib = qk.load_library()
    with qk.tuning(wait_limit_ms=50):
        assert lib.decode_attn_testing_skip_first_arm(1) == qk.DA_OK
        try:
            yield
        finally:
            assert lib.decode_attn_testing_skip_first_arm(0) == qk.DA_OK


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    import torch
    torch.cuda.empty_cache()


def _status():
    import torch
    return torch.zeros(1, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("mode", ["stream", "units", "split"])
def test_paged_wait_runs_out_then_recovers(mode):
    import torch
    case = wl.make_paged("abort_paged", 700, B=3, Hq=8, Hkv=2, D=128, block_size=16,
                         seq_lens=[300, 1000, 77], num_blocks=100)
    t = case.device_tensors("cuda")
    st = _status()
    with _waits_run_out():
        run_paged(case, t, mode, dev_status=st)
        torch.cuda.synchronize()
    assert int(st.item()) & qk.DEV_TIMEOUT
    st = _status()
    out, lse = run_paged(case, t, mode, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_out, ref_lse, _ = oracle_paged(case)
    assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse, f"after abort/{mode}")


def test_tiered_wait_runs_out_then_recovers():
    import torch
    case = wl.make_tiered("abort_tiered", 701, B=2, Hq=8, Hkv=2, D=128, block_size=16,
                          cold_len=300, hot_len=40, hot_window=64, hot_start=300)
    t = case.device_tensors("cuda")
    st = _status()
    with _waits_run_out():
        run_tiered(case, t, "stream", dev_status=st)
        torch.cuda.synchronize()
    assert int(st.item()) & qk.DEV_TIMEOUT
    st = _status()
    out, lse = run_tiered(case, t, "stream", dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_out, ref_lse, _ = oracle_tiered(case)
    assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse, "tiered after abort")
