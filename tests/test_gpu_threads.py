"""Several host threads make their first decode calls at the same moment.

The library keeps per-device state that is filled on first use (the SM
count and each kernel's shared-memory opt-in).  This test runs in a fresh
process, so that state starts empty, and starts four threads that each make
their first call together, on a stream of their own, with a workspace of
their own.  The threads use different cache kinds and kernels: paged, int8
tiered and f16 tiered.  Every result must match the oracle.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

from parity import assert_parity, oracle_paged, oracle_tiered
from quantized_kv_decode_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = {
    "paged": lambda: wl.make_paged("threads_paged", 901, B=5, Hq=16, Hkv=4, D=128,
                                   block_size=16, seq_lens=[3000, 17, 1024, 777, 2048],
                                   num_blocks=600),
    "paged64": lambda: wl.make_paged("threads_paged64", 902, B=3, Hq=8, Hkv=2, D=64,
                                     block_size=32, seq_lens=[900, 1, 4000], num_blocks=200),
    "tiered": lambda: wl.make_tiered("threads_tiered", 903, B=3, Hq=8, Hkv=2, D=128,
                                     block_size=16, cold_len=1500, hot_len=100, hot_window=128,
                                     hot_start=1500),
    "tiered_f16": lambda: wl.make_tiered("threads_tiered_f16", 904, B=3, Hq=8, Hkv=2, D=128,
                                         block_size=16, cold_len=1200, hot_len=64,
                                         hot_window=64, hot_start=1200, cold_f16=True),
}

# Runs in a fresh process: builds nothing, loads the library, starts the
# threads behind a barrier, and writes each thread's outputs to an .npz.
_SCRIPT = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np
import torch
import quantized_kv_decode_paged_gb300 as qk
from test_gpu_threads import CASES, run_case
out_path = sys.argv[2]
torch.cuda.init()
cases = {name: make() for name, make in CASES.items()}
tensors = {name: c.device_tensors("cuda") for name, c in cases.items()}
torch.cuda.synchronize()
qk.load_library()
barrier = threading.Barrier(len(cases))
results, errors = {}, []
def work(name):
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            barrier.wait()
            out, lse = run_case(cases[name], tensors[name], s)
        s.synchronize()
        results[name + "_out"] = out.cpu().numpy()
        results[name + "_lse"] = lse.cpu().numpy()
    except Exception as e:
        errors.append(repr(e))
threads = [threading.Thread(target=work, args=(n,)) for n in cases]
for t in threads: t.start()
for t in threads: t.join()
if errors:
    print("ERRORS", errors); sys.exit(1)
np.savez(out_path, **results)
"""


def run_case(case, t, stream):
    import torch
    import quantized_kv_decode_paged_gb300 as qk
    ws = torch.zeros(1 << 23, dtype=torch.uint8, device="cuda")
    if hasattr(case, "cold_lens"):
        kw = dict(hot_window=case.hot_window, max_seq_len=case.max_seq_len,
                  cold_len=int(case.cold_lens[0]), hot_len=int(case.hot_lens[0]),
                  hot_start=int(case.hot_starts[0]), workspace=ws, stream=stream)
        if case.cold_f16:
            return qk.decode_attn_tiered_f16(t["q"], t["k_hot"], t["v_hot"], t["k_cold"],
                                             t["v_cold"], t["block_table"], **kw)
        return qk.decode_attn_tiered_int8(t["q"], t["k_hot"], t["v_hot"], t["k_cold"],
                                          t["v_cold"], t["k_scale"], t["v_scale"],
                                          t["block_table"], **kw)
    return qk.decode_attn_paged(t["q"], t["k_pool"], t["v_pool"], t["block_table"],
                                t["seq_lens"], max_seq_len=case.max_seq_len, workspace=ws,
                                stream=stream)


def test_first_calls_from_four_threads_at_once(cuda_lib, tmp_path):
    out = tmp_path / "threads.npz"
    r = subprocess.run([sys.executable, "-c", _SCRIPT, ROOT, str(out)], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    got = np.load(out)
    for name, make in CASES.items():
        case = make()
        ref_out, ref_lse, flags = (oracle_tiered(case) if hasattr(case, "cold_lens")
                                   else oracle_paged(case))
        assert flags == 0
        assert_parity(got[name + "_out"].reshape(-1, case.D), got[name + "_lse"].reshape(-1),
                      ref_out, ref_lse, name)
