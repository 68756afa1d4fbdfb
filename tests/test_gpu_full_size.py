"""Every output row of every full-size serving workload against the oracle.

The workloads are the serving shapes of the benchmark, at full size:
paged, int8 tiered, window with softcap and outliers, long-context mix,
f16 tiered, and the paged shape with 2 or 4 query tokens per sequence.
Each is run through every schedule the library has for it:
- stream: stream-K with the in-kernel merge, the launch configuration the
  benchmark times for every workload but tiny;
- auto: the library's default choice with a workspace; for tiny (256 keys)
  that is whole units per CTA, the configuration the benchmark times there;
- units: whole units per CTA, no workspace;
- split: the explicit split-partial / merge pair, one-token paged only.
The block-sparse workload (the paged shape with four layouts) runs stream
and units.

Every row is compared with the oracle at the parity tolerance.  The oracle
runs once per workload.  With PARITY_REPORT set to a path, the largest
absolute, relative and LSE errors of each (workload, schedule) are written
there as JSON.
"""
import json
import os

import numpy as np
import pytest

from parity import (assert_parity, oracle_paged, oracle_sparse, oracle_tiered, run_paged,
                    run_sparse, run_tiered)
from quantized_kv_decode_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

PAGED = {"tiny": ("stream", "auto", "units", "split"), "paged": ("stream", "units", "split"),
         "window": ("stream", "units", "split"), "longctx": ("stream", "units", "split"),
         "paged_spec2": ("stream", "units"), "paged_spec4": ("stream", "units")}
TIERED = {"tiered": ("stream", "units"), "tiered_f16": ("stream", "units")}
SPARSE = {"paged_sparse": ("stream", "units")}
REPORT = {}


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    import torch
    torch.cuda.empty_cache()


def _errors(out, lse, ref_out, ref_lse):
    out = np.asarray(out, np.float64).reshape(ref_out.shape)
    lse = np.asarray(lse, np.float64).reshape(ref_lse.shape)
    err = np.abs(out - ref_out)
    rel = err / np.maximum(np.abs(ref_out), 1e-6)
    fin = np.isfinite(ref_lse)
    lerr = np.abs(lse[fin] - ref_lse[fin])
    return {"rows": int(ref_lse.size), "max_abs_err": float(err.max()),
            "max_rel_err": float(rel.max()),
            "max_lse_err": float(lerr.max()) if lerr.size else 0.0}


def _record(name, mode, errs):
    REPORT[f"{name}/{mode}"] = errs
    path = os.environ.get("PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump(REPORT, f, indent=1, sort_keys=True)


def _split_tokens(case):
    # about 8 splits of the longest row, a multiple of the block size
    L = max(case.max_seq_len, 1)
    st = max(case.block_size, -(-L // 8))
    return -(-st // case.block_size) * case.block_size


@pytest.mark.parametrize("name", list(PAGED))
def test_paged_workload_every_row_every_schedule(name):
    import torch
    case = wl.workload(name)
    ref_out, ref_lse, flags = oracle_paged(case)
    assert flags == 0
    t = case.device_tensors("cuda")
    for mode in PAGED[name]:
        out, lse = run_paged(case, t, mode, split_tokens=_split_tokens(case))
        _record(name, mode, _errors(out, lse, ref_out, ref_lse))
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse,
                      f"{name}/{mode}")
    del t
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", list(TIERED))
@pytest.mark.parametrize("per_seq", [False, True])
def test_tiered_workload_every_row_every_schedule(name, per_seq):
    import torch
    case = wl.workload(name)
    ref_out, ref_lse, flags = oracle_tiered(case)
    assert flags == 0
    t = case.device_tensors("cuda")
    for mode in TIERED[name]:
        out, lse = run_tiered(case, t, mode, per_seq=per_seq)
        tag = mode + ("/device-lengths" if per_seq else "")
        _record(name, tag, _errors(out, lse, ref_out, ref_lse))
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse,
                      f"{name}/{tag}")
    del t
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", list(SPARSE))
def test_sparse_workload_every_row_every_schedule(name):
    import torch
    case = wl.workload(name)
    ref_out, ref_lse, flags = oracle_sparse(case)
    assert flags == 0
    t = case.device_tensors("cuda")
    for mode in SPARSE[name]:
        out, lse = run_sparse(case, t, mode)
        _record(name, mode, _errors(out, lse, ref_out, ref_lse))
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse,
                      f"{name}/{mode}")
    del t
    torch.cuda.empty_cache()
