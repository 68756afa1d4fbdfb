#!/usr/bin/env python3
"""Benchmark: decode-attention KV-cache bandwidth and time per decode step.

One step = one decode step of the whole batch: a single call of the paged
(or tiered) decode attention through the library's public API, i.e. one
launch of the decode kernel (stream-K split-KV with the in-kernel merge).
Inputs are resident in HBM; the L2 is flushed (a write of 2x its size)
before every timed step, outside the step's CUDA-event interval.

value = algorithmic bytes per step (visible K/V rows, the block-table
entries of their pages, Q, out, lse, lengths) / device time per step.

Prints ONE JSON line on rank 0.  `--impl reference` times the CPU oracle on
a bounded sample of the same workload instead (the reference arm).
Under torchrun (N > 1) every rank runs an independent replica (the path
does not shard across GPUs) and rank 0 reports the sum of bytes over the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn KV-cache HBM GB/s (% of GB300 peak); µs per decode step"
SPEC_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = "longctx"
# The five serving shapes, and the paged one with block-sparse layouts: every
# run reports each of them in "configs".
CONFIG_WORKLOADS = ("tiny", "paged", "tiered", "window", "longctx", "paged_sparse")


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    pat = os.path.join(ROOT, "quantized_kv_decode_paged_gb300", "csrc", "*")
    for f in sorted(glob.glob(pat)):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch of the decode kernel on this workload, from the
    committed ncu record profiles/decode_attn_kernel_<workload>.json, when
    that record was taken from the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"decode_attn_kernel_{workload}.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    v = rec.get("dram_bytes_per_launch")
    return float(v) if v is not None else None


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU, read in-process
    through NVML (libnvidia-ml, read-only queries): one sample when the
    timed region starts, one every 2 ms during it and one when it ends.
    prepare() opens NVML and takes a first sample of every query before the
    warm-up, so that first-call costs of the driver's management interface
    (seconds on a freshly booted machine) stay out of the timed region.
    Nothing is changed on the GPU."""

    # clock-event reason bits of NVML
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index):
        self.cuda_index = cuda_index
        self.samples = []
        self.nvml = None
        self.dev = None
        self.error = None
        self._stop = threading.Event()

    def _open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        dev = ctypes.c_void_p()
        bus = None
        try:
            import torch
            pr = torch.cuda.get_device_properties(self.cuda_index)
            bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        except Exception:
            bus = None
        ok = bus is not None and lib.nvmlDeviceGetHandleByPciBusId_v2(
            bus.encode(), ctypes.byref(dev)) == 0
        if not ok:
            idx = self.cuda_index
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            if vis and all(x.strip().isdigit() for x in vis.split(",")):
                idx = int(vis.split(",")[self.cuda_index])
            if lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(dev)) != 0:
                raise RuntimeError("no NVML handle for the device")
        self.nvml, self.dev = lib, dev
        mx = ctypes.c_uint()
        self.sm_max = (float(mx.value)
                       if lib.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) == 0 else None)
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self._reasons_fn = fn or lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        import ctypes
        lib, dev = self.nvml, self.dev
        mhz, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if lib.nvmlDeviceGetClockInfo(dev, 1, ctypes.byref(mhz)) != 0:
            return
        p = float(mw.value) / 1e3 if lib.nvmlDeviceGetPowerUsage(dev, ctypes.byref(mw)) == 0 else None
        r = int(rs.value) if self._reasons_fn(dev, ctypes.byref(rs)) == 0 else 0
        self.samples.append((float(mhz.value), p, r))

    def _loop(self):
        while not self._stop.wait(0.002):
            self.sample()

    def prepare(self):
        if self.nvml is not None or self.error is not None:
            return self
        try:
            self._open()
            self.sample()
            self.samples.clear()  # the first sample only warms the queries
        except Exception as exc:  # clocks are reported as unavailable, never fatal
            self.error = f"{type(exc).__name__}: {exc}"
            self.nvml = None
        return self

    def __enter__(self):
        self.prepare()
        if self.nvml is None:
            return self
        try:
            self.sample()
            self.t = threading.Thread(target=self._loop, daemon=True)
            self.t.start()
        except Exception as exc:
            self.error = f"{type(exc).__name__}: {exc}"
            self.nvml = None
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self._stop.set()
            self.t.join(timeout=2)
            self.sample()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "nvml", "error": self.error or "no samples"}
        sm = sorted(x[0] for x in self.samples)
        bits = 0
        for _, _, r in self.samples:
            bits |= r
        power = [x[1] for x in self.samples if x[1] is not None]
        return {"sm_mhz": sm[len(sm) // 2], "sm_min_mhz": sm[0], "sm_max_mhz": self.sm_max,
                "reasons": sorted(n for b, n in self.REASONS.items() if bits & b),
                "power_w_max": round(max(power), 1) if power else None,
                "samples": len(sm), "source": "nvml, every 2 ms in the timed region"}


# ------------------------------------------------------------------ workloads
def load_case(name):
    from quantized_kv_decode_paged_gb300 import workloads as wl
    return wl.workload(name)


def describe(case):
    from quantized_kv_decode_paged_gb300.workloads import PagedCase
    if isinstance(case, PagedCase):
        lens = case.seq_lens
        T = case.q.shape[1] if case.q.ndim == 4 else 1
        d = {"workload": case.name, "kind": "paged f16", "B": case.B, "q_len": T, "Hq": case.Hq,
             "Hkv": case.Hkv, "D": case.D, "block_size": case.block_size,
             "num_blocks": case.num_blocks, "seq_len_min": int(lens.min()),
             "seq_len_max": int(lens.max()), "seq_len_mean": float(lens.mean()),
             "sliding_window": case.sliding_window, "softcap": case.softcap}
        if case.sparse:
            d.update(kind="paged f16, block-sparse layouts", sparse_block=case.sparse_block,
                     num_layouts=int(case.row_ptr.shape[0]))
        return d
    kind = "tiered f16 cold + f16 hot ring" if case.cold_f16 else "tiered int8 cold + f16 hot ring"
    return {"workload": case.name, "kind": kind, "B": case.B,
            "Hq": case.Hq, "Hkv": case.Hkv, "D": case.D, "block_size": case.block_size,
            "cold_len": int(case.cold_lens[0]), "hot_len": int(case.hot_lens[0]),
            "hot_window": case.hot_window, "hot_start": int(case.hot_starts[0])}


def _packed_f32(shapes, device="cuda", pin=False):
    """f32 tensors of the given shapes as views of one contiguous buffer
    (each view 16-byte aligned); returns the views and, last, the buffer."""
    import torch
    offs, n = [], 0
    for s in shapes:
        offs.append(n)
        k = 1
        for d in s:
            k *= int(d)
        n += (k + 3) // 4 * 4
    buf = torch.empty(max(n, 1), dtype=torch.float32, device=device)
    if pin:
        buf = buf.pin_memory()
    views = []
    for s, o in zip(shapes, offs):
        k = 1
        for d in s:
            k *= int(d)
        views.append(buf[o:o + k].view(*s))
    views.append(buf)
    return views


def _packed_bytes(arrays, device="cuda", pin=False):
    """Byte buffer holding the given arrays back to back (16-byte aligned);
    returns views of each with its dtype and shape and, last, the buffer."""
    import torch
    offs, n = [], 0
    for a in arrays:
        offs.append(n)
        n += (a.nbytes + 15) // 16 * 16
    buf = torch.empty(max(n, 1), dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = []
    for a, o in zip(arrays, offs):
        dt = {"float32": torch.float32, "int32": torch.int32}[str(a.dtype)]
        views.append(buf[o:o + a.nbytes].view(dt).view(*a.shape))
    views.append(buf)
    return views


def make_step(case, t):
    """Returns step() running one decode step on the current stream."""
    import quantized_kv_decode_paged_gb300 as qk
    from quantized_kv_decode_paged_gb300.workloads import PagedCase
    import torch
    # out and lse share one device buffer, so the end-to-end step reads the
    # result back with one copy
    multi = isinstance(case, PagedCase) and case.q.ndim == 4  # several query tokens
    o_shape = tuple(case.q.shape) if multi else (case.B, case.Hq, case.D)
    l_shape = tuple(case.q.shape[:3]) if multi else (case.B, case.Hq)
    out, lse, _res = _packed_f32([o_shape, l_shape])
    if isinstance(case, PagedCase):
        params = qk.make_params(t["q"][:, 0] if multi else t["q"], case.block_size, case.Hkv,
                                case.max_blocks, case.num_blocks, scale=case.scale,
                                softcap=case.softcap, sliding_window=case.sliding_window,
                                causal=case.causal, max_seq_len=case.max_seq_len)
        nbytes = qk.decode_attn_workspace_size(params)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        fn = qk.decode_attn_paged_multi if multi else qk.decode_attn_paged

        def step(q=None, block_table=None, seq_lens=None):
            if case.sparse:
                return qk.decode_attn_paged_sparse(
                    t["q"] if q is None else q, t["k_pool"], t["v_pool"],
                    t["block_table"] if block_table is None else block_table,
                    t["seq_lens"] if seq_lens is None else seq_lens, t["row_ptr"], t["col_idx"],
                    case.sparse_block, t["q_pos"], max_seq_len=case.max_seq_len,
                    scale=case.scale, softcap=case.softcap, sliding_window=case.sliding_window,
                    causal=case.causal, out=out, lse=lse, workspace=ws)
            return fn(
                t["q"] if q is None else q, t["k_pool"], t["v_pool"],
                t["block_table"] if block_table is None else block_table,
                t["seq_lens"] if seq_lens is None else seq_lens, t["q_pos"],
                scale=case.scale, softcap=case.softcap, sliding_window=case.sliding_window,
                causal=case.causal, max_seq_len=case.max_seq_len, out=out, lse=lse,
                workspace=ws)
    else:
        params = qk.make_params(t["q"], case.block_size, case.Hkv, case.max_blocks,
                                case.num_blocks, scale=case.scale, softcap=case.softcap,
                                sliding_window=case.sliding_window, causal=case.causal,
                                max_seq_len=case.max_seq_len)
        nbytes = qk.decode_attn_workspace_size(params)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")

        tier = dict(hot_window=case.hot_window, cold_len=int(case.cold_lens[0]),
                    hot_len=int(case.hot_lens[0]), hot_start=int(case.hot_starts[0]),
                    q_pos=t["q_pos"], scale=case.scale, softcap=case.softcap,
                    sliding_window=case.sliding_window, causal=case.causal,
                    max_seq_len=case.max_seq_len, out=out, lse=lse, workspace=ws)

        def step(q=None, block_table=None, seq_lens=None):
            q = t["q"] if q is None else q
            block_table = t["block_table"] if block_table is None else block_table
            if case.cold_f16:
                return qk.decode_attn_tiered_f16(q, t["k_hot"], t["v_hot"], t["k_cold"],
                                                 t["v_cold"], block_table, **tier)
            return qk.decode_attn_tiered_int8(q, t["k_hot"], t["v_hot"], t["k_cold"],
                                              t["v_cold"], t["k_scale"], t["v_scale"],
                                              block_table, **tier)
    step.result = _res
    return step, out, lse


# ------------------------------------------------------------ CPU / oracle arm
def oracle_sample(case, target_s, max_units=None):
    """Times the oracle on whole (sequence, kv head) units of the workload,
    adding units until about target_s seconds of CPU work.  Returns
    (GB/s of algorithmic bytes, seconds, description, threads)."""
    import numpy as np
    import oracle
    from quantized_kv_decode_paged_gb300.accounting import visible_range
    from quantized_kv_decode_paged_gb300.workloads import PagedCase
    G = case.Hq // case.Hkv
    units = [(b, kv) for b in range(case.B) for kv in range(case.Hkv)]
    rng = np.random.default_rng(0)
    order = rng.permutation(len(units))
    if max_units is not None:
        order = order[:max_units]
    is_paged = isinstance(case, PagedCase)
    T = case.q.shape[1] if case.q.ndim == 4 else 1  # query tokens per sequence

    def unit_bytes(b, kv):
        if is_paged and case.sparse:
            from quantized_kv_decode_paged_gb300.accounting import sparse_selection
            ranges, _ = sparse_selection(case, b)
            return sum(z - a for a, z in ranges[kv]) * case.D * 2 * 2 + G * case.D * 8
        if is_paged:
            L = int(case.seq_lens[b])
            lo, _ = visible_range(L, L - T, case.causal, case.sliding_window)
            _, hi = visible_range(L, L - 1, case.causal, case.sliding_window)
            return max(0, hi - lo) * case.D * 2 * 2 + T * G * case.D * 8
        cl, hl = int(case.cold_lens[b]), int(case.hot_lens[b])
        cold_row = case.D * 4 if case.cold_f16 else case.D * 2 + 4
        return cl * cold_row + hl * case.D * 4 + G * case.D * 8

    def run(sel):
        rows = np.array([(b * T + t) * case.Hq + kv * G + g for (b, kv) in sel
                         for t in range(T) for g in range(G)])
        seqs = sorted({b for b, _ in sel})
        if is_paged and case.sparse:
            kp, vp = case.host_pools(seqs)
            t0 = time.perf_counter()
            oracle.decode_paged_sparse(case.q, kp, vp, case.block_table, case.seq_lens,
                                       case.row_ptr, case.col_idx, case.sparse_block, case.q_pos,
                                       scale=case.scale, softcap=case.softcap,
                                       sliding_window=case.sliding_window, causal=case.causal,
                                       rows=rows)
        elif is_paged:
            kp, vp = case.host_pools(seqs)
            t0 = time.perf_counter()
            oracle.decode_paged(case.q, kp, vp, case.block_table, case.seq_lens, case.q_pos,
                                scale=case.scale, softcap=case.softcap,
                                sliding_window=case.sliding_window, causal=case.causal, rows=rows)
        elif case.cold_f16:
            h = case.host_arrays(seqs)
            t0 = time.perf_counter()
            oracle.decode_tiered_f16(case.q, h["k_hot"], h["v_hot"], h["k_cold"], h["v_cold"],
                                     case.block_table, case.cold_lens, case.hot_lens,
                                     case.hot_starts, hot_window=case.hot_window,
                                     q_pos=case.q_pos, scale=case.scale, softcap=case.softcap,
                                     sliding_window=case.sliding_window, causal=case.causal,
                                     rows=rows)
        else:
            h = case.host_arrays(seqs)
            t0 = time.perf_counter()
            oracle.decode_tiered(case.q, h["k_hot"], h["v_hot"], h["k_cold"], h["v_cold"],
                                 h["k_scale"], h["v_scale"], case.block_table, case.cold_lens,
                                 case.hot_lens, case.hot_starts, hot_window=case.hot_window,
                                 q_pos=case.q_pos, scale=case.scale, softcap=case.softcap,
                                 sliding_window=case.sliding_window, causal=case.causal,
                                 rows=rows)
        return time.perf_counter() - t0

    # calibrate on a few units, then size the sample; when the whole step is
    # quicker than the target, repeat it
    n = min(len(order), 4)
    sel = [units[i] for i in order[:n]]
    dt = run(sel)
    reps = 1
    if dt < target_s and n < len(order):
        per_unit = max(dt / n, 1e-6)
        n = int(min(len(order), max(n, target_s / per_unit)))
        sel = [units[i] for i in order[:n]]
        dt = run(sel)
    if dt < target_s and n == len(order):
        reps = max(1, int(target_s / max(dt, 1e-6)))
        dt = sum(run(sel) for _ in range(reps))
    nbytes = sum(unit_bytes(b, kv) for b, kv in sel) * reps
    desc = (f"{n} of {len(units)} (sequence, kv head) units of workload '{case.name}' "
            f"({n * G} query-head rows) x {reps} repetition(s), keys in logical order, "
            f"double precision")
    return nbytes / dt / 1e9, dt, desc, oracle.num_threads()


def reference_arm(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    case = load_case(args.workload)
    target = args.ref_step_seconds
    vals = []
    desc, threads = "", 1
    for i in range(args.warmup + args.steps):
        gbs, dt, desc, threads = oracle_sample(case, target)
        if i >= args.warmup:
            vals.append((gbs, dt))
    gbs = sum(v for v, _ in vals) / len(vals)
    ms = sum(d for _, d in vals) / len(vals) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {**describe(case), "sample": "bounded oracle sample per step"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ across ranks
def aggregate_ranks(dev_ms, e2e_ms, bytes_per_step, world, device):
    """One replica per rank (weak scaling): the job's time is the slowest
    rank's, its bytes the sum over ranks.  Returns (device ms, end-to-end
    ms, bytes per step) for the whole job; with one rank, the inputs."""
    if world <= 1:
        return float(dev_ms), float(e2e_ms), float(bytes_per_step)
    import torch
    import torch.distributed as dist
    stats = torch.tensor([dev_ms, e2e_ms, float(bytes_per_step)], dtype=torch.float64,
                         device=device)
    mx = stats.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    tot = stats.clone()
    dist.all_reduce(tot, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(mx[1]), float(tot[2])


def job_gbs(total_bytes_per_step, steps, ms):
    """Whole-job GB/s: every rank's bytes of `steps` steps over `ms`."""
    return total_bytes_per_step * steps / (ms * 1e-3) / 1e9


# ----------------------------------------------------------------- GPU arm
def time_device_steps(step, flush, steps, warmup, stream, barrier, clk=None):
    """`warmup` untimed steps, then `steps` steps each preceded by an L2
    flush outside its CUDA events.  Returns (per-step ms, wall seconds of
    the timed loop)."""
    import contextlib
    import torch
    for _ in range(warmup):
        flush.zero_()
        step()
    barrier()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with (clk if clk is not None else contextlib.nullcontext()):
        barrier()
        w0 = time.perf_counter()
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        barrier()
        wall = time.perf_counter() - w0
    return [a.elapsed_time(b) for a, b in zip(starts, ends)], wall


def copy_reference_us(nbytes, flush, stream, barrier, steps=50):
    """Time of one device-to-device copy that moves nbytes of DRAM traffic
    (nbytes/2 read, nbytes/2 written), timed like a decode step (L2 flushed
    before each copy, CUDA events): the rate this GPU reaches on a transfer
    of the same size, launch included."""
    import torch
    n = max(16, nbytes // 2 // 16 * 16)
    src = torch.ones(n, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    tms, _ = time_device_steps(lambda: dst.copy_(src), flush, steps, 3, stream, barrier)
    del src, dst
    torch.cuda.empty_cache()
    return sum(tms) / len(tms) * 1e3


def config_entry(case, times_ms, peak, copy_us=None):
    """One workload's line in "configs": time per step and bandwidth, and
    the time of a plain copy of the same byte count."""
    from quantized_kv_decode_paged_gb300.accounting import algorithmic_bytes
    nbytes = algorithmic_bytes(case)["total"]
    mean_ms = sum(times_ms) / len(times_ms)
    gbs = nbytes / (mean_ms * 1e-3) / 1e9
    e = {"us_per_step": round(mean_ms * 1e3, 2),
         "us_median": round(sorted(times_ms)[len(times_ms) // 2] * 1e3, 2),
         "gb_per_s": round(gbs, 1), "frac_of_measured": round(gbs / peak, 4),
         "frac_of_spec_8000": round(gbs / SPEC_HBM_GBS, 4),
         "bytes_per_step": int(nbytes), "steps": len(times_ms),
         "shape": describe(case)}
    if copy_us is not None:
        e["copy_same_bytes_us"] = round(copy_us, 2)
        e["frac_of_copy_same_bytes"] = round(copy_us / (mean_ms * 1e3), 4)
    return e


def gpu_arm(args, rank, world):
    import torch
    import torch.distributed as dist
    import quantized_kv_decode_paged_gb300 as qk
    from quantized_kv_decode_paged_gb300.accounting import algorithmic_bytes

    local = _env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    qk.build()
    qk.load_library()
    case = load_case(args.workload)
    t = case.device_tensors("cuda")
    step, out, lse = make_step(case, t)
    acc = algorithmic_bytes(case)
    bytes_per_step = acc["total"]
    launches_per_step = -(-case.B // 256)

    # L2 flush before every timed step: write a buffer of 4x the L2, then
    # read a second one of 2x the L2, so the step starts with none of its
    # inputs in L2 and no dirty lines left to write back during the step.
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush_w = torch.empty(max(4 * l2, 512 << 20), dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device="cuda")

    class _Flush:
        @staticmethod
        def zero_():
            flush_w.zero_()
            flush_r.sum()

    flush = _Flush()
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    clk = ClockSampler(local).prepare()
    times_ms, wall = time_device_steps(step, flush, args.steps, args.warmup, stream, barrier, clk)
    dev_ms = sum(times_ms)
    clocks = clk.summary()

    # e2e: host buffers in, host result out, every step.  The step's inputs
    # (q, block table, sequence lengths) sit back to back in one pinned host
    # buffer and go over in one copy; out and lse come back in one copy.
    import numpy as np
    from quantized_kv_decode_paged_gb300.workloads import PagedCase
    paged = isinstance(case, PagedCase)
    lens_np = (case.seq_lens if paged else case.cold_lens + case.hot_lens).astype("int32")
    ins = [np.ascontiguousarray(case.q, dtype=np.float32),
           np.ascontiguousarray(case.block_table, dtype=np.int32)] + ([lens_np] if paged else [])
    *views_h, in_h = _packed_bytes(ins, device="cpu", pin=True)
    for v, a in zip(views_h, ins):
        v.copy_(torch.from_numpy(a))
    *views, in_d = _packed_bytes(ins, device="cuda")
    q_d, bt_d = views[0], views[1]
    sl_d = views[2] if paged else None
    res_d = step.result  # out and lse, one buffer
    res_h = torch.empty(res_d.shape, dtype=res_d.dtype).pin_memory()

    def e2e_step():
        in_d.copy_(in_h, non_blocking=True)
        if paged:
            step(q=q_d, block_table=bt_d, seq_lens=sl_d)
        else:
            step(q=q_d, block_table=bt_d)
        res_h.copy_(res_d, non_blocking=True)

    h2d = int(in_h.numel())
    d2h = int(res_h.numel()) * 4
    e2e_steps = max(10, min(args.steps, 500))
    for _ in range(3):
        flush.zero_()
        e2e_step()
    barrier()
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        flush.zero_()
        e_s[i].record(stream)
        e2e_step()
        e_e[i].record(stream)
    barrier()
    e2e_ms = sum(s.elapsed_time(e) for s, e in zip(e_s, e_e)) / e2e_steps

    dev_ms_max, e2e_ms_max, total_bytes = aggregate_ranks(dev_ms, e2e_ms, bytes_per_step, world,
                                                          "cuda")
    peak, peak_src = measured_hbm_peak()

    # every serving shape, one GPU: same flush, fewer steps
    configs = None
    if world == 1 and not args.no_configs:
        configs = {}
        n_cfg = max(10, min(args.steps, args.config_steps))
        for name in CONFIG_WORKLOADS:
            if name == case.name:
                cp = copy_reference_us(bytes_per_step, flush, stream, barrier)
                configs[name] = config_entry(case, times_ms, peak, cp)
                continue
            c = load_case(name)
            tt = c.device_tensors("cuda")
            st, _, _ = make_step(c, tt)
            tms, _ = time_device_steps(st, flush, n_cfg, 3, stream, barrier)
            del tt, st
            torch.cuda.empty_cache()
            cp = copy_reference_us(algorithmic_bytes(c)["total"], flush, stream, barrier)
            configs[name] = config_entry(c, tms, peak, cp)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            import oracle
            oracle.build()
            gbs, dt, desc, threads = oracle_sample(case, args.cpu_seconds)
            cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                   "sample": desc, "seconds": round(dt, 2)}
        except Exception as exc:  # the baseline never blocks the GPU line
            cpu = {"value": None, "unit": "GB/s", "cores": None, "kind": "oracle",
                   "sample": f"failed: {exc}"}

    if rank == 0:
        ms_per_step = dev_ms_max / args.steps
        value = job_gbs(total_bytes, args.steps, dev_ms_max)
        per_launch_s = dev_ms / args.steps / launches_per_step * 1e-3
        achieved = bytes_per_step / launches_per_step / per_launch_s / 1e9
        traffic = profiled_traffic(case.name)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "us_per_step": round(ms_per_step * 1e3, 2),
            "frac_of_spec_8000": round(value / world / SPEC_HBM_GBS, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16 K/V, f32 softmax and accumulate", "data": "synthetic",
            "config": {**describe(case),
                       "l2": "flushed before every timed step, outside the step's events: "
                             "write of 4x L2 then read of 2x L2 (cold L2, no dirty lines)",
                       "bytes_per_step": bytes_per_step, "kv_bytes_per_step": acc["kv"],
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "launches_per_step": launches_per_step},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2),
                         "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_src == "measured" else "fallback",
                         "traffic": traffic},
            "cpu_baseline": cpu,
            "configs": configs,
            "e2e": {"value": round(job_gbs(total_bytes, 1, e2e_ms_max), 2), "unit": "GB/s",
                    "us_per_step": round(e2e_ms_max * 1e3, 2),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "kernel_source_hash": kernel_source_hash(),
            "clocks": clocks,
            "wall_s_timed_region": round(wall, 3),
            "step_us_min": round(min(times_ms) * 1e3, 2),
            "step_us_median": round(sorted(times_ms)[len(times_ms) // 2] * 1e3, 2),
        }
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=["tiny", "paged", "tiered", "window", "longctx", "paged_compact",
                             "tiered_f16", "paged_spec2", "paged_spec4", "paged_sparse",
                             "paged_sparse_compact", "longctx_compact", "window_compact"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work of the oracle baseline sample")
    ap.add_argument("--ref-step-seconds", type=float, default=4.0,
                    help="CPU work per step of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload entries of the five serving shapes")
    ap.add_argument("--config-steps", type=int, default=200,
                    help="timed steps of each entry in configs")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    if world != args.gpus:
        world = max(world, 1)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        if args.impl == "reference":
            return reference_arm(args, rank, world)
        return gpu_arm(args, rank, world)
    finally:
        if world > 1 and args.impl == "ours":
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
