"""Random shapes against the oracle, and the decode inside a CUDA graph.

The fuzz cases draw, from a fixed seed, every knob the paged, multi-token
and int8 tiered entries take (batch, heads and group size, head dim, block
size, lengths including 0 and 1, window, softcap, causal, explicit query
positions, query tokens) and compare all rows with the double-precision
oracle.  The graph test captures one decode step (with its workspace) into
a CUDA graph, replays it over new queries written into the same buffers,
and checks every replay against the oracle: the entries launch work only,
allocate nothing and never synchronise, so they can be captured.
"""
import numpy as np
import pytest

import quantized_kv_decode_paged_gb300 as qk
from quantized_kv_decode_paged_gb300 import workloads as wl
from parity import assert_parity, oracle_paged, oracle_tiered, run_paged, run_tiered

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    import torch
    torch.cuda.empty_cache()


def _paged_fuzz_case(rng, i):
    D = int(rng.choice([64, 128, 256]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))
    bs = int(rng.choice([8, 16, 32, 64]))
    B = int(rng.integers(1, 7))
    T = int(rng.choice([1, 1, 1, 2, 3]))
    lens = [int(x) for x in rng.choice([0, 1, 2, bs - 1, bs, bs + 1, 97, 300, 1000], size=B)]
    window = int(rng.choice([0, 0, 1, 5, 64, 400]))
    softcap = float(rng.choice([0.0, 0.0, 10.0, 50.0]))
    causal = bool(rng.integers(0, 2))
    q_pos = None
    if rng.integers(0, 3) == 0:
        q_pos = [int(rng.integers(0, max(L, 1) + 3)) for L in lens]
    return wl.make_paged(f"fz{i}", 900 + i, B=B, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs,
                         seq_lens=lens, num_blocks=sum((L + bs - 1) // bs for L in lens) + 2,
                         sliding_window=window, softcap=softcap, causal=causal, q_pos=q_pos,
                         q_len=T)


@pytest.mark.parametrize("i", range(24))
def test_paged_random_shapes(i):
    rng = np.random.default_rng(7000 + i)
    case = _paged_fuzz_case(rng, i)
    t = case.device_tensors("cuda")
    ref_out, ref_lse, _ = oracle_paged(case)
    modes = ("stream", "auto", "units") + (() if case.q.ndim == 4 else ("split",))
    for mode in modes:
        out, lse = run_paged(case, t, mode, split_tokens=case.block_size * 4)
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse,
                      f"{case.name}/{mode} D{case.D} Hq{case.Hq} Hkv{case.Hkv} bs{case.block_size}")


@pytest.mark.parametrize("i", range(12))
def test_tiered_random_shapes(i):
    rng = np.random.default_rng(8000 + i)
    D = int(rng.choice([128, 256]))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    B = int(rng.integers(1, 5))
    bs = int(rng.choice([8, 16, 32]))
    W = int(rng.choice([0, 16, 48, 100]))
    cold = [int(x) for x in rng.integers(0, 300, size=B)]
    cap = W if W > 0 else 64
    hot = [int(x) for x in rng.integers(0, cap + 1, size=B)]
    case = wl.make_tiered(f"tfz{i}", 950 + i, B=B, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs,
                          cold_len=cold, hot_len=hot, hot_window=W, hot_start=cold,
                          sliding_window=int(rng.choice([0, 0, 37, 200])),
                          softcap=float(rng.choice([0.0, 20.0])),
                          cold_f16=bool(rng.integers(0, 2)))
    t = case.device_tensors("cuda")
    ref_out, ref_lse, _ = oracle_tiered(case)
    for mode in ("stream", "units"):
        out, lse = run_tiered(case, t, mode, per_seq=True)
        assert_parity(out.reshape(-1, case.D), lse.reshape(-1), ref_out, ref_lse,
                      f"{case.name}/{mode}")


def test_decode_step_in_a_cuda_graph():
    import torch
    case = wl.make_paged("graph", 990, B=5, Hq=16, Hkv=4, D=128, block_size=16,
                         seq_lens=[1000, 17, 640, 2200, 1], num_blocks=260)
    t = case.device_tensors("cuda")
    out = torch.empty((case.B, case.Hq, case.D), dtype=torch.float32, device="cuda")
    lse = torch.empty((case.B, case.Hq), dtype=torch.float32, device="cuda")
    params = qk.make_params(t["q"], case.block_size, case.Hkv, case.max_blocks, case.num_blocks,
                            max_seq_len=case.max_seq_len)
    ws = torch.zeros(qk.decode_attn_workspace_size(params), dtype=torch.uint8, device="cuda")

    def step():
        qk.decode_attn_paged(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                             max_seq_len=case.max_seq_len, out=out, lse=lse, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm up outside the capture (library load, tensor maps)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    rng = np.random.default_rng(991)
    for rep in range(3):
        q_new = rng.standard_normal(case.q.shape).astype(np.float32)
        t["q"].copy_(torch.from_numpy(q_new))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        case.q = q_new
        ref_out, ref_lse, _ = oracle_paged(case)
        assert_parity(out.cpu().numpy().reshape(-1, case.D), lse.cpu().numpy().reshape(-1),
                      ref_out, ref_lse, f"graph replay {rep}")
