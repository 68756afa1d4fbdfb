"""Shared helpers for the GPU-vs-oracle parity tests (not collected)."""
import numpy as np

import oracle
import quantized_kv_decode_paged_gb300 as qk

# Tolerances from the benchmark spec of this path: per element
# |gpu - oracle| <= 1e-3 + 1e-3*|oracle| on the f32 outputs, |dLSE| <= 1e-4.
OUT_ATOL = 1e-3
OUT_RTOL = 1e-3
LSE_ATOL = 1e-4


def assert_parity(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    out_gpu = np.asarray(out_gpu, dtype=np.float64).reshape(out_ref.shape)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64).reshape(lse_ref.shape)
    assert np.isfinite(out_gpu).all(), f"{what}: non-finite output"
    err = np.abs(out_gpu - out_ref)
    bound = OUT_ATOL + OUT_RTOL * np.abs(out_ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} outputs off, max abs err {err.max():.3e}, "
                           f"worst at {np.unravel_index(np.argmax(err - bound), err.shape)}")
    ninf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), ninf), f"{what}: -inf LSE pattern differs"
    if (~ninf).any():
        lerr = np.abs(lse_gpu[~ninf] - lse_ref[~ninf])
        assert lerr.max() <= LSE_ATOL, f"{what}: max LSE err {lerr.max():.3e}"
    return float(err.max()) if err.size else 0.0


def oracle_paged(case, rows=None):
    T = case.q.shape[1] if case.q.ndim == 4 else 1  # query tokens per sequence
    seqs = None if rows is None else sorted({int(r) // (T * case.Hq) for r in rows})
    kp, vp = case.host_pools(seqs)
    return oracle.decode_paged(case.q, kp, vp, case.block_table, case.seq_lens, case.q_pos,
                               scale=case.scale, softcap=case.softcap,
                               sliding_window=case.sliding_window, causal=case.causal, rows=rows)


def run_paged(case, t, mode, split_tokens=256, dev_status=None):
    """Runs the CUDA path on device tensors ``t`` in one of the schedules:
    'stream' (auto workspace, keys split across CTAs whatever the lengths),
    'auto' (auto workspace, the library's default choice: short sequences
    run whole units), 'units' (no workspace) or 'split' (split_partial +
    split_merge).  Returns (out, lse) as numpy."""
    import torch
    kw = dict(scale=case.scale, softcap=case.softcap, sliding_window=case.sliding_window,
              causal=case.causal)
    if t["q"].dim() == 4:
        assert mode in ("stream", "auto", "units")
        with qk.tuning(**({"unsplit_max_len": 0} if mode == "stream" else {})):
            out, lse = qk.decode_attn_paged_multi(
                t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], t["q_pos"],
                max_seq_len=case.max_seq_len, workspace=None if mode == "units" else "auto",
                dev_status=dev_status, **kw)
    elif mode in ("stream", "auto", "units"):
        with qk.tuning(**({"unsplit_max_len": 0} if mode == "stream" else {})):
            out, lse = qk.decode_attn_paged(t["q"], t["k_pool"], t["v_pool"], t["block_table"],
                                            t["seq_lens"], t["q_pos"],
                                            max_seq_len=case.max_seq_len,
                                            workspace=None if mode == "units" else "auto",
                                            dev_status=dev_status, **kw)
    else:
        S = max(1, -(-max(case.max_seq_len, 1) // split_tokens))
        op, lp = qk.decode_attn_split_partial(t["q"], t["k_pool"], t["v_pool"], t["block_table"],
                                              t["seq_lens"], t["q_pos"], split_tokens=split_tokens,
                                              max_splits=S, dev_status=dev_status, **kw)
        out, lse = qk.decode_attn_split_merge(op, lp)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def oracle_tiered(case, rows=None):
    seqs = None if rows is None else sorted({int(r) // case.Hq for r in rows})
    h = case.host_arrays(seqs)
    if case.cold_f16:
        return oracle.decode_tiered_f16(case.q, h["k_hot"], h["v_hot"], h["k_cold"], h["v_cold"],
                                        case.block_table, case.cold_lens, case.hot_lens,
                                        case.hot_starts, hot_window=case.hot_window,
                                        q_pos=case.q_pos, scale=case.scale, softcap=case.softcap,
                                        sliding_window=case.sliding_window, causal=case.causal,
                                        rows=rows)
    return oracle.decode_tiered(case.q, h["k_hot"], h["v_hot"], h["k_cold"], h["v_cold"],
                                h["k_scale"], h["v_scale"], case.block_table, case.cold_lens,
                                case.hot_lens, case.hot_starts, hot_window=case.hot_window,
                                q_pos=case.q_pos, scale=case.scale, softcap=case.softcap,
                                sliding_window=case.sliding_window, causal=case.causal, rows=rows)


def run_tiered(case, t, mode, per_seq=None, dev_status=None):
    """CUDA tiered path; ``per_seq`` passes the tier lengths as device arrays
    (default: arrays unless every sequence has the same lengths)."""
    import torch
    if per_seq is None:
        per_seq = not case.uniform
    kw = dict(scale=case.scale, softcap=case.softcap, sliding_window=case.sliding_window,
              causal=case.causal, hot_window=case.hot_window, max_seq_len=case.max_seq_len)
    if per_seq:
        kw.update(cold_lens=t["cold_lens"], hot_lens=t["hot_lens"], hot_starts=t["hot_starts"])
    else:
        kw.update(cold_len=int(case.cold_lens[0]), hot_len=int(case.hot_lens[0]),
                  hot_start=int(case.hot_starts[0]))
    if case.cold_f16:
        out, lse = qk.decode_attn_tiered_f16(
            t["q"], t["k_hot"], t["v_hot"], t["k_cold"], t["v_cold"], t["block_table"],
            q_pos=t["q_pos"], workspace="auto" if mode == "stream" else None,
            dev_status=dev_status, **kw)
    else:
        out, lse = qk.decode_attn_tiered_int8(
            t["q"], t["k_hot"], t["v_hot"], t["k_cold"], t["v_cold"], t["k_scale"], t["v_scale"],
            t["block_table"], q_pos=t["q_pos"], workspace="auto" if mode == "stream" else None,
            dev_status=dev_status, **kw)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def oracle_sparse(case):
    kp, vp = case.host_pools()
    return oracle.decode_paged_sparse(case.q, kp, vp, case.block_table, case.seq_lens,
                                      case.row_ptr, case.col_idx, case.sparse_block, case.q_pos,
                                      scale=case.scale, softcap=case.softcap,
                                      sliding_window=case.sliding_window, causal=case.causal)


def run_sparse(case, t, mode, dev_status=None):
    """CUDA block-sparse path: 'stream' (auto workspace, always split),
    'auto' (auto workspace, the library's choice) or 'units'."""
    import torch
    with qk.tuning(**({"unsplit_max_len": 0} if mode == "stream" else {})):
        out, lse = qk.decode_attn_paged_sparse(
            t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], t["row_ptr"],
            t["col_idx"], case.sparse_block, t["q_pos"], max_seq_len=case.max_seq_len,
            scale=case.scale, softcap=case.softcap, sliding_window=case.sliding_window,
            causal=case.causal, workspace=None if mode == "units" else "auto",
            dev_status=dev_status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()
