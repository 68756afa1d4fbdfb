"""Algorithmic byte counts of one decode step (the roofline numerator).

Counts what the method must move: the visible K/V rows (int8 words plus
their scales, or f16 rows, for the cold tier), the block-table entries of the pages those
rows sit in, Q, out, lse and the length arrays.  Masked pages, unused pool
pages and split-KV partials are not counted.
"""
from __future__ import annotations

from .workloads import PagedCase, TieredCase


def visible_range(L: int, qpos: int, causal: bool, window: int):
    """[lo, hi) of absolute key positions a query at qpos sees among keys
    0..L-1 (causal and sliding-window masks)."""
    hi = min(L, qpos + 1) if causal else L
    lo = qpos - window + 1 if (window > 0 and qpos >= window) else 0
    return max(lo, 0), max(hi, 0)


def algorithmic_bytes(case) -> dict:
    """Bytes the decode step must read and write: visible K/V rows (int8 words
    and their scales for the cold tier), the block-table entries of the
    visible pages, Q, out, lse and the length arrays."""
    if isinstance(case, PagedCase) and case.sparse:
        return _sparse_bytes(case)
    if isinstance(case, PagedCase):
        T = case.q.shape[1] if case.q.ndim == 4 else 1  # query tokens per sequence
        kv = 0
        bt = 0
        for b in range(case.B):
            L = int(case.seq_lens[b])
            qp = int(case.q_pos[b]) if case.q_pos is not None else L - T
            # union of the tokens' ranges: token 0's lower bound, token T-1's upper
            lo, _ = visible_range(L, qp, case.causal, case.sliding_window)
            _, hi = visible_range(L, qp + T - 1, case.causal, case.sliding_window)
            n = max(0, hi - lo)
            kv += n * case.Hkv * case.D * 2 * 2
            if n:
                bs = case.block_size
                bt += ((hi - 1) // bs - lo // bs + 1) * 4
        io = T * (case.B * case.Hq * case.D * 4 * 2 + case.B * case.Hq * 4) + case.B * 4
        return dict(kv=kv, table=bt, io=io, total=kv + bt + io)
    kv = 0
    bt = 0
    for b in range(case.B):
        cl, hl, hs = int(case.cold_lens[b]), int(case.hot_lens[b]), int(case.hot_starts[b])
        qp = int(case.q_pos[b]) if case.q_pos is not None else (hs + hl - 1 if hl > 0 else cl - 1)
        lo, hi = visible_range(cl, qp, case.causal, case.sliding_window)
        nc = max(0, hi - lo)
        # int8 cold: D bytes of K and of V plus two f16 scales; f16 cold: 2D + 2D
        kv += nc * case.Hkv * (case.D * 2 * 2 if case.cold_f16 else case.D * 2 + 2 * 2)
        if nc:
            bt += ((hi - 1) // case.block_size - lo // case.block_size + 1) * 4
        for j in range(hl):
            pos = hs + j
            if (not case.causal or pos <= qp) and not (
                    case.sliding_window > 0 and qp >= case.sliding_window
                    and pos < qp - case.sliding_window + 1):
                kv += case.Hkv * case.D * 2 * 2
    io = case.B * case.Hq * case.D * 4 * 2 + case.B * case.Hq * 4 + case.B * 4 * 3
    return dict(kv=kv, table=bt, io=io, total=kv + bt + io)


def sparse_selection(case, b):
    """Per kv head of sequence b of a block-sparse case: the visible keys of
    the blocks any of its query heads' layouts selects, as a list of
    [a, z) ranges, and the CSR entries the selection reads."""
    G = case.Hq // case.Hkv
    NL = case.row_ptr.shape[0]
    SB = case.sparse_block
    L = int(case.seq_lens[b])
    qp = int(case.q_pos[b]) if case.q_pos is not None else L - 1
    lo, hi = visible_range(L, qp, case.causal, case.sliding_window)
    row = qp // SB
    sel, csr = {}, 0
    for l in range(min(NL, case.Hq)):
        s0, s1 = int(case.row_ptr[l, row]), int(case.row_ptr[l, row + 1])
        sel[l] = set(int(c) for c in case.col_idx[l, s0:s1])
        csr += 2 + (s1 - s0)
    ranges = []
    for k in range(case.Hkv):
        blocks = set().union(*(sel[(k * G + g) % NL] for g in range(G)))
        rk = []
        for c in sorted(blocks):
            a, z = max(c * SB, lo), min((c + 1) * SB, hi)
            if z > a:
                rk.append((a, z))
        ranges.append(rk)
    return ranges, csr


def _sparse_bytes(case) -> dict:
    """Block-sparse paged step: per (sequence, kv head), the visible keys of
    the blocks that any of its query heads' layouts selects (each read once
    for all of them), the block-table entries of their pages, and the CSR
    row pointers and columns the selection reads."""
    kv = bt = csr = 0
    for b in range(case.B):
        ranges, nc = sparse_selection(case, b)
        csr += nc * 4
        pages = set()
        for rk in ranges:
            for a, z in rk:
                kv += (z - a) * case.D * 2 * 2
                pages.update(range(a // case.block_size, (z - 1) // case.block_size + 1))
        bt += len(pages) * 4
    io = case.B * case.Hq * case.D * 4 * 2 + case.B * case.Hq * 4 + case.B * 4
    return dict(kv=kv, table=bt, io=io + csr, total=kv + bt + io + csr)
