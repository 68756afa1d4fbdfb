"""Pins of the block-sparse oracle to things other than itself.

The rule (com.microsoft.SparseAttention sparse-attention.wgsl.jinja, the
attention pass): head h reads layout h % NUM_LAYOUT; the query at position
qp reads CSR row qp / SPARSE_BLOCK; each listed column c selects the keys
c*SPARSE_BLOCK .. (c+1)*SPARSE_BLOCK - 1; the mask is boolean (a repeated
column adds nothing); causality bounds the keys at qp.

The pins:
- a layout that lists every block up to the query's row equals the plain
  paged decode (pinned on its own elsewhere), bit for bit;
- any selection equals the log-sum-exp merge of one plain paged decode per
  selected block, each restricted to that block by an explicit query
  position and a window of one block (the merge of softmax states over
  disjoint key sets, the combine_partials identity of the same page);
- the last k blocks of a row equal a sliding window of the plain decode;
- torch float64 scaled_dot_product_attention with the boolean block mask;
- invariances: column order and repeated columns change nothing, and head
  h gives the same row as a one-layout call with layout h % NUM_LAYOUT;
- conventions: an invalid column id or a malformed row raises flag 1 and
  selects nothing; an empty selection gives out = 0 and lse = -inf.
"""
import math

import numpy as np
import pytest

import oracle

FLAG_BAD_BLOCK = 1


def _paged(rng, B, L, H, D, bs, extra=2):
    """Random f16 K/V for B sequences of L keys in a shuffled page pool."""
    npg = (L + bs - 1) // bs
    NB = B * npg + extra
    ids = rng.permutation(NB)
    table = ids[:B * npg].reshape(B, npg).astype(np.int32)
    kp = rng.standard_normal((NB, bs, H, D)).astype(np.float16)
    vp = rng.standard_normal((NB, bs, H, D)).astype(np.float16)
    return kp, vp, table


def _csr(rows_of_layouts, num_rows):
    """CSR arrays from, per layout, a list (per row) of column lists."""
    NL = len(rows_of_layouts)
    nnz = max(1, max(sum(len(r) for r in lay) for lay in rows_of_layouts))
    rp = np.zeros((NL, num_rows + 1), np.int32)
    ci = np.full((NL, nnz), -7, np.int32)  # unused entries hold junk
    for l, lay in enumerate(rows_of_layouts):
        pos = 0
        for r in range(num_rows):
            cols = lay[r] if r < len(lay) else []
            rp[l, r] = pos
            ci[l, pos:pos + len(cols)] = cols
            pos += len(cols)
        rp[l, num_rows] = pos
    return rp, ci


def _strided_layouts(NL, num_rows, local, stride):
    """Row r of layout l: the last `local` blocks up to r, plus every block
    c <= r with (c + l) % stride == 0 (the local + vertical-stride pattern)."""
    lays = []
    for l in range(NL):
        rows = []
        for r in range(num_rows):
            cols = set(range(max(0, r - local + 1), r + 1))
            cols |= {c for c in range(r + 1) if (c + l) % stride == 0}
            rows.append(sorted(cols))
        lays.append(rows)
    return lays


def _merge(parts):
    """Log-sum-exp merge of (out [D], lse) states over disjoint key sets."""
    lses = np.array([l for _, l in parts])
    if np.all(np.isneginf(lses)):
        return np.zeros_like(parts[0][0]), -np.inf
    M = lses.max()
    w = np.exp(lses - M)
    out = sum(wi * o for wi, (o, _) in zip(w, parts)) / w.sum()
    return out, M + math.log(w.sum())


def test_every_causal_block_listed_equals_plain_paged_bitwise():
    rng = np.random.default_rng(21)
    B, Hq, H, D, bs, SB = 3, 8, 2, 16, 8, 16
    lens = np.array([77, 16, 130], np.int32)
    kp, vp, table = _paged(rng, B, int(lens.max()), H, D, bs)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    rows = (int(lens.max()) + SB - 1) // SB
    full = [[list(range(r + 1)) for r in range(rows)] for _ in range(3)]
    rp, ci = _csr(full, rows)
    a = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp, ci, SB, softcap=9.0)
    b = oracle.decode_paged(q, kp, vp, table, lens, softcap=9.0)
    assert a[2] == 0 and b[2] == 0
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("NL", [1, 2, 3, 4])
@pytest.mark.parametrize("causal", [True, False])
def test_selection_equals_merge_of_per_block_plain_decodes(NL, causal):
    rng = np.random.default_rng(30 + NL + 10 * causal)
    B, Hq, H, D, bs, SB = 3, 8, 2, 16, 8, 16
    lens = np.array([200, 45, 160], np.int32)
    L = int(lens.max())
    kp, vp, table = _paged(rng, B, L, H, D, bs)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    rows = (L + SB - 1) // SB
    lays = []
    for l in range(NL):  # random rows, unsorted, with repeats and blocks past the row
        lay = []
        for r in range(rows):
            k = int(rng.integers(0, rows + 1))
            lay.append([int(c) for c in rng.integers(0, rows, size=k)])
        lays.append(lay)
    rp, ci = _csr(lays, rows)
    qpos = np.array([150, 44, 100], np.int32)
    out, lse, flags = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp, ci, SB, q_pos=qpos,
                                                 causal=causal, softcap=5.0)
    assert flags == 0
    for b in range(B):
        Lb = int(lens[b])
        for h in range(Hq):
            cols = set(lays[h % NL][qpos[b] // SB])
            parts = []
            for c in sorted(cols):
                # block c alone: query at its last key, window of one block
                end = min((c + 1) * SB, Lb) - 1
                if end < c * SB:
                    continue
                if causal:
                    end = min(end, int(qpos[b]))
                    if end < c * SB:
                        continue
                o, l_, f = oracle.decode_paged(q[b:b + 1], kp, vp, table[b:b + 1], lens[b:b + 1],
                                               np.array([end], np.int32),
                                               sliding_window=end - c * SB + 1, softcap=5.0,
                                               rows=[h])
                assert f == 0
                parts.append((o[0], l_[0]))
            if not parts:
                assert np.isneginf(lse[b * Hq + h]) and not out[b * Hq + h].any()
                continue
            mo, ml = _merge(parts)
            np.testing.assert_allclose(out[b * Hq + h], mo, rtol=0, atol=1e-12)
            assert abs(lse[b * Hq + h] - ml) < 1e-12


@pytest.mark.parametrize("k", [1, 2, 3])
def test_last_k_blocks_equal_a_sliding_window(k):
    rng = np.random.default_rng(40 + k)
    B, Hq, H, D, bs, SB = 2, 4, 1, 8, 16, 32
    lens = np.array([300, 90], np.int32)
    L = int(lens.max())
    kp, vp, table = _paged(rng, B, L, H, D, bs)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    rows = (L + SB - 1) // SB
    lay = [[list(range(max(0, r - k + 1), r + 1)) for r in range(rows)]]
    rp, ci = _csr(lay, rows)
    a = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp, ci, SB)
    for b in range(B):
        qp = int(lens[b]) - 1
        first = max(0, qp // SB - k + 1) * SB
        w = oracle.decode_paged(q[b:b + 1], kp, vp, table[b:b + 1], lens[b:b + 1],
                                sliding_window=qp - first + 1)
        np.testing.assert_allclose(a[0][b * Hq:(b + 1) * Hq], w[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(a[1][b * Hq:(b + 1) * Hq], w[1], rtol=0, atol=1e-13)


def test_matches_torch_sdpa_with_the_boolean_block_mask():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(50)
    B, Hq, H, D, bs, SB, NL = 2, 8, 2, 32, 16, 16, 4
    lens = np.array([250, 131], np.int32)
    L = int(lens.max())
    kp, vp, table = _paged(rng, B, L, H, D, bs)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    rows = (L + SB - 1) // SB
    lays = _strided_layouts(NL, rows, local=2, stride=4)
    rp, ci = _csr(lays, rows)
    out, lse, flags = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp, ci, SB)
    assert flags == 0
    G = Hq // H
    scale = float(np.float32(1 / math.sqrt(D)))
    for b in range(B):
        Lb = int(lens[b])
        pages = table[b]
        kd = np.concatenate([kp[p] for p in pages], 0)[:Lb].astype(np.float64)  # [L, H, D]
        vd = np.concatenate([vp[p] for p in pages], 0)[:Lb].astype(np.float64)
        qp = Lb - 1
        for h in range(Hq):
            cols = set(lays[h % NL][qp // SB])
            mask = np.array([(t // SB) in cols and t <= qp for t in range(Lb)])
            qt = torch.from_numpy(q[b, h].astype(np.float64)).view(1, 1, 1, D)
            kt = torch.from_numpy(kd[:, h // G]).view(1, 1, Lb, D)
            vt = torch.from_numpy(vd[:, h // G]).view(1, 1, Lb, D)
            mt = torch.from_numpy(mask).view(1, 1, 1, Lb)
            ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mt,
                                                                   scale=scale)
            np.testing.assert_allclose(out[b * Hq + h], ref.view(D).numpy(), rtol=0, atol=1e-12)
            s = (kd[:, h // G] @ q[b, h].astype(np.float64)) * scale
            ref_lse = torch.logsumexp(torch.from_numpy(s[mask]), 0).item()
            assert abs(lse[b * Hq + h] - ref_lse) < 1e-12


def test_column_order_and_repeats_change_nothing_bitwise():
    rng = np.random.default_rng(60)
    B, Hq, H, D, bs, SB, NL = 2, 4, 2, 16, 8, 16, 2
    lens = np.array([180, 99], np.int32)
    L = int(lens.max())
    kp, vp, table = _paged(rng, B, L, H, D, bs)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    rows = (L + SB - 1) // SB
    lays = _strided_layouts(NL, rows, local=1, stride=3)
    rp, ci = _csr(lays, rows)
    shuffled = [[list(rng.permutation(r)) + list(r[:2]) for r in lay] for lay in lays]
    rp2, ci2 = _csr(shuffled, rows)
    a = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp, ci, SB)
    b = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp2, ci2, SB)
    assert a[2] == 0 and b[2] == 0
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_heads_cycle_over_the_layouts():
    rng = np.random.default_rng(70)
    B, Hq, H, D, bs, SB, NL = 2, 8, 2, 16, 8, 16, 3
    lens = np.array([150, 70], np.int32)
    L = int(lens.max())
    kp, vp, table = _paged(rng, B, L, H, D, bs)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    rows = (L + SB - 1) // SB
    lays = _strided_layouts(NL, rows, local=2, stride=2 + NL)
    rp, ci = _csr(lays, rows)
    a = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp, ci, SB)
    for l in range(NL):
        rp1, ci1 = _csr([lays[l]], rows)
        one = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp1, ci1, SB)
        for b in range(B):
            for h in range(Hq):
                if h % NL == l:
                    r = b * Hq + h
                    assert np.array_equal(a[0][r], one[0][r]) and a[1][r] == one[1][r]
    # and the layouts differ, so the cycle matters
    assert not np.allclose(a[0][0], oracle.decode_paged_sparse(
        q, kp, vp, table, lens, *_csr([lays[1]], rows), SB)[0][0])


def test_invalid_columns_and_rows_are_flagged_and_select_nothing():
    rng = np.random.default_rng(80)
    B, Hq, H, D, bs, SB = 1, 2, 1, 8, 8, 16
    lens = np.array([64], np.int32)
    kp, vp, table = _paged(rng, B, 64, H, D, bs)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    rows = 4
    good = [[[0], [1], [0, 2], [1, 3]]]
    rp, ci = _csr(good, rows)
    ref = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp, ci, SB)
    assert ref[2] == 0
    bad = [[[0], [1], [0, 2], [1, 3, -1, 4, 99]]]  # row 3 also lists invalid ids
    rp2, ci2 = _csr(bad, rows)
    got = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp2, ci2, SB)
    assert got[2] == FLAG_BAD_BLOCK
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    # a malformed row (end < start) selects nothing
    rp3 = rp.copy()
    rp3[0, 3], rp3[0, 4] = rp[0, 4], rp[0, 3]
    got = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp3, ci, SB)
    assert got[2] == FLAG_BAD_BLOCK
    assert np.isneginf(got[1]).all() and not got[0].any()


def test_empty_selection_gives_zero_and_minus_infinity():
    rng = np.random.default_rng(90)
    B, Hq, H, D, bs, SB = 2, 4, 2, 8, 8, 16
    lens = np.array([40, 33], np.int32)
    kp, vp, table = _paged(rng, B, 40, H, D, bs)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    rows = 3
    lays = [[[], [], []]]
    rp, ci = _csr(lays, rows)
    out, lse, flags = oracle.decode_paged_sparse(q, kp, vp, table, lens, rp, ci, SB)
    assert flags == 0 and np.isneginf(lse).all() and not out.any()
