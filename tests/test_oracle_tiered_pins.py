"""Pins of the tiered oracle's position, ring-slot and error rules.

The tiered decode (int8 cold tier or f16 cold tier, f16 hot ring) is
compared with dense attention in float64 over an explicit list of
(absolute position, K row, V row) that each test writes out by hand:

- cold key t sits at position t, fetched through the block table;
- hot key j sits at position hot_start + j, in ring slot
  (hot_start + j) % hot_window, or slot j when hot_window is 0
  (@simulatte/doppler 0.1.0 attention_decode_tiered_int8_f16kv.wgsl,
  get_hot_pos and the absolute positions of main);
- the query sits at q_pos[b] when given, else at the last cached key
  (hot_start + hot_len - 1, or cold_len - 1 with no hot keys), and the
  causal and window rules of attention_f16kv.wgsl is_masked apply there;
- device-visible errors follow the library's conventions: a cold block id
  outside the pool masks exactly its keys (flag 1), a cold length beyond the
  table is clamped (flag 2), q_pos < 0 empties the row (flag 4), and a
  negative tier length or start, or more hot keys than the ring holds, is
  clamped (flag 16).

Every ring slot and pool page that the rule under test should not read holds
random values, so reading the wrong slot or page changes the result.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle

FLAG_BAD_BLOCK = 1
FLAG_BAD_SEQ_LEN = 2
FLAG_BAD_QPOS = 4
FLAG_BAD_TIER = 16


def _pack_int8(codes):
    """int8 codes [..., D] -> little-endian u32 words [..., D/4]."""
    u = np.asarray(codes, np.int64).astype(np.int8).view(np.uint8).astype(np.uint32)
    u = u.reshape(*u.shape[:-1], -1, 4)
    return u[..., 0] | (u[..., 1] << 8) | (u[..., 2] << 16) | (u[..., 3] << 24)


class Tier:
    """A tiny tiered cache written by hand, plus the dense rows it holds."""

    def __init__(self, rng, kind, B, Hkv, D, bs, max_blocks, cap, extra_pages=3):
        self.kind, self.B, self.Hkv, self.D, self.bs = kind, B, Hkv, D, bs
        NB = B * max_blocks + extra_pages
        self.NB = NB
        ids = rng.permutation(NB)
        self.table = ids[:B * max_blocks].reshape(B, max_blocks).astype(np.int32)
        # every pool page and ring slot starts with random values
        if kind == "int8":
            kc = rng.integers(-128, 128, size=(NB, bs, Hkv, D))
            vc = rng.integers(-128, 128, size=(NB, bs, Hkv, D))
            self.k_scale = (rng.random((NB, bs, Hkv)) * 0.04 + 0.005).astype(np.float16)
            self.v_scale = (rng.random((NB, bs, Hkv)) * 0.04 + 0.005).astype(np.float16)
            self.k_cold = _pack_int8(kc)
            self.v_cold = _pack_int8(vc)
            self.kc_val = kc * self.k_scale[..., None].astype(np.float64)
            self.vc_val = vc * self.v_scale[..., None].astype(np.float64)
        else:
            self.k_cold = rng.standard_normal((NB, bs, Hkv, D)).astype(np.float16)
            self.v_cold = rng.standard_normal((NB, bs, Hkv, D)).astype(np.float16)
            self.kc_val = self.k_cold.astype(np.float64)
            self.vc_val = self.v_cold.astype(np.float64)
        self.k_hot = rng.standard_normal((B, cap, Hkv, D)).astype(np.float16)
        self.v_hot = rng.standard_normal((B, cap, Hkv, D)).astype(np.float16)

    def cold_row(self, b, t):
        """Dense (K, V) of cold key t of sequence b: page table[b][t/bs], row t%bs."""
        blk = self.table[b, t // self.bs]
        return self.kc_val[blk, t % self.bs], self.vc_val[blk, t % self.bs]

    def hot_row(self, b, slot):
        return (self.k_hot[b, slot].astype(np.float64), self.v_hot[b, slot].astype(np.float64))

    def decode(self, q, cold_lens, hot_lens, hot_starts, W, **kw):
        if self.kind == "int8":
            return oracle.decode_tiered(q, self.k_hot, self.v_hot, self.k_cold, self.v_cold,
                                        self.k_scale, self.v_scale, self.table, cold_lens,
                                        hot_lens, hot_starts, hot_window=W, **kw)
        return oracle.decode_tiered_f16(q, self.k_hot, self.v_hot, self.k_cold, self.v_cold,
                                        self.table, cold_lens, hot_lens, hot_starts,
                                        hot_window=W, **kw)


def dense_attention(q, keys, qpos, causal, window, scale, softcap, G):
    """Attention of q [Hq, D] over keys = [(position, K [Hkv, D], V [Hkv, D])]:
    scale, softcap, the causal and window masks at qpos, softmax, V average.
    Returns out [Hq, D], lse [Hq]; an empty visible set gives 0 and -inf."""
    Hq, D = q.shape
    out = np.zeros((Hq, D))
    lse = np.full(Hq, -np.inf)
    vis = [(p, k, v) for (p, k, v) in keys
           if not (causal and p > qpos) and not (window > 0 and qpos >= window and p < qpos - window + 1)]
    if qpos < 0 or not vis:
        return out, lse
    K = np.stack([k for _, k, _ in vis])  # [n, Hkv, D]
    V = np.stack([v for _, _, v in vis])
    for h in range(Hq):
        s = K[:, h // G] @ q[h].astype(np.float64) * scale
        if softcap > 0:
            s = softcap * np.tanh(s / softcap)
        lse[h] = logsumexp(s)
        out[h] = np.exp(s - lse[h]) @ V[:, h // G]
    return out, lse


def check(tier, q, got, want_rows, flags, want_flags):
    out, lse, f = got
    assert f == want_flags, (f, want_flags)
    B, Hq, D = q.shape
    for b in range(B):
        wo, wl = want_rows[b]
        for h in range(Hq):
            r = b * Hq + h
            if np.isneginf(wl[h]):
                assert np.isneginf(lse[r]) and not np.any(out[r]), (b, h)
            else:
                np.testing.assert_allclose(out[r], wo[h], rtol=0, atol=1e-12)
                assert abs(lse[r] - wl[h]) < 1e-12, (b, h, lse[r], wl[h])


def reference(tier, q, cold_lens, hot_lens, hot_starts, slot_of, qpos_of, *, causal=True,
              window=0, scale=0.0, softcap=0.0, bad_pages=()):
    """Dense rows of every sequence: cold keys 0..cold_len-1 (minus the keys of
    bad pages), then hot keys j at hot_start + j read from slot_of(b, j)."""
    B, Hq, D = q.shape
    G = Hq // tier.Hkv
    sc = scale if scale > 0 else float(np.float32(1 / math.sqrt(D)))
    rows = []
    for b in range(B):
        keys = []
        for t in range(cold_lens[b]):
            if (b, t // tier.bs) in bad_pages:
                continue
            k, v = tier.cold_row(b, t)
            keys.append((t, k, v))
        for j in range(hot_lens[b]):
            k, v = tier.hot_row(b, slot_of(b, j))
            keys.append((hot_starts[b] + j, k, v))
        rows.append(dense_attention(q[b], keys, qpos_of(b), causal, window, sc, softcap, G))
    return rows


KINDS = ["int8", "f16"]


@pytest.mark.parametrize("kind", KINDS)
def test_zero_ring_window_reads_hot_key_j_from_slot_j(kind):
    """hot_window = 0: hot key j lives in slot j whatever its position.  Hot
    starts are chosen so that (hot_start + j) % capacity is never j."""
    rng = np.random.default_rng(101)
    B, Hq, H, D, bs, cap = 3, 4, 2, 16, 4, 8
    tier = Tier(rng, kind, B, H, D, bs, max_blocks=4, cap=cap)
    cold = np.array([13, 9, 16], np.int32)
    hot = np.array([5, 8, 3], np.int32)
    starts = np.array([13, 12, 21], np.int32)  # contiguous, overlapping, gap of 5
    for b in range(B):
        assert all((starts[b] + j) % cap != j for j in range(hot[b]))
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    got = tier.decode(q, cold, hot, starts, 0)
    want = reference(tier, q, cold, hot, starts, lambda b, j: j,
                     lambda b: starts[b] + hot[b] - 1)
    check(tier, q, got, want, got[2], 0)


@pytest.mark.parametrize("kind", KINDS)
def test_ring_slot_follows_absolute_position(kind):
    """hot_window W > 0: hot key j lives in slot (hot_start + j) % W, for
    starts that are not multiples of W and rings that are not full."""
    rng = np.random.default_rng(102)
    B, Hq, H, D, bs, W = 3, 8, 2, 16, 4, 6
    tier = Tier(rng, kind, B, H, D, bs, max_blocks=4, cap=W)
    cold = np.array([11, 16, 3], np.int32)
    hot = np.array([6, 4, 1], np.int32)
    starts = np.array([11, 17, 5], np.int32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    got = tier.decode(q, cold, hot, starts, W, softcap=7.0)
    want = reference(tier, q, cold, hot, starts, lambda b, j: (starts[b] + j) % W,
                     lambda b: starts[b] + hot[b] - 1, softcap=7.0)
    check(tier, q, got, want, got[2], 0)


@pytest.mark.parametrize("kind", KINDS)
def test_default_query_position_with_a_window(kind):
    """Default query position: the last hot key, or cold_len - 1 without hot
    keys.  A window of 5 makes the choice visible, including a hot tier that
    starts past the end of the cold tier."""
    rng = np.random.default_rng(103)
    B, Hq, H, D, bs, W = 4, 4, 1, 8, 4, 8
    tier = Tier(rng, kind, B, H, D, bs, max_blocks=5, cap=W)
    cold = np.array([17, 17, 9, 20], np.int32)
    hot = np.array([0, 3, 7, 2], np.int32)
    starts = np.array([17, 23, 9, 20], np.int32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)

    def qp(b):
        return starts[b] + hot[b] - 1 if hot[b] > 0 else cold[b] - 1

    got = tier.decode(q, cold, hot, starts, W, sliding_window=5)
    want = reference(tier, q, cold, hot, starts, lambda b, j: (starts[b] + j) % W, qp,
                     window=5)
    check(tier, q, got, want, got[2], 0)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window", [0, 4])
def test_explicit_query_positions(kind, causal, window):
    """q_pos[b] sets the query position: inside the cold tier, at the
    boundary, inside the hot tier, at the last key and past it."""
    rng = np.random.default_rng(104 + 2 * causal + window)
    B, Hq, H, D, bs, W = 5, 4, 2, 8, 4, 8
    tier = Tier(rng, kind, B, H, D, bs, max_blocks=4, cap=W)
    cold = np.full(B, 12, np.int32)
    hot = np.full(B, 6, np.int32)
    starts = np.full(B, 12, np.int32)
    qpos = np.array([5, 11, 14, 17, 30], np.int32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    got = tier.decode(q, cold, hot, starts, W, q_pos=qpos, causal=causal,
                      sliding_window=window)
    want = reference(tier, q, cold, hot, starts, lambda b, j: (starts[b] + j) % W,
                     lambda b: qpos[b], causal=causal, window=window)
    check(tier, q, got, want, got[2], 0)
    if causal and window == 0:
        # the first row sees exactly keys 0..5: not the default position's 18
        base = tier.decode(q, cold, hot, starts, W)
        assert not np.allclose(got[0][:Hq], base[0][:Hq])


@pytest.mark.parametrize("kind", KINDS)
def test_bad_cold_block_masks_exactly_its_keys(kind):
    rng = np.random.default_rng(105)
    B, Hq, H, D, bs, W = 2, 4, 2, 8, 4, 4
    tier = Tier(rng, kind, B, H, D, bs, max_blocks=4, cap=W)
    cold = np.array([14, 16], np.int32)
    hot = np.array([4, 2], np.int32)
    starts = np.array([14, 16], np.int32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    want_ok = reference(tier, q, cold, hot, starts, lambda b, j: (starts[b] + j) % W,
                        lambda b: starts[b] + hot[b] - 1)
    tier.table[0, 1] = tier.NB          # one past the pool
    tier.table[1, 3] = -1               # negative
    got = tier.decode(q, cold, hot, starts, W)
    want = reference(tier, q, cold, hot, starts, lambda b, j: (starts[b] + j) % W,
                     lambda b: starts[b] + hot[b] - 1, bad_pages={(0, 1), (1, 3)})
    check(tier, q, got, want, got[2], FLAG_BAD_BLOCK)
    assert not np.allclose(got[0], np.concatenate([w[0] for w in want_ok]))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("causal", [True, False])
def test_negative_query_position_empties_only_its_row(kind, causal):
    """q_pos < 0 empties the row even where no mask would (non-causal)."""
    rng = np.random.default_rng(106)
    B, Hq, H, D, bs, W = 3, 4, 2, 8, 4, 4
    tier = Tier(rng, kind, B, H, D, bs, max_blocks=4, cap=W)
    cold = np.full(B, 10, np.int32)
    hot = np.full(B, 3, np.int32)
    starts = np.full(B, 10, np.int32)
    qpos = np.array([12, -1, 7], np.int32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    got = tier.decode(q, cold, hot, starts, W, q_pos=qpos, causal=causal)
    want = reference(tier, q, cold, hot, starts, lambda b, j: (starts[b] + j) % W,
                     lambda b: qpos[b], causal=causal)
    assert np.isneginf(want[1][1]).all()
    check(tier, q, got, want, got[2], FLAG_BAD_QPOS)


@pytest.mark.parametrize("kind", KINDS)
def test_tier_lengths_are_clamped_and_flagged(kind):
    """Per sequence: more hot keys than the ring holds (clamped to W), a
    negative cold length (0), a negative hot start (0), a negative hot length
    (0), and a cold length beyond the table (clamped to max_blocks * bs, flag
    2).  Each result is the dense attention of the clamped cache."""
    rng = np.random.default_rng(107)
    B, Hq, H, D, bs, W, MB = 5, 4, 2, 8, 4, 4, 3
    tier = Tier(rng, kind, B, H, D, bs, max_blocks=MB, cap=W)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    cold = np.array([8, -3, 8, 5, 40], np.int32)
    hot = np.array([9, 2, 3, -2, 1], np.int32)
    starts = np.array([8, 0, -6, 5, 12], np.int32)
    got = tier.decode(q, cold, hot, starts, W)
    c_cold = np.array([8, 0, 8, 5, MB * bs], np.int32)
    c_hot = np.array([W, 2, 3, 0, 1], np.int32)
    c_start = np.array([8, 0, 0, 5, 12], np.int32)

    def qp(b):
        return c_start[b] + c_hot[b] - 1 if c_hot[b] > 0 else c_cold[b] - 1

    want = reference(tier, q, c_cold, c_hot, c_start, lambda b, j: (c_start[b] + j) % W, qp)
    check(tier, q, got, want, got[2], FLAG_BAD_TIER | FLAG_BAD_SEQ_LEN)
    # each clamp alone raises only its own flag
    for b, flag in [(0, FLAG_BAD_TIER), (1, FLAG_BAD_TIER), (2, FLAG_BAD_TIER),
                    (3, FLAG_BAD_TIER), (4, FLAG_BAD_SEQ_LEN)]:
        sel = np.arange(B) == b
        ok_c = np.where(sel, cold, c_cold)
        ok_h = np.where(sel, hot, c_hot)
        ok_s = np.where(sel, starts, c_start)
        assert tier.decode(q, ok_c, ok_h, ok_s, W)[2] == flag
        assert tier.decode(q, c_cold, c_hot, c_start, W)[2] == 0


@pytest.mark.parametrize("kind", KINDS)
def test_zero_ring_window_clamps_hot_length_to_capacity(kind):
    """With hot_window = 0 the ring's bound is its capacity."""
    rng = np.random.default_rng(108)
    B, Hq, H, D, bs, cap = 2, 4, 1, 8, 4, 5
    tier = Tier(rng, kind, B, H, D, bs, max_blocks=2, cap=cap)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    cold = np.array([8, 6], np.int32)
    starts = np.array([8, 9], np.int32)
    got = tier.decode(q, cold, np.array([7, 5], np.int32), starts, 0)
    want = reference(tier, q, cold, np.array([cap, 5]), starts, lambda b, j: j,
                     lambda b: starts[b] + (cap if b == 0 else 5) - 1)
    check(tier, q, got, want, got[2], FLAG_BAD_TIER)
