"""Pins of the CPU oracle to things other than itself.

Each test checks the oracle against something the pages or the mathematics
fix independently of the oracle's code: hand-decoded formats, hand-worked
tiny cases, library routines (numpy's binary16 decoder, torch's float64
scaled_dot_product_attention, scipy's logsumexp), closed forms, and
invariances of the definition.  Together they are meant to catch a dropped
term, a wrong sign or index, or a transposed operand anywhere in the oracle.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# helpers: tiny caches laid out by hand (no attention arithmetic here)
# ---------------------------------------------------------------------------

def paged_from_dense(k, v, bs, rng=None, extra_pages=0):
    """Place dense K/V [B, L, Hkv, D] into a pool [NB, bs, Hkv, D] through a
    block table, optionally with shuffled page ids and unused pages."""
    B, L, H, D = k.shape
    npg = (L + bs - 1) // bs
    NB = B * npg + extra_pages
    ids = np.arange(NB) if rng is None else rng.permutation(NB)
    table = ids[:B * npg].reshape(B, npg).astype(np.int32)
    kp = np.zeros((NB, bs, H, D), np.float16)
    vp = np.zeros((NB, bs, H, D), np.float16)
    for b in range(B):
        for t in range(L):
            kp[table[b, t // bs], t % bs] = k[b, t]
            vp[table[b, t // bs], t % bs] = v[b, t]
    return kp, vp, table


def rand_dense(rng, B, L, Hkv, D, scale=1.0):
    k = (rng.standard_normal((B, L, Hkv, D)) * scale).astype(np.float16)
    v = (rng.standard_normal((B, L, Hkv, D)) * scale).astype(np.float16)
    return k, v


# ---------------------------------------------------------------------------
# formats
# ---------------------------------------------------------------------------

def test_half_decoder_matches_numpy_for_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero
    assert math.copysign(1.0, got[0x8000]) == -1.0


def test_half_decoder_golden():
    n = 0
    with open(os.path.join(GOLDEN, "f16_bits.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            bits, val = line.split()
            want = float(val)
            got = oracle.half_to_double(int(bits, 16))
            assert got == want, (bits, got, want)
            if want == 0.0:
                assert math.copysign(1.0, got) == math.copysign(1.0, want)
            n += 1
    assert n >= 16


def test_int8_word_decode_golden():
    n = 0
    with open(os.path.join(GOLDEN, "int8_words.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            word, *vals = line.split()
            assert oracle.unpack_int8_word(int(word, 16)) == [int(x) for x in vals], word
            n += 1
    assert n >= 10


# ---------------------------------------------------------------------------
# hand-worked cases
# ---------------------------------------------------------------------------

def _eval(expr):
    ns = {"e": math.e, "exp": math.exp, "log": math.log, "tanh": math.tanh, "inf": math.inf}
    return float(eval(expr, {"__builtins__": {}}, ns))


def _hand_cases():
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _hand_cases(), ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    D, bs = case["D"], case["block_size"]
    k = np.array(case["k"], dtype=np.float16).reshape(1, -1, 1, D)
    v = np.array(case["v"], dtype=np.float16).reshape(1, -1, 1, D)
    kp, vp, table = paged_from_dense(k, v, bs)
    q = np.array(case["q"], dtype=np.float32).reshape(1, 1, D)
    q_pos = None if case["q_pos"] is None else np.array([case["q_pos"]], np.int32)
    out, lse, flags = oracle.decode_paged(
        q, kp, vp, table, np.array([case["seq_len"]], np.int32), q_pos,
        scale=case["scale"], softcap=case["softcap"], sliding_window=case["window"],
        causal=bool(case["causal"]))
    assert flags == 0
    want_out = np.array([_eval(x) for x in case["out"]])
    want_lse = _eval(case["lse"])
    np.testing.assert_allclose(out[0], want_out, rtol=1e-14, atol=1e-15)
    if math.isinf(want_lse):
        assert lse[0] == want_lse
    else:
        assert abs(lse[0] - want_lse) < 1e-14


# ---------------------------------------------------------------------------
# library routines: torch float64 SDPA and scipy logsumexp on the dense cache
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed,B,Hq,Hkv,D,bs,window,causal", [
    (0, 2, 4, 2, 16, 4, 0, True),
    (1, 3, 8, 2, 32, 8, 0, False),
    (2, 2, 6, 3, 8, 2, 5, True),
    (3, 1, 4, 4, 64, 16, 17, True),
    (4, 2, 8, 1, 24, 8, 3, False),
])
def test_matches_torch_sdpa_float64(seed, B, Hq, Hkv, D, bs, window, causal):
    torch = pytest.importorskip("torch")
    from scipy.special import logsumexp

    rng = np.random.default_rng(seed)
    Lmax = 37
    lens = rng.integers(1, Lmax + 1, size=B).astype(np.int32)
    k, v = rand_dense(rng, B, Lmax, Hkv, D)
    kp, vp, table = paged_from_dense(k, v, bs, rng=rng, extra_pages=3)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    qpos = np.array([rng.integers(0, L) if causal else rng.integers(0, Lmax) for L in lens],
                    dtype=np.int32)
    scale = np.float32(1.0 / math.sqrt(D))
    out, lse, flags = oracle.decode_paged(q, kp, vp, table, lens, qpos, scale=float(scale),
                                          sliding_window=window, causal=causal)
    assert flags == 0
    G = Hq // Hkv
    for b in range(B):
        L = int(lens[b])
        p = int(qpos[b])
        t = np.arange(L)
        vis = np.ones(L, bool)
        if causal:
            vis &= t <= p
        if window > 0 and p >= window:
            vis &= t >= p - window + 1
        Kd = torch.from_numpy(k[b, :L].astype(np.float64)).permute(1, 0, 2)  # [Hkv, L, D]
        Vd = torch.from_numpy(v[b, :L].astype(np.float64)).permute(1, 0, 2)
        Kd = Kd.repeat_interleave(G, dim=0)
        Vd = Vd.repeat_interleave(G, dim=0)
        Qd = torch.from_numpy(q[b].astype(np.float64)).unsqueeze(1)  # [Hq, 1, D]
        mask = torch.from_numpy(vis).view(1, 1, L).expand(Hq, 1, L)
        ref = torch.nn.functional.scaled_dot_product_attention(
            Qd, Kd, Vd, attn_mask=mask, scale=float(scale))[:, 0, :].numpy()
        scores = (Qd @ Kd.transpose(1, 2))[:, 0, :].numpy() * float(scale)
        ref_lse = logsumexp(np.where(vis[None, :], scores, -np.inf), axis=1)
        np.testing.assert_allclose(out[b * Hq:(b + 1) * Hq], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[b * Hq:(b + 1) * Hq], ref_lse, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def test_single_visible_key_returns_its_value_row():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, D, bs, L = 2, 4, 2, 16, 4, 11
    k, v = rand_dense(rng, B, L, Hkv, D)
    kp, vp, table = paged_from_dense(k, v, bs, rng=rng)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    out, lse, _ = oracle.decode_paged(q, kp, vp, table, np.full(B, L, np.int32),
                                      scale=0.25, sliding_window=1)
    for b in range(B):
        for h in range(Hq):
            kv = h // (Hq // Hkv)
            assert np.array_equal(out[b * Hq + h], v[b, L - 1, kv].astype(np.float64))
            s = 0.25 * float(np.dot(q[b, h].astype(np.float64), k[b, L - 1, kv].astype(np.float64)))
            assert abs(lse[b * Hq + h] - s) < 1e-12


def test_constant_value_rows_return_the_constant():
    rng = np.random.default_rng(6)
    B, Hq, Hkv, D, bs, L = 1, 4, 1, 8, 4, 29
    k, _ = rand_dense(rng, B, L, Hkv, D)
    v = np.broadcast_to(np.arange(D, dtype=np.float16) - 3, (B, L, Hkv, D)).copy()
    kp, vp, table = paged_from_dense(k, v, bs, rng=rng)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32) * 3
    out, _, _ = oracle.decode_paged(q, kp, vp, table, np.array([L], np.int32))
    np.testing.assert_allclose(out, np.broadcast_to(np.arange(D) - 3.0, out.shape), atol=1e-13)


def test_zero_keys_give_log_count_and_mean_value():
    rng = np.random.default_rng(7)
    B, Hq, Hkv, D, bs = 3, 2, 1, 8, 4
    lens = np.array([1, 7, 23], np.int32)
    k = np.zeros((B, 23, Hkv, D), np.float16)
    _, v = rand_dense(rng, B, 23, Hkv, D)
    kp, vp, table = paged_from_dense(k, v, bs, rng=rng)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    out, lse, _ = oracle.decode_paged(q, kp, vp, table, lens, sliding_window=5)
    for b in range(B):
        n = min(int(lens[b]), 5)
        for h in range(Hq):
            assert abs(lse[b * Hq + h] - math.log(n)) < 1e-14
            want = v[b, lens[b] - n:lens[b], 0].astype(np.float64).mean(axis=0)
            np.testing.assert_allclose(out[b * Hq + h], want, atol=1e-14)


def test_softcap_saturation_closed_form():
    # cap = 1 and |q.k| huge: every score becomes +-1 (tanh saturates).
    D, bs = 4, 2
    k = np.array([[100, 0, 0, 0], [-100, 0, 0, 0], [100, 0, 0, 0]], np.float16).reshape(1, 3, 1, D)
    v = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [0, 0, 1, 0]], np.float16).reshape(1, 3, 1, D)
    kp, vp, table = paged_from_dense(k, v, bs)
    q = np.array([[[100, 0, 0, 0]]], np.float32)
    out, lse, _ = oracle.decode_paged(q, kp, vp, table, np.array([3], np.int32), scale=1.0,
                                      softcap=1.0)
    Z = 2 * math.e + math.exp(-1)
    np.testing.assert_allclose(out[0], [math.e / Z, math.exp(-1) / Z, math.e / Z, 0], atol=1e-15)
    assert abs(lse[0] - math.log(Z)) < 1e-14


# ---------------------------------------------------------------------------
# invariances of the definition
# ---------------------------------------------------------------------------

def test_block_permutation_invariance_is_bitwise():
    rng = np.random.default_rng(8)
    B, Hq, Hkv, D, bs, L = 2, 4, 2, 16, 4, 30
    k, v = rand_dense(rng, B, L, Hkv, D)
    kp, vp, table = paged_from_dense(k, v, bs, extra_pages=4)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    lens = np.array([30, 13], np.int32)
    a = oracle.decode_paged(q, kp, vp, table, lens, softcap=7.0)
    perm = rng.permutation(kp.shape[0])          # new id of old page i is perm[i]
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    table2 = perm[table].astype(np.int32)
    b_ = oracle.decode_paged(q, kp2, vp2, table2, lens, softcap=7.0)
    assert np.array_equal(a[0], b_[0]) and np.array_equal(a[1], b_[1])


def test_sliding_window_equals_truncated_dense_cache():
    rng = np.random.default_rng(9)
    B, Hq, Hkv, D, bs, L, W = 2, 4, 2, 16, 4, 41, 9
    k, v = rand_dense(rng, B, L, Hkv, D)
    kp, vp, table = paged_from_dense(k, v, bs, rng=rng)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    a_out, a_lse, _ = oracle.decode_paged(q, kp, vp, table, np.full(B, L, np.int32),
                                          sliding_window=W)
    kt, vt = k[:, L - W:], v[:, L - W:]
    kp2, vp2, table2 = paged_from_dense(kt, vt, bs)
    b_out, b_lse, _ = oracle.decode_paged(q, kp2, vp2, table2, np.full(B, W, np.int32))
    assert np.array_equal(a_out, b_out) and np.array_equal(a_lse, b_lse)


def test_huge_softcap_equals_no_softcap():
    rng = np.random.default_rng(10)
    B, Hq, Hkv, D, bs, L = 2, 4, 2, 32, 8, 50
    k, v = rand_dense(rng, B, L, Hkv, D)
    kp, vp, table = paged_from_dense(k, v, bs, rng=rng)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    a = oracle.decode_paged(q, kp, vp, table, np.full(B, L, np.int32))
    b_ = oracle.decode_paged(q, kp, vp, table, np.full(B, L, np.int32), softcap=1e12)
    np.testing.assert_allclose(a[0], b_[0], atol=1e-12)
    np.testing.assert_allclose(a[1], b_[1], atol=1e-12)
    c = oracle.decode_paged(q, kp, vp, table, np.full(B, L, np.int32), softcap=0.5)
    assert np.abs(c[1] - a[1]).max() > 1e-3   # a small cap does change the result


def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(11)
    B, Hq, Hkv, D, bs, L = 2, 8, 2, 16, 4, 21
    G = Hq // Hkv
    k, v = rand_dense(rng, B, L, Hkv, D)
    kp, vp, table = paged_from_dense(k, v, bs, rng=rng)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    a = oracle.decode_paged(q, kp, vp, table, np.full(B, L, np.int32), softcap=3.0)
    k2 = np.repeat(k, G, axis=2)
    v2 = np.repeat(v, G, axis=2)
    kp2, vp2, table2 = paged_from_dense(k2, v2, bs, rng=rng)
    b_ = oracle.decode_paged(q, kp2, vp2, table2, np.full(B, L, np.int32), softcap=3.0)
    assert np.array_equal(a[0], b_[0]) and np.array_equal(a[1], b_[1])


@pytest.mark.parametrize("split_tokens", [4, 8, 16, 64])
def test_split_merge_equals_unsplit(split_tokens):
    rng = np.random.default_rng(12)
    B, Hq, Hkv, D, bs = 3, 4, 2, 16, 4
    lens = np.array([0, 19, 57], np.int32)
    k, v = rand_dense(rng, B, 57, Hkv, D, scale=2.0)
    kp, vp, table = paged_from_dense(k, v, bs, rng=rng)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    S = (57 + split_tokens - 1) // split_tokens
    out, lse, _ = oracle.decode_paged(q, kp, vp, table, lens, sliding_window=40)
    op, lp, flags = oracle.decode_paged_split(q, kp, vp, table, lens, split_tokens=split_tokens,
                                              max_splits=S, sliding_window=40)
    assert flags == 0
    mo, ml = oracle.split_merge(op, lp)
    np.testing.assert_allclose(mo, out, atol=1e-12)
    np.testing.assert_allclose(ml, lse, atol=1e-12)


def test_split_overflow_flag():
    rng = np.random.default_rng(13)
    k, v = rand_dense(rng, 1, 40, 1, 8)
    kp, vp, table = paged_from_dense(k, v, 4)
    q = rng.standard_normal((1, 1, 8)).astype(np.float32)
    _, _, flags = oracle.decode_paged_split(q, kp, vp, table, np.array([40], np.int32),
                                            split_tokens=8, max_splits=4)
    assert flags & oracle.FLAG_SPLIT_OVERFLOW


# ---------------------------------------------------------------------------
# tiered cache
# ---------------------------------------------------------------------------

def _tiered_from_dense(kc_int, vc_int, ks, vs, kh, vh, bs, hot_window, hot_start, rng=None):
    """Cold int8 values [B, C, H, D] with f16 scales [B, C, H] into pages; hot
    rows [B, Hl, H, D] into the ring at slot (hot_start + j) % W."""
    B, C, H, D = kc_int.shape
    npg = max(1, (C + bs - 1) // bs)
    NB = B * npg
    ids = np.arange(NB) if rng is None else rng.permutation(NB)
    table = ids.reshape(B, npg).astype(np.int32)
    words_k = np.zeros((NB, bs, H, D // 4), np.uint32)
    words_v = np.zeros_like(words_k)
    sk = np.zeros((NB, bs, H), np.float16)
    sv = np.zeros_like(sk)
    def pack(x):
        u = x.astype(np.int8).view(np.uint8).astype(np.uint32).reshape(-1, 4)
        return u[:, 0] | (u[:, 1] << 8) | (u[:, 2] << 16) | (u[:, 3] << 24)
    for b in range(B):
        for t in range(C):
            for h in range(H):
                words_k[table[b, t // bs], t % bs, h] = pack(kc_int[b, t, h])
                words_v[table[b, t // bs], t % bs, h] = pack(vc_int[b, t, h])
                sk[table[b, t // bs], t % bs, h] = ks[b, t, h]
                sv[table[b, t // bs], t % bs, h] = vs[b, t, h]
    Hl = kh.shape[1]
    cap = max(hot_window, Hl, 1)
    hk = np.zeros((B, cap, H, D), np.float16)
    hv = np.zeros_like(hk)
    for j in range(Hl):
        slot = (hot_start + j) % hot_window if hot_window > 0 else j
        hk[:, slot] = kh[:, j]
        hv[:, slot] = vh[:, j]
    return hk, hv, words_k, words_v, sk, sv, table


def test_int8_tier_with_unit_scales_equals_f16_paged_bitwise():
    rng = np.random.default_rng(14)
    B, Hq, H, D, bs, C = 2, 4, 2, 16, 4, 22
    kc = rng.integers(-127, 128, size=(B, C, H, D))
    vc = rng.integers(-127, 128, size=(B, C, H, D))
    ones = np.ones((B, C, H), np.float16)
    empty = np.zeros((B, 0, H, D), np.float16)
    hk, hv, wk, wv, sk, sv, table = _tiered_from_dense(kc, vc, ones, ones, empty, empty, bs,
                                                       hot_window=0, hot_start=C, rng=rng)
    q = (rng.standard_normal((B, Hq, D)) * 0.05).astype(np.float32)
    a = oracle.decode_tiered(q, hk, hv, wk, wv, sk, sv, table, C, 0, C, hot_window=0,
                             softcap=30.0)
    kp, vp, table2 = paged_from_dense(kc.astype(np.float16), vc.astype(np.float16), bs, rng=rng)
    b_ = oracle.decode_paged(q, kp, vp, table2, np.full(B, C, np.int32), softcap=30.0)
    assert a[2] == 0 and b_[2] == 0
    assert np.array_equal(a[0], b_[0]) and np.array_equal(a[1], b_[1])


def test_int8_scales_multiply_each_value():
    # one cold key: out must be int8 * v_scale; lse = scale * sum q_d int8_d * k_scale
    D = 8
    kc = np.array([[[[1, -2, 3, -4, 127, -128, 0, 5]]]])
    vc = np.array([[[[-1, 2, -3, 4, -127, 127, 9, 0]]]])
    ks = np.array([[[0.5]]], np.float16)
    vs = np.array([[[0.25]]], np.float16)
    empty = np.zeros((1, 0, 1, D), np.float16)
    hk, hv, wk, wv, sk, sv, table = _tiered_from_dense(kc, vc, ks, vs, empty, empty, 16, 0, 1)
    q = np.arange(D, dtype=np.float32).reshape(1, 1, D)
    out, lse, _ = oracle.decode_tiered(q, hk, hv, wk, wv, sk, sv, table, 1, 0, 1, hot_window=0,
                                       scale=1.0)
    np.testing.assert_array_equal(out[0], vc[0, 0, 0] * 0.25)
    assert lse[0] == float(np.dot(np.arange(D), kc[0, 0, 0]) * 0.5)


def test_tiered_equals_dense_attention_over_logical_order():
    """Cold + hot keys against a dense f16 cache holding the dequantised cold
    rows followed by the hot rows (positions contiguous)."""
    rng = np.random.default_rng(15)
    B, Hq, H, D, bs, C, Hl, W = 2, 4, 2, 16, 4, 13, 6, 8
    kc = rng.integers(-127, 128, size=(B, C, H, D))
    vc = rng.integers(-127, 128, size=(B, C, H, D))
    ks = (rng.random((B, C, H)) * 0.05 + 0.001).astype(np.float16)
    vs = (rng.random((B, C, H)) * 0.05 + 0.001).astype(np.float16)
    kh, vh = rand_dense(rng, B, Hl, H, D)
    hk, hv, wk, wv, sk, sv, table = _tiered_from_dense(kc, vc, ks, vs, kh, vh, bs, W, C, rng=rng)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    a_out, a_lse, flags = oracle.decode_tiered(q, hk, hv, wk, wv, sk, sv, table, C, Hl, C,
                                               hot_window=W, softcap=20.0, sliding_window=15)
    assert flags == 0
    # dense reference in float64 through scipy
    from scipy.special import logsumexp
    G = Hq // H
    kd = np.concatenate([kc * ks[..., None].astype(np.float64), kh.astype(np.float64)], axis=1)
    vd = np.concatenate([vc * vs[..., None].astype(np.float64), vh.astype(np.float64)], axis=1)
    L = C + Hl
    vis = np.arange(L) >= L - 15
    scale = float(np.float32(1 / math.sqrt(D)))
    for b in range(B):
        for h in range(Hq):
            s = kd[b, :, h // G] @ q[b, h].astype(np.float64) * scale
            s = 20.0 * np.tanh(s / 20.0)
            s = np.where(vis, s, -np.inf)
            lse = logsumexp(s)
            w = np.exp(s - lse)
            np.testing.assert_allclose(a_out[b * Hq + h], w @ vd[b, :, h // G], atol=1e-12)
            assert abs(a_lse[b * Hq + h] - lse) < 1e-12


def _tiered_f16_from_dense(kc, vc, kh, vh, bs, hot_window, hot_start, rng=None):
    """f16 cold rows [B, C, H, D] into pages [NB, bs, H, D]; hot rows into the
    ring as in _tiered_from_dense."""
    B, C, H, D = kc.shape
    zc = np.zeros((B, C, H, D), np.int64)
    zs = np.zeros((B, C, H), np.float16)
    hk, hv, _, _, _, _, table = _tiered_from_dense(zc, zc, zs, zs, kh, vh, bs, hot_window,
                                                   hot_start, rng=rng)
    NB = table.size
    pk = np.zeros((NB, bs, H, D), np.float16)
    pv = np.zeros_like(pk)
    for b in range(B):
        for t in range(C):
            pk[table[b, t // bs], t % bs] = kc[b, t]
            pv[table[b, t // bs], t % bs] = vc[b, t]
    return hk, hv, pk, pv, table


def test_f16_tier_equals_int8_tier_on_integer_data_bitwise():
    """Cold values that are integers in [-127, 127] are exact in f16: the f16
    cold tier must give bit-identical results to the int8 tier with unit
    scales holding the same integers (hot ring shared)."""
    rng = np.random.default_rng(18)
    B, Hq, H, D, bs, C, Hl, W = 2, 8, 2, 16, 8, 19, 5, 8
    kc = rng.integers(-127, 128, size=(B, C, H, D))
    vc = rng.integers(-127, 128, size=(B, C, H, D))
    kh, vh = rand_dense(rng, B, Hl, H, D)
    ones = np.ones((B, C, H), np.float16)
    hk, hv, wk, wv, sk, sv, table = _tiered_from_dense(kc, vc, ones, ones, kh, vh, bs, W, C,
                                                       rng=np.random.default_rng(3))
    hk2, hv2, pk, pv, table2 = _tiered_f16_from_dense(kc.astype(np.float16),
                                                      vc.astype(np.float16), kh, vh, bs, W, C,
                                                      rng=np.random.default_rng(3))
    q = (rng.standard_normal((B, Hq, D)) * 0.05).astype(np.float32)
    a = oracle.decode_tiered(q, hk, hv, wk, wv, sk, sv, table, C, Hl, C, hot_window=W,
                             softcap=30.0)
    b_ = oracle.decode_tiered_f16(q, hk2, hv2, pk, pv, table2, C, Hl, C, hot_window=W,
                                  softcap=30.0)
    assert a[2] == 0 and b_[2] == 0
    assert np.array_equal(a[0], b_[0]) and np.array_equal(a[1], b_[1])


def test_f16_tier_equals_dense_attention_over_logical_order():
    """f16 cold + hot keys against a dense f16 cache holding the cold rows
    followed by the hot rows (positions contiguous), with window and softcap."""
    rng = np.random.default_rng(19)
    B, Hq, H, D, bs, C, Hl, W = 2, 4, 2, 16, 4, 13, 6, 8
    kc, vc = rand_dense(rng, B, C, H, D)
    kh, vh = rand_dense(rng, B, Hl, H, D)
    hk, hv, pk, pv, table = _tiered_f16_from_dense(kc, vc, kh, vh, bs, W, C, rng=rng)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    a_out, a_lse, flags = oracle.decode_tiered_f16(q, hk, hv, pk, pv, table, C, Hl, C,
                                                   hot_window=W, softcap=20.0, sliding_window=15)
    assert flags == 0
    from scipy.special import logsumexp
    G = Hq // H
    kd = np.concatenate([kc, kh], axis=1).astype(np.float64)
    vd = np.concatenate([vc, vh], axis=1).astype(np.float64)
    L = C + Hl
    vis = np.arange(L) >= L - 15
    scale = float(np.float32(1 / math.sqrt(D)))
    for b in range(B):
        for h in range(Hq):
            s = kd[b, :, h // G] @ q[b, h].astype(np.float64) * scale
            s = 20.0 * np.tanh(s / 20.0)
            s = np.where(vis, s, -np.inf)
            lse = logsumexp(s)
            w = np.exp(s - lse)
            np.testing.assert_allclose(a_out[b * Hq + h], w @ vd[b, :, h // G], atol=1e-12)
            assert abs(a_lse[b * Hq + h] - lse) < 1e-12


def test_hot_ring_rotation_invariance():
    """The same hot keys stored at a different ring phase (hot_start not a
    multiple of the window) give bit-identical results."""
    rng = np.random.default_rng(16)
    B, Hq, H, D, bs, Hl, W = 1, 2, 1, 8, 4, 7, 10
    kh, vh = rand_dense(rng, B, Hl, H, D)
    zero_c = np.zeros((B, 0, H, D), np.int64)
    zs = np.zeros((B, 0, H), np.float16)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    res = []
    for hot_start in (0, 3, 13, 27):
        hk, hv, wk, wv, sk, sv, table = _tiered_from_dense(zero_c, zero_c, zs, zs, kh, vh, bs, W,
                                                           hot_start)
        res.append(oracle.decode_tiered(q, hk, hv, wk, wv, sk, sv, table, 0, Hl, hot_start,
                                        hot_window=W))
    for r in res[1:]:
        assert np.array_equal(r[0], res[0][0]) and np.array_equal(r[1], res[0][1])
    # a wrong phase (reading slot j instead of (start+j)%W) would differ
    hk, hv, wk, wv, sk, sv, table = _tiered_from_dense(zero_c, zero_c, zs, zs, kh, vh, bs, W, 3)
    wrong = oracle.decode_tiered(q, hk, hv, wk, wv, sk, sv, table, 0, Hl, 0, hot_window=W)
    assert not np.array_equal(wrong[0], res[0][0])


# ---------------------------------------------------------------------------
# device-visible error conventions (restated in the oracle)
# ---------------------------------------------------------------------------

def test_bad_block_id_masks_its_keys_and_flags():
    rng = np.random.default_rng(17)
    k, v = rand_dense(rng, 1, 12, 1, 8)
    kp, vp, table = paged_from_dense(k, v, 4)
    q = rng.standard_normal((1, 2, 8)).astype(np.float32)
    bad = table.copy()
    bad[0, 1] = 999
    out, lse, flags = oracle.decode_paged(q, kp, vp, bad, np.array([12], np.int32))
    assert flags & oracle.FLAG_BAD_BLOCK
    # equals attention over keys 0-3 and 8-11 only
    keep = np.r_[0:4, 8:12]
    kp2, vp2, t2 = paged_from_dense(k[:, keep], v[:, keep], 4)
    ref = oracle.decode_paged(q, kp2, vp2, t2, np.array([8], np.int32), causal=False)
    np.testing.assert_array_equal(out, ref[0])


def test_length_beyond_table_is_clamped_and_flagged():
    rng = np.random.default_rng(18)
    k, v = rand_dense(rng, 1, 8, 1, 8)
    kp, vp, table = paged_from_dense(k, v, 4)
    q = rng.standard_normal((1, 1, 8)).astype(np.float32)
    a = oracle.decode_paged(q, kp, vp, table, np.array([100], np.int32), causal=False)
    b_ = oracle.decode_paged(q, kp, vp, table, np.array([8], np.int32), causal=False)
    assert a[2] & oracle.FLAG_BAD_SEQ_LEN and b_[2] == 0
    np.testing.assert_array_equal(a[0], b_[0])


def test_negative_qpos_gives_empty_row():
    rng = np.random.default_rng(19)
    k, v = rand_dense(rng, 1, 8, 1, 8)
    kp, vp, table = paged_from_dense(k, v, 4)
    q = rng.standard_normal((1, 1, 8)).astype(np.float32)
    out, lse, flags = oracle.decode_paged(q, kp, vp, table, np.array([8], np.int32),
                                          np.array([-3], np.int32))
    assert flags & oracle.FLAG_BAD_QPOS
    assert not out.any() and lse[0] == -np.inf


# ---------------------------------------------------------------------------
# KV append and int8 demotion
# ---------------------------------------------------------------------------

def test_float_to_half_matches_numpy_round_to_nearest_even():
    """The oracle's binary16 encoder against numpy's f32 -> f16 cast (IEEE
    round to nearest even) on every exact tie between neighbouring f16
    values, the f32 values either side of each tie, and random patterns."""
    h = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + h[1:]) / 2  # exact in f32 (12 significant bits)
    m32 = mids.astype(np.float32)
    cand = np.concatenate([m32, np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(1e9)),
                           np.float32([0.0, 65504.0, 65519.996, 65520.0, 1e9, 2.0 ** -25,
                                       2.0 ** -24, 3 * 2.0 ** -26])])
    rng = np.random.default_rng(20)
    rnd = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    cand = np.concatenate([cand, -cand, rnd])
    cand = cand[np.isfinite(cand)]
    with np.errstate(over="ignore"):
        want = cand.astype(np.float16).view(np.uint16)
    got = oracle.float_to_half(cand)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (cand[bad[:5]], got[bad[:5]], want[bad[:5]])
    assert oracle.float_to_half(np.float32([np.inf, -np.inf]))[0] == 0x7c00
    assert oracle.float_to_half(np.float32([np.nan]))[0] & 0x7fff > 0x7c00


def test_demotion_quantizer_golden_and_ties():
    code, s = oracle.quantize_row_int8(np.array([127, -127, 63.5, 62.5, 0.5, -1.5, 1.5, 0],
                                                np.float16))
    assert s == 0x3c00  # f16(127 / 127) = 1.0
    assert code.tolist() == [127, -127, 64, 62, 0, -2, 2, 0]  # ties to even
    code, s = oracle.quantize_row_int8(np.zeros(8, np.float16))
    assert s == 0 and not code.any()
    # scale = f16(max|x| / 127) with the division in f32
    x = np.array([3.0, -0.1, 2.9], np.float16)
    code, s = oracle.quantize_row_int8(x)
    assert s == int(np.array(np.float32(3.0) / np.float32(127.0), np.float32)
                    .astype(np.float16).view(np.uint16))


def test_demotion_quantizer_error_bound_and_agreement_with_input_quantizer():
    """Every code reconstructs its value within half a scale step (no value
    exceeds 127 steps), and the oracle's quantizer agrees bit for bit with
    the independent numpy quantizer that makes the int8 workload inputs."""
    from quantized_kv_decode_paged_gb300.workloads import quantize_int8_rows
    rng = np.random.default_rng(21)
    for D in (8, 64, 128, 256):
        for sc in (1e-4, 0.01, 1.0, 300.0):
            x = (rng.standard_normal(D) * sc).astype(np.float16)
            code, s = oracle.quantize_row_int8(x)
            s_val = float(np.uint16(s).view(np.float16))
            q_ref, s_ref = quantize_int8_rows(x[None])
            assert int(s_ref.view(np.uint16)[0]) == s
            assert np.array_equal(q_ref[0], code)
            err = np.abs(code.astype(np.float64) * s_val - x.astype(np.float64))
            lim = np.abs(x.astype(np.float64)) <= 127 * s_val
            assert (err[lim] <= s_val / 2 * (1 + 1e-6)).all()
            assert np.abs(code).max() <= 127
            if s_val >= 2.0 ** -14:  # a normal f16 scale is within 2^-11 of max|x|/127
                assert np.abs(code).max() >= 126


def _empty_tier(B, H, D, bs, W, npages, rng, f16=False):
    NB = B * npages
    table = rng.permutation(NB).reshape(B, npages).astype(np.int32)
    kh = np.zeros((B, W, H, D), np.float16)
    if f16:
        kc = np.zeros((NB, bs, H, D), np.float16)
        ks = None
    else:
        kc = np.zeros((NB, bs, H, D // 4), np.uint32)
        ks = np.zeros((NB, bs, H), np.float16)
    return kh, kc, ks, table


def _words_to_int8(words):
    return words.view(np.uint8).view(np.int8)


@pytest.mark.parametrize("f16", [False, True])
def test_append_tiered_state_machine(f16):
    """W = 4: the first four appends fill the ring; each later append first
    moves the oldest hot token (position hot_start) to cold position
    cold_len (quantized, or copied for the f16 tier) and then writes the new
    token into the freed slot."""
    rng = np.random.default_rng(22)
    B, H, D, bs, W = 2, 2, 16, 4, 4
    kh, kc, ks, table = _empty_tier(B, H, D, bs, W, 3, rng, f16)
    st = dict(k_hot=kh, v_hot=kh.copy(), k_cold=kc, v_cold=kc.copy(), k_scale=ks,
              v_scale=None if ks is None else ks.copy(), cold_lens=np.full(B, 5, np.int32),
              hot_lens=np.zeros(B, np.int32), hot_starts=np.full(B, 5, np.int32))
    toks_k = rng.standard_normal((7, B, H, D)).astype(np.float16)
    toks_v = rng.standard_normal((7, B, H, D)).astype(np.float16)
    for i in range(7):
        st, flags = oracle.append_tiered(toks_k[i], toks_v[i], st["k_hot"], st["v_hot"],
                                         st["k_cold"], st["v_cold"], st.get("k_scale"),
                                         st.get("v_scale"), table, st["cold_lens"],
                                         st["hot_lens"], st["hot_starts"], hot_window=W)
        assert flags == 0
        n_demoted = max(0, i + 1 - W)
        assert (st["hot_lens"] == min(i + 1, W)).all()
        assert (st["cold_lens"] == 5 + n_demoted).all() and (st["hot_starts"] == 5 + n_demoted).all()
    for b in range(B):
        # hot token j (position 5 + 3 + j) sits in slot (8 + j) % 4 and is token 3 + j
        for j in range(W):
            slot = (8 + j) % W
            assert np.array_equal(st["k_hot"][b, slot], toks_k[3 + j, b])
            assert np.array_equal(st["v_hot"][b, slot], toks_v[3 + j, b])
        # cold positions 5, 6, 7 hold tokens 0, 1, 2
        for j in range(3):
            pos = 5 + j
            page, row = table[b, pos // bs], pos % bs
            for h in range(H):
                if f16:
                    assert np.array_equal(st["k_cold"][page, row, h], toks_k[j, b, h])
                    assert np.array_equal(st["v_cold"][page, row, h], toks_v[j, b, h])
                else:
                    code, s = oracle.quantize_row_int8(toks_k[j, b, h])
                    assert np.array_equal(_words_to_int8(st["k_cold"][page, row, h]), code)
                    assert int(st["k_scale"][page, row, h].view(np.uint16)) == s
                    code, s = oracle.quantize_row_int8(toks_v[j, b, h])
                    assert np.array_equal(_words_to_int8(st["v_cold"][page, row, h]), code)
                    assert int(st["v_scale"][page, row, h].view(np.uint16)) == s


def test_append_then_decode_equals_dense_attention():
    """After appends that demote tokens, the tiered decode of the updated
    cache equals dense attention over (dequantized demoted tokens, hot
    tokens) in logical order."""
    from scipy.special import logsumexp
    rng = np.random.default_rng(23)
    B, Hq, H, D, bs, W = 2, 4, 2, 16, 4, 6
    kh, kc, ks, table = _empty_tier(B, H, D, bs, W, 4, rng)
    st = dict(k_hot=kh, v_hot=kh.copy(), k_cold=kc, v_cold=kc.copy(), k_scale=ks,
              v_scale=ks.copy(), cold_lens=np.zeros(B, np.int32),
              hot_lens=np.zeros(B, np.int32), hot_starts=np.zeros(B, np.int32))
    n = 11
    tk = rng.standard_normal((n, B, H, D)).astype(np.float16)
    tv = rng.standard_normal((n, B, H, D)).astype(np.float16)
    for i in range(n):
        st, flags = oracle.append_tiered(tk[i], tv[i], st["k_hot"], st["v_hot"], st["k_cold"],
                                         st["v_cold"], st["k_scale"], st["v_scale"], table,
                                         st["cold_lens"], st["hot_lens"], st["hot_starts"],
                                         hot_window=W)
        assert flags == 0
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    out, lse, flags = oracle.decode_tiered(q, st["k_hot"], st["v_hot"], st["k_cold"],
                                           st["v_cold"], st["k_scale"], st["v_scale"], table,
                                           st["cold_lens"], st["hot_lens"], st["hot_starts"],
                                           hot_window=W)
    assert flags == 0
    nd = n - W
    G = Hq // H
    scale = float(np.float32(1 / math.sqrt(D)))
    for b in range(B):
        kd, vd = [], []
        for i in range(n):
            if i < nd:
                rk, rv = [], []
                for h in range(H):
                    c, s = oracle.quantize_row_int8(tk[i, b, h])
                    rk.append(c * float(np.uint16(s).view(np.float16)))
                    c, s = oracle.quantize_row_int8(tv[i, b, h])
                    rv.append(c * float(np.uint16(s).view(np.float16)))
                kd.append(np.array(rk)); vd.append(np.array(rv))
            else:
                kd.append(tk[i, b].astype(np.float64)); vd.append(tv[i, b].astype(np.float64))
        kd, vd = np.array(kd), np.array(vd)
        for h in range(Hq):
            s_ = kd[:, h // G] @ q[b, h].astype(np.float64) * scale
            l_ = logsumexp(s_)
            np.testing.assert_allclose(out[b * Hq + h], np.exp(s_ - l_) @ vd[:, h // G], atol=1e-12)
            assert abs(lse[b * Hq + h] - l_) < 1e-12


def test_append_tiered_inconsistent_state_is_flagged_and_left_unchanged():
    rng = np.random.default_rng(24)
    B, H, D, bs, W = 3, 1, 8, 4, 2
    kh, kc, ks, table = _empty_tier(B, H, D, bs, W, 2, rng)
    table[2, 1] = 999  # out-of-range page for cold position 4..7
    cl = np.array([3, 2, 4], np.int32)
    hl = np.array([2, 2, 2], np.int32)
    hs = np.array([4, 2, 4], np.int32)  # sequence 0: cold_len != hot_start with a full ring
    new = rng.standard_normal((B, H, D)).astype(np.float16)
    st, flags = oracle.append_tiered(new, new, kh, kh, kc, kc, ks, ks, table, cl, hl, hs,
                                     hot_window=W)
    assert flags == oracle.FLAG_BAD_TIER | oracle.FLAG_BAD_BLOCK
    assert (st["cold_lens"] == [3, 3, 4]).all() and (st["hot_starts"] == [4, 3, 4]).all()
    assert (st["hot_lens"] == [2, 2, 2]).all()
    assert not st["k_hot"][0].any() and not st["k_hot"][2].any()  # untouched


def test_append_paged_writes_the_row_and_flags_bad_positions():
    rng = np.random.default_rng(25)
    B, H, D, bs, npg = 3, 2, 8, 4, 2
    NB = B * npg
    table = rng.permutation(NB).reshape(B, npg).astype(np.int32)
    table[1, 1] = -1
    kp = np.zeros((NB, bs, H, D), np.float16)
    new = rng.standard_normal((B, H, D)).astype(np.float16)
    pos = np.array([5, 6, 8], np.int32)  # seq 1: page -1; seq 2: past the table
    k2, v2, flags = oracle.append_paged(new, -new, pos, table, kp, kp)
    assert flags == oracle.FLAG_BAD_BLOCK | oracle.FLAG_BAD_SEQ_LEN
    assert np.array_equal(k2[table[0, 1], 1], new[0]) and np.array_equal(v2[table[0, 1], 1], -new[0])
    assert np.count_nonzero(k2) == np.count_nonzero(new[0])


# ---------------------------------------------------------------------------
# multi-token query decode
# ---------------------------------------------------------------------------

def test_multi_token_rows_equal_single_token_calls_at_their_positions():
    """A T-token call is T single-token decodes: token t of sequence b is
    the one-token decode at position q_pos[b] + t (window and softcap on)."""
    rng = np.random.default_rng(30)
    B, T, Hq, H, D, bs = 3, 5, 8, 2, 16, 4
    lens = np.array([40, 23, 9], np.int32)
    k, v = rand_dense(rng, B, int(lens.max()), H, D)
    kp, vp, table = paged_from_dense(k, v, bs, rng=rng)
    q = rng.standard_normal((B, T, Hq, D)).astype(np.float32)
    base = np.array([30, 18, 2], np.int32)
    multi = oracle.decode_paged(q, kp, vp, table, lens, base, softcap=15.0, sliding_window=11)
    assert multi[2] == 0
    for t in range(T):
        single = oracle.decode_paged(np.ascontiguousarray(q[:, t]), kp, vp, table, lens,
                                     base + t, softcap=15.0, sliding_window=11)
        for b in range(B):
            rows = slice((b * T + t) * Hq, (b * T + t + 1) * Hq)
            assert np.array_equal(multi[0][rows], single[0][b * Hq:(b + 1) * Hq])
            assert np.array_equal(multi[1][rows], single[1][b * Hq:(b + 1) * Hq])


def test_multi_token_default_positions_are_the_last_cached_keys():
    """Without q_pos, token t sits at seq_len - T + t: the last token sees
    every key (the one-token default), token t sees keys 0 .. L-T+t (dense
    causal reference)."""
    from scipy.special import logsumexp
    rng = np.random.default_rng(31)
    B, T, Hq, H, D, bs = 2, 4, 4, 2, 8, 8
    lens = np.array([21, 13], np.int32)
    k, v = rand_dense(rng, B, int(lens.max()), H, D)
    kp, vp, table = paged_from_dense(k, v, bs, rng=rng)
    q = rng.standard_normal((B, T, Hq, D)).astype(np.float32)
    out, lse, flags = oracle.decode_paged(q, kp, vp, table, lens)
    assert flags == 0
    last = oracle.decode_paged(np.ascontiguousarray(q[:, T - 1]), kp, vp, table, lens)
    G = Hq // H
    scale = float(np.float32(1 / math.sqrt(D)))
    for b in range(B):
        rows = slice((b * T + T - 1) * Hq, (b * T + T) * Hq)
        assert np.array_equal(out[rows], last[0][b * Hq:(b + 1) * Hq])
        for t in range(T):
            n = int(lens[b]) - T + t + 1
            for h in range(Hq):
                s = k[b, :n, h // G].astype(np.float64) @ q[b, t, h].astype(np.float64) * scale
                l_ = logsumexp(s)
                r = (b * T + t) * Hq + h
                np.testing.assert_allclose(out[r], np.exp(s - l_) @ v[b, :n, h // G].astype(np.float64),
                                           atol=1e-12)
                assert abs(lse[r] - l_) < 1e-12
