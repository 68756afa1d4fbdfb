"""GPU KV append (paged, tiered int8 with demotion, tiered f16) against the
oracle: every buffer and every tier length must match bit for bit, the
int8 codes and f16 scales included (both sides take the quantizer's
decisions in f32 with IEEE division, ties to even)."""
import numpy as np
import pytest

import oracle
import quantized_kv_decode_paged_gb300 as qk
from parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield
    import torch
    torch.cuda.empty_cache()


def _dev(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to("cuda")


def _host(t, dtype):
    return t.cpu().numpy().view(dtype)


def _status():
    import torch
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _rand_rows(rng, shape, kind):
    """f16 rows of a few kinds: normal, wide range, tiny (subnormal scales),
    exact ties of the quantizer, all zero."""
    x = rng.standard_normal(shape).astype(np.float32)
    if kind == "wide":
        x *= np.float32(2000.0)
    elif kind == "tiny":
        x *= np.float32(3e-6)
    elif kind == "ties":
        # max 127 -> scale 1.0, so every half-integer is a tie
        x = (rng.integers(-254, 255, size=shape) / 2.0).astype(np.float32)
        x[..., 0] = 127.0
    elif kind == "zero":
        x[:] = 0
    return x.astype(np.float16)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_append_paged_matches_oracle(D):
    rng = np.random.default_rng(300 + D)
    B, H, bs, npg = 6, 2, 16, 4
    NB = B * npg + 3
    table = rng.permutation(NB)[: B * npg].reshape(B, npg).astype(np.int32)
    table[4, 2] = NB + 5  # bad page
    pos = np.array([0, 17, 63, 30, 40, 64], np.int32)  # seq 5 is past the table
    kp = rng.standard_normal((NB, bs, H, D)).astype(np.float16)
    vp = rng.standard_normal((NB, bs, H, D)).astype(np.float16)
    kn = rng.standard_normal((B, H, D)).astype(np.float16)
    vn = rng.standard_normal((B, H, D)).astype(np.float16)
    ref_k, ref_v, flags = oracle.append_paged(kn, vn, pos, table, kp, vp)
    assert flags == oracle.FLAG_BAD_BLOCK | oracle.FLAG_BAD_SEQ_LEN
    tk, tv, st = _dev(kp), _dev(vp), _status()
    qk.decode_attn_append_paged(_dev(kn), _dev(vn), _dev(pos), _dev(table), tk, tv, dev_status=st)
    assert int(st.item()) == qk.DEV_BAD_BLOCK | qk.DEV_BAD_SEQ_LEN
    assert np.array_equal(_host(tk, np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(_host(tv, np.uint16), ref_v.view(np.uint16))


def _tier_state(rng, B, H, D, bs, W, npg, f16):
    NB = B * npg
    table = rng.permutation(NB).reshape(B, npg).astype(np.int32)
    kh = rng.standard_normal((B, W + 2, H, D)).astype(np.float16)  # capacity W + 2
    vh = rng.standard_normal((B, W + 2, H, D)).astype(np.float16)
    if f16:
        kc = rng.standard_normal((NB, bs, H, D)).astype(np.float16)
        vc = rng.standard_normal((NB, bs, H, D)).astype(np.float16)
        ks = vs = None
    else:
        kc = rng.integers(0, 2 ** 32, size=(NB, bs, H, D // 4), dtype=np.uint64).astype(np.uint32)
        vc = rng.integers(0, 2 ** 32, size=(NB, bs, H, D // 4), dtype=np.uint64).astype(np.uint32)
        ks = rng.random((NB, bs, H)).astype(np.float16)
        vs = rng.random((NB, bs, H)).astype(np.float16)
    return dict(k_hot=kh, v_hot=vh, k_cold=kc, v_cold=vc, k_scale=ks, v_scale=vs), table


def _gpu_append(st, table, kn, vn, W, f16, status):
    d = {k: (None if v is None else _dev(v)) for k, v in st.items()}
    if f16:
        qk.decode_attn_append_tiered_f16(_dev(kn), _dev(vn), d["k_hot"], d["v_hot"], d["k_cold"],
                                         d["v_cold"], _dev(table), d["cold_lens"], d["hot_lens"],
                                         d["hot_starts"], hot_window=W, dev_status=status)
    else:
        qk.decode_attn_append_tiered_int8(_dev(kn), _dev(vn), d["k_hot"], d["v_hot"], d["k_cold"],
                                          d["v_cold"], d["k_scale"], d["v_scale"], _dev(table),
                                          d["cold_lens"], d["hot_lens"], d["hot_starts"],
                                          hot_window=W, dev_status=status)
    out = {}
    for k, v in d.items():
        if v is None:
            out[k] = None
        elif k in ("k_cold", "v_cold") and not f16:
            out[k] = _host(v, np.uint32)
        elif v.dtype == __import__("torch").float16:
            out[k] = _host(v, np.uint16)
        else:
            out[k] = v.cpu().numpy()
    return out


def _compare(gpu, ref, f16):
    for k in ("k_hot", "v_hot", "k_cold", "v_cold", "k_scale", "v_scale"):
        if ref.get(k) is None:
            continue
        r = ref[k].view(np.uint32 if (k in ("k_cold", "v_cold") and not f16) else np.uint16)
        g = gpu[k]
        bad = np.argwhere(g != r)
        assert bad.size == 0, (k, bad[:5])
    for k in ("cold_lens", "hot_lens", "hot_starts"):
        assert np.array_equal(gpu[k], ref[k]), (k, gpu[k], ref[k])


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("D,H", [(64, 1), (128, 2), (128, 8), (256, 2)])
def test_append_tiered_one_step_matches_oracle(f16, D, H):
    rng = np.random.default_rng(310 + D + H + f16)
    B, bs, W, npg = 9, 8, 6, 5
    st, table = _tier_state(rng, B, H, D, bs, W, npg, f16)
    # per sequence: (cold_len, hot_len, hot_start) covering empty, partial,
    # full rings, a page boundary, and the flagged cases
    cl = np.array([0, 5, 8, 15, 7, 3, 39, 40, 2], np.int32)
    hl = np.array([0, 3, 6, 6, 6, 7, 6, 6, 6], np.int32)
    hs = np.array([0, 5, 8, 15, 7, 3, 39, 40, 9], np.int32)
    table[4, 0] = -7  # seq 4: cold page 0 is bad -> flag 1, unchanged
    # seq 5: hot_len > W -> flag 16; seq 7: cold position 40 is past 5 pages of 8 -> flag 2;
    # seq 8: cold_len != hot_start with a full ring -> flag 16
    st.update(cold_lens=cl, hot_lens=hl, hot_starts=hs)
    kinds = ["normal", "wide", "tiny", "ties", "zero"]
    kn = np.stack([_rand_rows(rng, (H, D), kinds[b % 5]) for b in range(B)])
    vn = np.stack([_rand_rows(rng, (H, D), kinds[(b + 2) % 5]) for b in range(B)])
    # the hot rows that get demoted carry the same special kinds
    for b in range(B):
        slot = int(hs[b]) % W
        st["k_hot"][b, slot] = _rand_rows(rng, (H, D), kinds[(b + 1) % 5])
        st["v_hot"][b, slot] = _rand_rows(rng, (H, D), kinds[(b + 3) % 5])
    ref, flags = oracle.append_tiered(kn, vn, st["k_hot"], st["v_hot"], st["k_cold"],
                                      st["v_cold"], st["k_scale"], st["v_scale"], table, cl, hl,
                                      hs, hot_window=W)
    assert flags == oracle.FLAG_BAD_BLOCK | oracle.FLAG_BAD_TIER | oracle.FLAG_BAD_SEQ_LEN
    status = _status()
    gpu = _gpu_append(st, table, kn, vn, W, f16, status)
    assert int(status.item()) == qk.DEV_BAD_BLOCK | qk.DEV_BAD_TIER | qk.DEV_BAD_SEQ_LEN
    _compare(gpu, ref, f16)


@pytest.mark.parametrize("f16", [False, True])
def test_append_tiered_many_steps_then_decode(f16):
    """Twenty appends on the GPU (demoting from the sixth on) leave the same
    cache as the oracle's, and decoding that cache matches the oracle's
    decode of its own cache."""
    import torch
    rng = np.random.default_rng(330 + f16)
    B, Hq, H, D, bs, W, npg = 3, 8, 2, 128, 16, 5, 4
    st, table = _tier_state(rng, B, H, D, bs, W, npg, f16)
    cl = np.array([0, 16, 30], np.int32)
    hl = np.array([0, 2, 5], np.int32)
    hs = cl.copy()
    ref = dict(st, cold_lens=cl, hot_lens=hl, hot_starts=hs)
    dev = {k: (None if v is None else _dev(v)) for k, v in ref.items()}
    tbl = _dev(table)
    status = _status()
    for i in range(20):
        kn = rng.standard_normal((B, H, D)).astype(np.float16)
        vn = rng.standard_normal((B, H, D)).astype(np.float16)
        ref, flags = oracle.append_tiered(kn, vn, ref["k_hot"], ref["v_hot"], ref["k_cold"],
                                          ref["v_cold"], ref.get("k_scale"), ref.get("v_scale"),
                                          table, ref["cold_lens"], ref["hot_lens"],
                                          ref["hot_starts"], hot_window=W)
        assert flags == 0
        args = (_dev(kn), _dev(vn), dev["k_hot"], dev["v_hot"], dev["k_cold"], dev["v_cold"])
        tail = (tbl, dev["cold_lens"], dev["hot_lens"], dev["hot_starts"])
        if f16:
            qk.decode_attn_append_tiered_f16(*args, *tail, hot_window=W, dev_status=status)
        else:
            qk.decode_attn_append_tiered_int8(*args, dev["k_scale"], dev["v_scale"], *tail,
                                              hot_window=W, dev_status=status)
    assert int(status.item()) == 0
    assert np.array_equal(dev["cold_lens"].cpu().numpy(), ref["cold_lens"])
    assert np.array_equal(dev["hot_starts"].cpu().numpy(), ref["hot_starts"])
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    kw = dict(hot_window=W, cold_lens=dev["cold_lens"], hot_lens=dev["hot_lens"],
              hot_starts=dev["hot_starts"], max_seq_len=int((ref["cold_lens"] + ref["hot_lens"]).max()))
    if f16:
        out, lse = qk.decode_attn_tiered_f16(_dev(q), dev["k_hot"], dev["v_hot"], dev["k_cold"],
                                             dev["v_cold"], tbl, **kw)
        r_out, r_lse, fl = oracle.decode_tiered_f16(q, ref["k_hot"], ref["v_hot"], ref["k_cold"],
                                                    ref["v_cold"], table, ref["cold_lens"],
                                                    ref["hot_lens"], ref["hot_starts"],
                                                    hot_window=W)
    else:
        out, lse = qk.decode_attn_tiered_int8(_dev(q), dev["k_hot"], dev["v_hot"], dev["k_cold"],
                                              dev["v_cold"], dev["k_scale"], dev["v_scale"], tbl,
                                              **kw)
        r_out, r_lse, fl = oracle.decode_tiered(q, ref["k_hot"], ref["v_hot"], ref["k_cold"],
                                                ref["v_cold"], ref["k_scale"], ref["v_scale"],
                                                table, ref["cold_lens"], ref["hot_lens"],
                                                ref["hot_starts"], hot_window=W)
    torch.cuda.synchronize()
    assert fl == 0
    assert_parity(out.cpu().numpy().reshape(-1, D), lse.cpu().numpy().reshape(-1), r_out, r_lse,
                  "append+decode")
