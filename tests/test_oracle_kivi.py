"""Pins of the KIVI-style control arm's oracle (oracle/kivi.c).

The arm is the "Control baseline arm" of "TurboQuant Family Design Study for
CPU and Browser WASM KV Caches" (section 'Candidate key and value
algorithms'): asymmetric quantization of keys per channel and of values per
token, with the fp16 recent window.  Each pin checks the oracle against a
property fixed by that definition, computed here by other means: brute force
over every quantization level, exact reconstruction of constant groups, which
values a key or value group may depend on, hand-packed bits, the byte
accounting, and textbook softmax attention.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
import tq_inputs as ti


class KF:
    def __init__(self, d=128, kb=4, vb=4, P=64, H=2):
        self.head_dim, self.k_bits, self.v_bits, self.page_size, self.num_kv_heads = d, kb, vb, P, H


def _groups(rng):
    """fp16 groups of many shapes: Gaussian, heavy-tailed with outliers,
    all-equal, two-valued, negative-only, tiny, near the fp16 range."""
    out = [rng.standard_normal(64), rng.standard_t(3, 128) * np.where(rng.random(128) < 0.03, 20, 1),
           np.full(40, 1.5), np.where(rng.random(50) < 0.5, -2.0, 3.0), -np.abs(rng.standard_normal(33)) - 4,
           rng.standard_normal(17) * 1e-4, rng.uniform(-6e4, 6e4, 64), np.array([0.0, -0.0, 0.0])]
    return [np.asarray(g, np.float16) for g in out]


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
def test_group_codes_are_the_nearest_level(bits):
    """Each code selects the nearest of the 2^b levels z + s*c (brute force
    over all levels, fp64), except where two levels are equally near; the
    zero is the group minimum and the scale the fp16 value of the level step."""
    rng = np.random.default_rng(bits)
    top = (1 << bits) - 1
    for x in _groups(rng):
        s, z, codes = oracle.kivi_quantize_group(x, bits)
        xf = x.astype(np.float64)
        assert float(z) == xf.min() and not (float(z) == 0.0 and math.copysign(1.0, float(z)) < 0)
        step = min((xf.max() - xf.min()) / top, 65504.0)  # the largest fp16 caps a 1-bit step
        assert abs(float(s) - step) <= 2.0 ** -11 * step * (1 + 1e-6) + 2.0 ** -25
        if float(s) == 0.0:
            assert np.all(codes == 0)
            continue
        levels = float(z) + float(s) * np.arange(top + 1)
        dist = np.abs(xf[:, None] - levels[None, :])
        best = dist.min(1)
        chosen = dist[np.arange(len(xf)), codes]
        # fp32 arithmetic in the oracle: a tie margin of a few fp32 ulps
        assert np.all(chosen <= best + 4e-7 * np.maximum(np.abs(xf), float(s))), (bits, x)
        assert codes.min() >= 0 and codes.max() <= top


def test_constant_group_is_exact():
    for v in (0.0, 1.25, -3.5, 65504.0):
        s, z, codes = oracle.kivi_quantize_group(np.full(9, v, np.float16), 2)
        assert float(s) == 0.0 and float(z) == v and np.all(codes == 0)


def test_tie_goes_up():
    # levels 0, 1, 2, 3 (scale 1): 0.5, 1.5, 2.5 are ties and take the upper level
    s, z, codes = oracle.kivi_quantize_group(np.array([0, 3, 0.5, 1.5, 2.5], np.float16), 2)
    assert float(s) == 1.0 and float(z) == 0.0
    assert codes.tolist() == [0, 3, 1, 2, 3]


def _encode(f, N, seed=0, num_pages=None, layer=0):
    d, H, P = f.head_dim, f.num_kv_heads, f.page_size
    K = ti.kv_history(1, N, H, d, layer, 0, base=seed).numpy()[0]
    V = ti.kv_history(1, N, H, d, layer, 1, base=seed).numpy()[0]
    npg = (N + P - 1) // P
    num_pages = num_pages or npg + 2
    perm = ti.page_permutation(num_pages).numpy()[:npg].astype(np.int32)
    lay = oracle.kivi_layout(f)
    pool = np.full(num_pages * lay["page_bytes"], 0x5A, np.uint8)
    assert oracle.kivi_encode_keys(f, K, perm, pool, num_pages) == 0
    slots = (perm[np.arange(N) // P] * P + np.arange(N) % P).astype(np.int32)
    assert oracle.kivi_encode_values(f, V, slots, pool, num_pages) == 0
    return K, V, perm, slots, pool, num_pages, lay


@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 4), (3, 2)])
def test_key_groups_are_channels_of_a_page(kb, vb):
    """A decoded key channel over one page is a b-bit asymmetric quantization
    of that channel's tokens in that page: its levels are z + s*c with z the
    page-channel minimum, and every token sits at its nearest level."""
    f = KF(128, kb, vb, 32, 2)
    N = 32 * 3 + 11  # three full pages and a partial one
    K, V, perm, slots, pool, npg, lay = _encode(f, N)
    rc, kh = oracle.kivi_decode(f, 0, pool, npg, slots)
    assert rc == 0
    top = (1 << kb) - 1
    for g in range(4):
        rows = np.arange(g * 32, min(N, (g + 1) * 32))
        for h in range(2):
            x = K[rows, h].astype(np.float64)  # [n, d]
            xh = kh[rows, h]
            mn, mx = x.min(0), x.max(0)
            step = (mx - mn) / top
            # reconstruction error at most half a step (plus fp16 rounding of s)
            assert np.all(np.abs(xh - x) <= 0.5 * step * (1 + 2.0 ** -10) + 1e-30), (g, h)
            # the minimum is reproduced exactly
            assert np.array_equal(xh[x.argmin(0), np.arange(128)], mn)


def test_key_group_depends_only_on_its_page_and_channel():
    f = KF(128, 4, 4, 16, 1)
    N = 48
    K, V, perm, slots, pool, npg, lay = _encode(f, N)
    K2 = K.copy()
    K2[20, 0, 5] = np.float16(1000.0)  # page 1, channel 5
    pool2 = np.full_like(pool, 0x5A)
    assert oracle.kivi_encode_keys(f, K2, perm, pool2, npg) == 0
    assert oracle.kivi_encode_values(f, V, slots, pool2, npg) == 0
    rc, a = oracle.kivi_decode(f, 0, pool, npg, slots)
    rc2, b = oracle.kivi_decode(f, 0, pool2, npg, slots)
    changed = np.argwhere(np.any(a != b, axis=2)[:, 0])
    assert set(changed.ravel()) <= set(range(16, 32))  # page 1 only
    per_channel = np.any(a[16:32, 0] != b[16:32, 0], axis=0)
    assert per_channel.tolist() == [j == 5 for j in range(128)]


@pytest.mark.parametrize("vb", [2, 3, 4])
def test_value_groups_are_tokens(vb):
    f = KF(128, 4, vb, 32, 2)
    N = 70
    K, V, perm, slots, pool, npg, lay = _encode(f, N, seed=3)
    rc, vh = oracle.kivi_decode(f, 1, pool, npg, slots)
    assert rc == 0
    top = (1 << vb) - 1
    x = V.astype(np.float64)  # [N, H, d]
    mn, mx = x.min(-1, keepdims=True), x.max(-1, keepdims=True)
    step = (mx - mn) / top
    assert np.all(np.abs(vh - x) <= 0.5 * step * (1 + 2.0 ** -10) + 1e-30)
    assert np.all(vh.min(-1) == x.min(-1))
    # a value token depends on that token alone
    V2 = V.copy()
    V2[7, 1, 3] = np.float16(-900.0)
    pool2 = pool.copy()
    assert oracle.kivi_encode_values(f, V2, slots, pool2, npg) == 0
    rc, vh2 = oracle.kivi_decode(f, 1, pool2, npg, slots)
    changed = np.argwhere(np.any(vh != vh2, axis=2))
    assert changed.tolist() == [[7, 1]]


def test_bitstreams_hand_packed():
    """Keys LSB-first per token; values in the grouped chunk order."""
    f = KF(16, 2, 2, 16, 1)
    # keys: channel j holds j mod 4 in every token but token 0, which holds 0
    # (channel 1: 3), so channel j's group spans [0, j mod 4] (channel 1: [1, 3])
    x = np.zeros((16, 1, 16), np.float16)
    x[1:, 0, :] = np.arange(16)[None, :] % 4
    x[0, 0, 1] = 3
    lay = oracle.kivi_layout(f)
    pool = np.zeros(lay["page_bytes"], np.uint8)
    assert oracle.kivi_encode_keys(f, x, np.array([0], np.int32), pool, 1) == 0
    # token 5 (value j mod 4) by hand: channels 0 mod 4 have a zero range
    # (code 0), channel 1 holds its group minimum 1 (code 0), the others sit at
    # their group's top level (code 3)
    codes = [0 if j % 4 == 0 or j == 1 else 3 for j in range(16)]
    packed = bytes(sum(codes[4 * i + k] << (2 * k) for k in range(4)) for i in range(4))
    assert bytes(pool[lay["k_codes"] + 5 * 4: lay["k_codes"] + 6 * 4]) == packed
    # channel 1 at token 0 holds its maximum 3 (code 3), token 5 holds 1 (code 0)
    assert pool[lay["k_codes"]] & 0b1100 == 0b1100
    # values: token 5 holds 0,1,2,3,0,1,... (levels 0..3, scale 1): chunk 0 of
    # token 5 sits at slot 4*((5%8)//2) + 2*(5//8) + 5%2 = 9 of group 0
    V = np.zeros((16, 1, 16), np.float16)
    V[5, 0, :] = np.array([0, 1, 2, 3] * 4)
    assert oracle.kivi_encode_values(f, V, np.arange(16, dtype=np.int32), pool, 1) == 0
    vc = pool[lay["v_codes"]:lay["v_codes"] + 16 * 4]
    assert bytes(vc[9 * 4:10 * 4]) == bytes([0b11100100] * 4)


def test_layout_bytes():
    for d, kb, vb, P, H in ((128, 4, 4, 64, 8), (128, 2, 2, 64, 8), (128, 2, 2, 128, 8), (64, 3, 2, 32, 2)):
        L = oracle.kivi_layout(KF(d, kb, vb, P, H))
        assert L["k_params"] == 0 and L["k_codes"] == 4 * d
        assert L["v_params"] == L["k_codes"] + -(-P * d * kb // 8 // 16) * 16
        assert L["v_codes"] == L["v_params"] + -(-4 * P // 16) * 16
        assert L["slab_bytes"] == L["v_codes"] + -(-P * d * vb // 8 // 16) * 16
        assert L["page_bytes"] == H * L["slab_bytes"]
    # per token-head at the Llama-3-8B shape: 4-bit K and V, P = 64
    L = oracle.kivi_layout(KF(128, 4, 4, 64, 8))
    assert L["slab_bytes"] / 64 == 512 / 64 + 64 + 4 + 64  # 140 B


def _setup(f, B, Hq, comp, W, wl, seed=0, q_zero=False):
    d, H, P = f.head_dim, f.num_kv_heads, f.page_size
    maxp = max(1, max(-(-c // P) for c in comp))
    num_pages = B * maxp + 2
    perm = ti.page_permutation(num_pages).numpy()
    bt = perm[: B * maxp].reshape(B, maxp).astype(np.int32)
    lay = oracle.kivi_layout(f)
    pool = np.zeros(num_pages * lay["page_bytes"], np.uint8)
    T = max(comp) + max(W, 1)
    K = ti.kv_history(B, T, H, d, 0, 0, base=seed).numpy()
    V = ti.kv_history(B, T, H, d, 0, 1, base=seed).numpy()
    kwin = np.zeros((B, H, max(W, 1), d), np.float16)
    vwin = np.zeros((B, H, max(W, 1), d), np.float16)
    for b in range(B):
        c = comp[b]
        if c:
            npg = -(-c // P)
            assert oracle.kivi_encode_keys(f, K[b, :c], bt[b, :npg], pool, num_pages) == 0
            sl = (bt[b, np.arange(c) // P] * P + np.arange(c) % P).astype(np.int32)
            assert oracle.kivi_encode_values(f, V[b, :c], sl, pool, num_pages) == 0
        kwin[b, :, :wl[b]] = K[b, c:c + wl[b]].transpose(1, 0, 2)
        vwin[b, :, :wl[b]] = V[b, c:c + wl[b]].transpose(1, 0, 2)
    q = np.zeros((B, Hq, d), np.float16) if q_zero else ti.query(B, Hq, d).numpy()
    return dict(q=q, pool=pool, num_pages=num_pages, bt=bt, comp=np.array(comp, np.int32), kwin=kwin if W else None,
                vwin=vwin if W else None, wl=np.array(wl, np.int32), K=K, V=V)


def test_attention_window_only_is_textbook():
    f = KF(128, 2, 2, 32, 2)
    s = _setup(f, 2, 4, [0, 0], 24, [24, 9])
    rc, out = oracle.kivi_attention(f, s["q"], s["pool"], s["num_pages"], s["bt"], s["comp"], s["kwin"], s["vwin"], s["wl"])
    assert rc == 0
    for b in range(2):
        for qh in range(4):
            h = qh // 2
            n = s["wl"][b]
            k = s["kwin"][b, h, :n].astype(np.float64)
            v = s["vwin"][b, h, :n].astype(np.float64)
            p = softmax(k @ s["q"][b, qh].astype(np.float64) / math.sqrt(128))
            np.testing.assert_allclose(out[b, qh], p @ v, rtol=1e-12, atol=1e-12 * np.abs(v).max())


@pytest.mark.parametrize("kb,vb,P", [(4, 4, 64), (2, 2, 32), (2, 3, 16)])
def test_attention_equals_softmax_over_decoded_cache(kb, vb, P):
    """The attention pass on a KIVI cache equals textbook softmax attention
    (scipy) over the cache's own reconstructions plus the raw window."""
    f = KF(128, kb, vb, P, 2)
    comp, W, wl = [3 * P + 5, 70], 16, [16, 4]
    s = _setup(f, 2, 8, comp, W, wl, seed=2)
    rc, out = oracle.kivi_attention(f, s["q"], s["pool"], s["num_pages"], s["bt"], s["comp"], s["kwin"], s["vwin"], s["wl"])
    assert rc == 0
    for b in range(2):
        c = comp[b]
        sl = (s["bt"][b, np.arange(c) // P] * P + np.arange(c) % P).astype(np.int32)
        _, kh = oracle.kivi_decode(f, 0, s["pool"], s["num_pages"], sl)
        _, vh = oracle.kivi_decode(f, 1, s["pool"], s["num_pages"], sl)
        for qh in range(8):
            h = qh // 4
            k = np.concatenate([kh[:, h], s["kwin"][b, h, :wl[b]].astype(np.float64)])
            v = np.concatenate([vh[:, h], s["vwin"][b, h, :wl[b]].astype(np.float64)])
            p = softmax(k @ s["q"][b, qh].astype(np.float64) / math.sqrt(128))
            np.testing.assert_allclose(out[b, qh], p @ v, rtol=1e-11, atol=1e-11 * np.abs(v).max())
    # the head-subset entry point returns the same rows
    rc, sub = oracle.kivi_attention(f, s["q"], s["pool"], s["num_pages"], s["bt"], s["comp"], s["kwin"], s["vwin"], s["wl"],
                                    heads=np.array([15, 0], np.int32))
    np.testing.assert_array_equal(sub[0], out[1, 7])
    np.testing.assert_array_equal(sub[1], out[0, 0])


def test_attention_one_token_and_uniform_logits():
    f = KF(128, 4, 2, 16, 1)
    s = _setup(f, 1, 2, [1], 0, [0])
    rc, out = oracle.kivi_attention(f, s["q"], s["pool"], s["num_pages"], s["bt"], s["comp"], None, None, s["wl"])
    _, vh = oracle.kivi_decode(f, 1, s["pool"], s["num_pages"], np.array([s["bt"][0, 0] * 16], np.int32))
    np.testing.assert_array_equal(out[0, 0], vh[0, 0])
    np.testing.assert_array_equal(out[0, 1], vh[0, 0])
    s = _setup(f, 1, 1, [40], 8, [5], q_zero=True)
    rc, out = oracle.kivi_attention(f, s["q"], s["pool"], s["num_pages"], s["bt"], s["comp"], s["kwin"], s["vwin"], s["wl"])
    sl = (s["bt"][0, np.arange(40) // 16] * 16 + np.arange(40) % 16).astype(np.int32)
    _, vh = oracle.kivi_decode(f, 1, s["pool"], s["num_pages"], sl)
    allv = np.concatenate([vh[:, 0], s["vwin"][0, 0, :5].astype(np.float64)])
    np.testing.assert_allclose(out[0, 0], allv.mean(0), rtol=1e-12, atol=1e-12 * np.abs(allv).max())


def test_out_of_range_page_is_reported():
    f = KF(128, 4, 4, 16, 1)
    s = _setup(f, 1, 1, [32], 0, [0])
    bt = s["bt"].copy()
    bt[0, 1] = s["num_pages"] + 3
    rc, out = oracle.kivi_attention(f, s["q"], s["pool"], s["num_pages"], bt, s["comp"], None, None, s["wl"])
    assert rc == -2
    rc2, ref = oracle.kivi_attention(f, s["q"], s["pool"], s["num_pages"], s["bt"], np.array([16], np.int32), None, None, s["wl"])
    np.testing.assert_allclose(out, ref, rtol=1e-13)
