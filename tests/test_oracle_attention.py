"""Pins of the oracle's page layout (byte accounting) and decode attention.

Bytes: the capacity formulas of "TurboQuant Family Design Study ...", sections
'Capacity model' and 'Packed format and complete bit accounting', and the
aither-kvcache README tables 'Compression Ratios' and 'KV Cache Memory by
Model / by Context Length'.

Attention: logits q.k/sqrt(d), softmax, o = sum p_i v_i ('Why keys and values
need different treatment'); the oracle materializes every token and takes the
exact softmax.  It is pinned against (1) textbook softmax attention when only
the fp16 window is present, (2) one-token and uniform-logit special cases, and
(3) the rotated-domain computation of the README's 'Zero-buffer fused
attention' (rotate q once, score packed codes through the centroids plus the
QJL correction, accumulate values in the rotated domain, rotate back once),
written here in numpy directly from the packed bytes.
"""
import math

import numpy as np
import pytest
from scipy.linalg import hadamard
from scipy.special import softmax

import oracle
import tq_inputs as ti
from tq_testlib import value_codes


# ---------------------------------------------------------------- bytes ----
@pytest.mark.parametrize(
    "fmt,page_bytes",
    [
        (ti.Format(128, 4, 4, 0, 128, 64, 8), 69632),
        (ti.Format(128, 3, 4, 1, 128, 64, 2), 17920),
        (ti.Format(128, 2, 2, 1, 128, 128, 8), 94208),
    ],
)
def test_page_bytes_of_the_workload_formats(fmt, page_bytes):
    L = oracle.page_layout(fmt)
    assert L["page_bytes"] == page_bytes
    for k in ("k_norm", "k_gamma", "k_codes", "k_signs", "v_norm", "v_codes", "slab_bytes"):
        assert L[k] % 16 == 0
    P = fmt.page_size
    # per token-head payload = norms + codes (+ gamma + signs for QJL keys)
    per_tok = 4 + 16 * fmt.k_bits + 4 + 16 * fmt.v_bits + (4 + fmt.qjl_m // 8 if fmt.k_qjl else 0)
    assert L["slab_bytes"] == P * per_tok  # no padding needed at these sizes


def test_bytes_per_vector_and_ratios(golden):
    g = golden("compression_ratios.json")
    for b in (2, 3, 4):
        L = oracle.page_layout(ti.Format(128, b, b, 0, 128, 64, 1))
        per_vec = 4 + L["k_code_bytes"]  # fp32 norm + packed codes
        assert per_vec == g["bytes_per_vector"][str(b)]
        assert round(256 / per_vec, 1) == g["vs_fp16"][str(b)]


def test_kv_memory_tables(golden):
    g = golden("kv_memory_llama31_8b.json")
    Lyr, H, d = g["model"]["layers"], g["model"]["kv_heads"], g["model"]["head_dim"]
    GiB, MiB = 2.0 ** 30, 2.0 ** 20

    def tq_bytes(b, T):
        lay = oracle.page_layout(ti.Format(d, b, b, 0, 128, 64, H))
        per_tok = lay["page_bytes"] / 64  # all heads, K and V
        return Lyr * T * per_tok

    fp16 = lambda T: 2 * Lyr * H * d * 2 * T  # bytes per token = 2 L Hkv d s, s = 2
    assert fp16(32768) / GiB == g["at_32k_gib"]["fp16"]
    for name, b in (("tq4", 4), ("tq3", 3), ("tq2", 2)):
        assert round(tq_bytes(b, 32768) / GiB, 1) == g["at_32k_gib"][name]
        assert tq_bytes(b, 8192) / MiB == g["by_context"]["8192"][name + "_mib"]
        # the README rounds half up (2.25 -> 2.3)
        assert math.floor(tq_bytes(b, 131072) / GiB * 10 + 0.5) / 10 == g["by_context"]["131072"][name + "_gib"]
    assert fp16(8192) / GiB == g["by_context"]["8192"]["fp16_gib"]
    assert fp16(131072) / GiB == g["by_context"]["131072"]["fp16_gib"]


def test_capacity_formulas(golden):
    g = golden("formulas.json")
    r = g["rmem"]
    assert round(4 / ((r["b_k"] + r["b_v"]) / 8), 2) == r["value"]
    a = g["all_in_bits"]
    L = oracle.page_layout(ti.Format(a["d"], a["b_nominal"], a["b_nominal"], 0, 128, 64, 1))
    assert (4 + L["k_code_bytes"]) * 8 / a["d"] == a["value"] == a["b_nominal"] + a["b_norm"] / a["d"]
    # M(T) with a W-token fp16 window: payload bits + fp16 window, plus the
    # fp32 norms this format stores (the formula counts payload only)
    Lyr, H, d, T, W, bk, bv = 32, 8, 128, 32768, 128, 4, 4
    lay = oracle.page_layout(ti.Format(d, bk, bv, 0, 128, 64, H))
    stored = Lyr * (T - W) * lay["page_bytes"] / 64 + Lyr * H * d * W * 4
    formula = Lyr * H * d * ((T - W) * (bk + bv) / 8 + W * 4)
    assert stored - formula == Lyr * H * (T - W) * 8


# ------------------------------------------------------------ attention ----
def _setup(fmt, B, Hq, comp_lens, W, win_lens, seed=0, q_zero=False):
    """Encode synthetic K/V with the oracle into permuted pages."""
    d, H, P = fmt.head_dim, fmt.num_kv_heads, fmt.page_size
    max_pages = max(1, max((c + P - 1) // P for c in comp_lens))
    num_pages = B * max_pages + 3
    perm = ti.page_permutation(num_pages, seed=7).numpy()
    bt = perm[: B * max_pages].reshape(B, max_pages).astype(np.int32)
    lay = oracle.page_layout(fmt)
    pool = np.zeros(num_pages * lay["page_bytes"], np.uint8)
    T = max(comp_lens) + W
    K = ti.kv_history(B, max(T, 1), H, d, layer=seed, kind=0).numpy()
    V = ti.kv_history(B, max(T, 1), H, d, layer=seed, kind=1).numpy()
    ks, vs = ti.sign_bits(ti.SEED_SIGNS_K, d), ti.sign_bits(ti.SEED_SIGNS_V, d)
    kc, kt = oracle.kind_codebook(fmt, 0)  # mixed keys: both widths' codebooks
    vc, vt = oracle.kind_codebook(fmt, 1)
    S = ti.gaussian_matrix(ti.SEED_QJL, fmt.qjl_m, d) if fmt.k_qjl else None
    kwin = np.zeros((B, H, max(W, 1), d), np.float16)
    vwin = np.zeros((B, H, max(W, 1), d), np.float16)
    for b in range(B):
        c = comp_lens[b]
        slots = np.array([bt[b, i // P] * P + i % P for i in range(c)], np.int32)
        if c:
            assert oracle.encode(fmt, 0, K[b, :c], slots, pool, num_pages, ks, kc, kt, S) == 0
            assert oracle.encode(fmt, 1, V[b, :c], slots, pool, num_pages, vs, vc, vt) == 0
        wl = win_lens[b] if W else 0
        kwin[b, :, :wl] = K[b, c:c + wl].transpose(1, 0, 2)
        vwin[b, :, :wl] = V[b, c:c + wl].transpose(1, 0, 2)
    q = ti.query(B, Hq, d).numpy()
    if q_zero:
        q[:] = 0
    return dict(q=q, pool=pool, num_pages=num_pages, bt=bt, comp=np.array(comp_lens, np.int32), kwin=kwin if W else None,
                vwin=vwin if W else None, wl=np.array(win_lens, np.int32), ks=ks, vs=vs, kc=kc, vc=vc, S=S, lay=lay, K=K, V=V)


def _run(fmt, s, heads=None):
    return oracle.attention(fmt, s["q"], s["pool"], s["num_pages"], s["bt"], s["comp"], s["kwin"], s["vwin"], s["wl"], s["ks"],
                            s["vs"], s["kc"], s["vc"], s["S"], heads=heads)


def test_window_only_equals_textbook_attention():
    fmt = ti.Format(128, 4, 4, 0, 128, 64, 2)
    B, Hq, W = 2, 4, 24
    s = _setup(fmt, B, Hq, [0, 0], W, [24, 17])
    rc, out = _run(fmt, s)
    assert rc == 0
    for b in range(B):
        for qh in range(Hq):
            h = qh // 2
            n = s["wl"][b]
            k = s["kwin"][b, h, :n].astype(np.float64)
            v = s["vwin"][b, h, :n].astype(np.float64)
            q = s["q"][b, qh].astype(np.float64)
            want = softmax(k @ q / math.sqrt(128)) @ v
            np.testing.assert_allclose(out[b, qh], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_single_token_and_uniform_logits():
    fmt = ti.Format(128, 3, 2, 1, 128, 64, 1)
    s = _setup(fmt, 1, 2, [1], 0, [0])
    rc, out = _run(fmt, s)
    rc2, vh = oracle.decode(fmt, 1, s["pool"], s["num_pages"], np.array([s["bt"][0, 0] * 64], np.int32), s["vs"], s["vc"])
    assert rc == 0 and rc2 == 0
    np.testing.assert_allclose(out[0, 0], vh[0, 0], rtol=1e-14, atol=1e-14 * np.abs(vh).max())
    np.testing.assert_allclose(out[0, 1], vh[0, 0], rtol=1e-14, atol=1e-14 * np.abs(vh).max())
    # q = 0: every logit is 0, the output is the plain mean of the values
    s = _setup(fmt, 1, 1, [70], 8, [5], q_zero=True)
    rc, out = _run(fmt, s)
    slots = np.array([s["bt"][0, i // 64] * 64 + i % 64 for i in range(70)], np.int32)
    _, vh = oracle.decode(fmt, 1, s["pool"], s["num_pages"], slots, s["vs"], s["vc"])
    allv = np.concatenate([vh[:, 0], s["vwin"][0, 0, :5].astype(np.float64)])
    np.testing.assert_allclose(out[0, 0], allv.mean(0), rtol=1e-12, atol=1e-12 * np.abs(allv).max())


def _unpack(buf, nbits, count):
    bits = np.unpackbits(buf, bitorder="little")[: nbits * count].reshape(count, nbits)
    return (bits * (1 << np.arange(nbits))).sum(1)


def _key_centroids(fmt, raw, d):
    """Centroid of each channel of one key, from its code stream: uniform
    keys at k_bits per channel; mixed keys with the channels j mod 16 < 8 at
    k_bits + 1 bits first, then the others at k_bits (LSB-first)."""
    if not fmt.k_mixed:
        kc, _ = oracle.make_codebook(fmt.k_bits)
        return kc.astype(np.float64)[_unpack(raw, fmt.k_bits, d)]
    hi = (np.arange(d) % 16) < 8
    bh, bl, nh = fmt.k_bits + 1, fmt.k_bits, int(hi.sum())
    bits = np.unpackbits(raw, bitorder="little")
    ih = (bits[: nh * bh].reshape(nh, bh) * (1 << np.arange(bh))).sum(1)
    il = (bits[nh * bh: nh * bh + (d - nh) * bl].reshape(d - nh, bl) * (1 << np.arange(bl))).sum(1)
    out = np.empty(d)
    out[hi] = oracle.make_codebook(bh)[0].astype(np.float64)[ih]
    out[~hi] = oracle.make_codebook(bl)[0].astype(np.float64)[il]
    return out


def _rotated_domain_attention(fmt, s, b, qh):
    """The README's fused form, from raw bytes: rotate q once, score codes via
    centroids (+ QJL term), weight values in the rotated domain, rotate back."""
    d, H, P, m = fmt.head_dim, fmt.num_kv_heads, fmt.page_size, fmt.qjl_m
    G = s["q"].shape[1] // H
    h = qh // G
    L = s["lay"]
    Hm = hadamard(d).astype(np.float64)
    Dk = np.where(s["ks"] == 1, -1.0, 1.0)
    Dv = np.where(s["vs"] == 1, -1.0, 1.0)
    q = s["q"][b, qh].astype(np.float64)
    q_rot = Hm @ (Dk * q) / math.sqrt(d)
    if fmt.k_qjl:
        q_s = s["S"].astype(np.float64) @ q_rot
    logits, vrot = [], []
    for i in range(s["comp"][b]):
        pg = s["bt"][b, i // P]
        off = i % P
        slab = s["pool"][pg * L["page_bytes"] + h * L["slab_bytes"]:][: L["slab_bytes"]]
        nk = slab[L["k_norm"] + 4 * off:][:4].view(np.float32)[0]
        cent = _key_centroids(fmt, slab[L["k_codes"] + off * L["k_code_bytes"]:][: L["k_code_bytes"]], d)
        score = q_rot @ cent / math.sqrt(d)
        if fmt.k_qjl:
            gam = slab[L["k_gamma"] + 4 * off:][:4].view(np.float32)[0]
            z = _unpack(slab[L["k_signs"] + off * L["k_sign_bytes"]:][: L["k_sign_bytes"]], 1, m)
            # the format's coefficient: qjl_scale when given, else sqrt(pi/2) / m
            # (the format field is an fp32 value)
            coef = float(np.float32(fmt.qjl_scale)) if fmt.qjl_scale > 0 else math.sqrt(math.pi / 2) / m
            score += coef * float(gam) * (q_s @ (2.0 * z - 1.0))
        logits.append(float(nk) * score / math.sqrt(d))
        nv = slab[L["v_norm"] + 4 * off:][:4].view(np.float32)[0]
        vidx = value_codes(slab[L["v_codes"]:][: P * L["v_code_bytes"]], off, d, fmt.v_bits)
        vrot.append(float(nv) * s["vc"].astype(np.float64)[vidx] / math.sqrt(d))
    nw = s["wl"][b] if s["kwin"] is not None else 0
    kw = s["kwin"][b, h, :nw].astype(np.float64) if nw else np.zeros((0, d))
    vw = s["vwin"][b, h, :nw].astype(np.float64) if nw else np.zeros((0, d))
    lw = list(kw @ q / math.sqrt(d))
    p = softmax(np.array(logits + lw))
    pc, pw = p[: len(logits)], p[len(logits):]
    acc_rot = pc @ np.array(vrot).reshape(-1, d) if logits else np.zeros(d)
    return Dv * (Hm @ acc_rot) / math.sqrt(d) + pw @ vw  # rotate back once


@pytest.mark.parametrize(
    "fmt,B,Hq,comp,W,wl",
    [
        (ti.Format(128, 4, 4, 0, 128, 64, 2), 2, 8, [130, 64], 0, [0, 0]),
        (ti.Format(128, 3, 4, 1, 128, 64, 1), 1, 4, [200], 16, [16]),
        (ti.Format(128, 2, 2, 1, 128, 32, 2), 2, 4, [33, 95], 8, [8, 3]),
        # mixed-rate keys (3.5 and 2.5 bits), one with a given QJL scale
        (ti.Format(128, 3, 4, 0, 128, 64, 2, k_mixed=1), 2, 8, [150, 40], 8, [8, 2]),
        (ti.Format(128, 2, 3, 1, 128, 32, 1, k_mixed=1, qjl_scale=0.05), 1, 4, [90], 0, [0]),
        # norm-corrected keys and values (the stored norms are n / ||y_hat||)
        (ti.Format(128, 4, 3, 0, 128, 64, 2, norm_correct=1), 1, 4, [77], 4, [4]),
    ],
)
def test_materialized_equals_rotated_domain(fmt, B, Hq, comp, W, wl):
    s = _setup(fmt, B, Hq, comp, W, wl, seed=1)
    rc, out = _run(fmt, s)
    assert rc == 0
    for b in range(B):
        for qh in range(Hq):
            want = _rotated_domain_attention(fmt, s, b, qh)
            np.testing.assert_allclose(out[b, qh], want, rtol=0, atol=1e-10 * np.abs(want).max())
    # the head-subset entry point returns the same rows
    heads = np.array([Hq * (B - 1) + Hq - 1, 0], np.int32)
    rc, sub = _run(fmt, s, heads=heads)
    np.testing.assert_array_equal(sub[0], out[B - 1, Hq - 1])
    np.testing.assert_array_equal(sub[1], out[0, 0])


def test_out_of_range_page_is_skipped_and_reported():
    fmt = ti.Format(128, 4, 4, 0, 128, 64, 1)
    s = _setup(fmt, 1, 1, [128], 0, [0])
    good = _run(fmt, s)[1]
    s_bad = dict(s)
    bt = s["bt"].copy()
    bt[0, 1] = s["num_pages"] + 5
    s_bad["bt"] = bt
    rc, out = _run(fmt, s_bad)
    assert rc == -2
    s_short = dict(s)
    s_short["comp"] = np.array([64], np.int32)  # only the valid first page
    np.testing.assert_allclose(out, _run(fmt, s_short)[1], rtol=1e-13, atol=1e-13)
    assert not np.allclose(out, good)
