"""Pins of the oracle's mixed-channel (fractional) key rates.

"TurboQuant Family Design Study for CPU and Browser WASM KV Caches", section
'Packed format and complete bit accounting': 3.5 bits per channel are 64
channels packed at 4 bits and 64 at 3 bits, 2.5 bits are 64 at 3 and 64 at 2,
exact rates with fixed offsets.  The page leaves open which channels take the
extra bit; the oracle (and the GPU path) give it to channel j when
(j mod 16) < 8 and store the high channels' codes first.

Checks: the per-channel widths and the packed stream against numpy (scipy's
Hadamard matrix, searchsorted on the thresholds, hand-packed bits) on tiny
vectors; the reconstruction MSE against the mean of the two widths' validated
MSE values the aither-kvcache README prints; the bit accounting.
"""
import numpy as np
import pytest
from scipy.linalg import hadamard

import oracle
import tq_inputs as ti


def _high(d):
    return (np.arange(d) % 16) < 8


@pytest.mark.parametrize("b", [2, 3])
def test_mixed_codes_per_channel_and_stream(b):
    d = 16
    fmt = ti.Format(d, b, b, 0, 8, 16, 1, k_mixed=1)
    lay = oracle.page_layout(fmt)
    assert lay["k_code_bytes"] == (d // 2) * (2 * b + 1) // 8
    ch, th = oracle.make_codebook(b + 1)
    cl, tl = oracle.make_codebook(b)
    signs = (np.arange(d) * 7 % 3 == 0).astype(np.uint8)
    rng = np.random.default_rng(b)
    x = rng.standard_normal((5, 1, d)).astype(np.float16)
    pool = np.zeros(lay["page_bytes"], np.uint8)
    slots = np.arange(5, dtype=np.int32)
    assert oracle.encode(fmt, 0, x, slots, pool, 1, signs, *oracle.kind_codebook(fmt, 0)) == 0
    H = hadamard(d).astype(np.float64)
    D = np.where(signs == 1, -1.0, 1.0)
    hi = _high(d)
    for n in range(5):
        xv = x[n, 0].astype(np.float64)
        u = H @ (D * xv) / np.linalg.norm(xv)
        idx = np.where(hi, np.searchsorted(th, u, side="right"), np.searchsorted(tl, u, side="right"))
        # hand-packed stream: high channels at b+1 bits, then low channels at b bits, LSB-first
        bits = [(int(v) >> i) & 1 for v in idx[hi] for i in range(b + 1)]
        bits += [(int(v) >> i) & 1 for v in idx[~hi] for i in range(b)]
        want = np.packbits(np.array(bits, np.uint8), bitorder="little")
        got = pool[lay["k_codes"] + n * lay["k_code_bytes"]: lay["k_codes"] + (n + 1) * lay["k_code_bytes"]]
        np.testing.assert_array_equal(got, want)
        # decode uses each channel's own codebook
        rc, out = oracle.decode(fmt, 0, pool, 1, slots[n:n + 1], signs, oracle.kind_codebook(fmt, 0)[0])
        assert rc == 0
        y = np.array([ch[i] if h else cl[i] for i, h in zip(idx, hi)]) / np.sqrt(d)
        np.testing.assert_allclose(out[0, 0], np.linalg.norm(xv) * D * (H @ y) / np.sqrt(d), rtol=0, atol=1e-5)


@pytest.mark.parametrize("b", [2, 3])
def test_mixed_mse_is_the_mean_of_the_two_widths(golden, b):
    g = golden("validated_mse.json")["mse"]
    want = 0.5 * (g[str(b + 1)] + g[str(b)])  # 0.0220 at 3.5 bits, 0.0760 at 2.5
    d = 128
    ch, th = oracle.make_codebook(b + 1)
    cl, tl = oracle.make_codebook(b)
    signs = ti.sign_bits(ti.SEED_SIGNS_K, d)
    rng = np.random.default_rng(10 + b)
    hi = _high(d)
    err = 0.0
    n_vec = 1500
    for _ in range(n_vec):
        x = rng.standard_normal(d)
        x /= np.linalg.norm(x)
        e = oracle.encode_vector(x, b + 1, signs, ch, th, lo_codebook=(cl, tl))
        xr = oracle.decode_vector(e["norm"], e["idx"], b + 1, signs, ch, lo_centroids=cl)
        sq = ((x - xr) ** 2).sum()
        err += sq
        # paired identity: the error is that of the (b+1)-bit quantizer on the
        # high channels plus the b-bit one on the low channels (rotated domain)
        eh = oracle.encode_vector(x, b + 1, signs, ch, th)
        el = oracle.encode_vector(x, b, signs, cl, tl)
        u = eh["u"]
        split = (((u - ch[eh["idx"]]) ** 2)[hi].sum() + ((u - cl[el["idx"]]) ** 2)[~hi].sum()) / d
        assert abs(sq - split) <= 1e-9 * max(sq, 1e-12)
    mse = err / n_vec
    # the pages' values are rounded and measured on their own vectors: 5 %
    assert abs(mse - want) / want < 0.05, (b, mse, want)
    # strictly between the two uniform rates
    assert g[str(b + 1)] < mse < g[str(b)]


def test_mixed_bit_accounting():
    for b, rate in ((3, 3.5), (2, 2.5)):
        lay = oracle.page_layout(ti.Format(128, b, 4, 0, 128, 64, 8, k_mixed=1))
        assert lay["k_code_bytes"] * 8 / 128 == rate
        # one K code stream per token-head: 56 B at 3.5 bits, 40 B at 2.5, plus the fp32 norm
        assert lay["k_code_bytes"] == {3: 56, 2: 40}[b]
    with pytest.raises(Exception):
        oracle.page_layout(ti.Format(128, 8, 4, 0, 128, 64, 8, k_mixed=1))  # 9-bit high channels
