"""Pins of the oracle's rotation, encode/decode, bit packing and QJL sketch.

Rotation: the structured transform (Rademacher signs, then a Walsh-Hadamard
transform) of "TurboQuant Family Design Study ...", section 'Dense and
structured transform comparison', and the identity q.k = (Tq).(Tk) of section
'Placement relative to RoPE and attention'.  Encode/decode: the steps of the
aither-kvcache README, section 'Algorithm'.  QJL: Gaussian S with scale
sqrt(pi/2)/d, unbiased for inner products ("From 0% to 100%...", section 'The
QJL detective story').  Each check compares the oracle with something it does
not share code with: scipy's Sylvester Hadamard matrix, brute force over all
code vectors, hand-packed bit strings, dense numpy formulas, or a statistical
property over many seeds.
"""
import itertools
import math

import numpy as np
import pytest
from scipy.linalg import hadamard

import oracle
import tq_inputs as ti


def _dsign(signs):
    return np.where(np.asarray(signs) == 1, -1.0, 1.0)


@pytest.mark.parametrize("d", [2, 4, 8, 16, 32, 64, 128])
def test_fwht_is_sylvester_hadamard(d):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((5, d))
    H = hadamard(d).astype(np.float64)
    for row in x:
        np.testing.assert_allclose(oracle.fwht(row), H @ row, rtol=0, atol=1e-12 * np.abs(row).sum())
    # involution up to scale: H H = d I
    np.testing.assert_allclose(oracle.fwht(oracle.fwht(x[0])), d * x[0], atol=1e-12 * d * np.abs(x[0]).sum())


def test_rotation_is_orthogonal_and_preserves_inner_products():
    d = 128
    s = ti.sign_bits(ti.SEED_SIGNS_K, d)
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal(d), rng.standard_normal(d) * 30
    Tq, Tk = oracle.rotate(q, s), oracle.rotate(k, s)
    assert abs(np.linalg.norm(Tk) - np.linalg.norm(k)) / np.linalg.norm(k) < 1e-14
    assert abs(Tq @ Tk - q @ k) < 1e-12 * np.linalg.norm(q) * np.linalg.norm(k)
    T = hadamard(d) @ np.diag(_dsign(s)) / math.sqrt(d)
    np.testing.assert_allclose(Tk, T @ k, atol=1e-12 * np.abs(k).sum())
    np.testing.assert_allclose(oracle.unrotate(Tk, s), k, atol=1e-12 * np.abs(k).sum())
    # fp32 evaluation of the same transform keeps the norm to 1e-6
    T32 = T.astype(np.float32)
    k32 = k.astype(np.float32)
    assert abs(np.linalg.norm(T32 @ k32) - np.linalg.norm(k32)) / np.linalg.norm(k32) < 1e-6


def _explicit_u(x, signs):
    d = x.shape[0]
    n = np.linalg.norm(x)
    return hadamard(d) @ (_dsign(signs) * x) / n


def _adversarial(d):
    one_hot = np.zeros(d)
    one_hot[d // 2 - 1] = 3.0
    return [np.full(d, 65504.0), np.full(d, -65504.0), one_hot, np.arange(1, d + 1, dtype=np.float64) * (-1.0) ** np.arange(d)]


@pytest.mark.parametrize("d,bits", [(8, 1), (8, 2), (4, 3), (2, 4)])
def test_encoder_is_brute_force_nearest_code_vector(d, bits):
    c, t = oracle.make_codebook(bits)
    c64 = c.astype(np.float64)
    signs = ti.sign_bits(ti.SEED_SIGNS_K, d)
    L = 1 << bits
    allcodes = np.array(list(itertools.product(range(L), repeat=d)), dtype=np.int64)  # [L^d, d]
    recon = c64[allcodes]  # [L^d, d]
    rng = np.random.default_rng(100 * d + bits)
    xs = list(rng.standard_t(3, size=(40, d)) * rng.choice([1e-3, 1.0, 300.0], size=(40, 1))) + _adversarial(d)
    for x in xs:
        enc = oracle.encode_vector(x, bits, signs, c, t)
        u = _explicit_u(x, signs)
        np.testing.assert_allclose(enc["u"], u, rtol=0, atol=1e-12 * np.abs(u).max())
        dist = ((recon - u[None, :]) ** 2).sum(1)
        got = ((c64[enc["idx"]] - u) ** 2).sum()
        assert got <= dist.min() + 1e-12, (x, u)
        best = allcodes[np.argmin(dist)]
        tie = np.min(np.abs(u[:, None] - t.astype(np.float64)[None, :]), axis=1) < 1e-12
        assert np.array_equal(enc["idx"][~tie], best[~tie]), (x, u)
        # an exact tie between two centroids goes to the upper code
        assert np.all(enc["idx"][tie] == best[tie] + 1), (x, u)
        assert abs(enc["norm"] - np.linalg.norm(x)) <= 1e-15 * np.linalg.norm(x)


def test_zero_vector_is_a_true_zero_block():
    d, bits, m = 8, 2, 8
    c, t = oracle.make_codebook(bits)
    s = ti.sign_bits(ti.SEED_SIGNS_K, d)
    S = ti.gaussian_matrix(ti.SEED_QJL, m, d)
    enc = oracle.encode_vector(np.zeros(d), bits, s, c, t, S=S, qjl_m=m)
    assert enc["norm"] == 0.0 and enc["gamma"] == 0.0
    assert not enc["idx"].any() and not enc["z"].any()
    out = oracle.decode_vector(0.0, enc["idx"], bits, s, c, gamma=0.0, z=enc["z"], S=S, qjl_m=m)
    assert np.array_equal(out, np.zeros(d))


@pytest.mark.parametrize("bits,qjl", [(2, False), (3, True), (4, False), (4, True), (1, True)])
def test_decode_matches_dense_formula(bits, qjl):
    d, m = 16, 24
    c, t = oracle.make_codebook(bits)
    s = ti.sign_bits(ti.SEED_SIGNS_V, d)
    S = ti.gaussian_matrix(ti.SEED_QJL, m, d).astype(np.float64) if qjl else None
    rng = np.random.default_rng(bits)
    x = rng.standard_normal(d) * 5
    enc = oracle.encode_vector(x, bits, s, c, t, S=S, qjl_m=m if qjl else 0)
    D = np.diag(_dsign(s))
    H = hadamard(d).astype(np.float64)
    y = c.astype(np.float64)[enc["idx"]] / math.sqrt(d)
    if qjl:
        # residual, gamma and sign bits written out with dense matrices
        u = H @ D @ x / np.linalg.norm(x)
        e = (u - c.astype(np.float64)[enc["idx"]]) / math.sqrt(d)
        assert abs(enc["gamma"] - np.linalg.norm(e)) < 1e-13
        assert np.array_equal(enc["z"], (S @ e >= 0).astype(np.uint8))
        y = y + math.sqrt(math.pi / 2) / m * enc["gamma"] * (S.T @ (2.0 * enc["z"] - 1.0))
    want = enc["norm"] * D @ H @ y / math.sqrt(d)
    got = oracle.decode_vector(enc["norm"], enc["idx"], bits, s, c, gamma=enc["gamma"], z=enc["z"] if qjl else None,
                               S=S, qjl_m=m if qjl else 0)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12 * np.abs(want).max())


@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_pack_is_lsb_first_bitstream(b):
    rng = np.random.default_rng(b)
    vals = rng.integers(0, 1 << b, size=128)
    acc = 0
    for j, v in enumerate(vals):  # hand packing with a Python integer
        acc |= int(v) << (j * b)
    want = np.frombuffer(acc.to_bytes(128 * b // 8, "little"), dtype=np.uint8)
    got = oracle.pack_bits(vals, b)
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.unpack_bits(got, 128, b), vals)
    if b == 4:  # low nibble holds the even coordinate
        assert got[0] == (vals[0] | (vals[1] << 4))


def test_qjl_inner_product_is_unbiased_over_seeds():
    d, m, bits, nseeds = 128, 128, 2, 2000
    c, t = oracle.make_codebook(bits)
    s = ti.sign_bits(ti.SEED_SIGNS_K, d)
    rng = np.random.default_rng(11)
    x = rng.standard_t(3, d) * 4
    y = x.copy()  # MSE-only quantization is biased low for <x, x>
    truth = x @ y
    est = np.empty(nseeds)
    mse_only = None
    for i in range(nseeds):
        S = ti.gaussian_matrix(1000 + i, m, d)
        enc = oracle.encode_vector(x, bits, s, c, t, S=S, qjl_m=m)
        xh = oracle.decode_vector(enc["norm"], enc["idx"], bits, s, c, gamma=enc["gamma"], z=enc["z"], S=S, qjl_m=m)
        est[i] = xh @ y
        if mse_only is None:
            mse_only = oracle.decode_vector(enc["norm"], enc["idx"], bits, s, c) @ y
    se = est.std(ddof=1) / math.sqrt(nseeds)
    assert abs(est.mean() - truth) < 4 * se, (est.mean(), truth, se)
    assert abs(mse_only - truth) > 20 * se  # the correction is what removes the bias


def test_gaussian_sign_identity():
    # E[sign(s.e) (s.y)] = sqrt(2/pi) <e, y> / ||e|| for s ~ N(0, I): the reason the
    # dequantizer multiplies by sqrt(pi/2)
    d = 128
    S = ti.gaussian_matrix(77, 20000, d).astype(np.float64)
    rng = np.random.default_rng(5)
    e, y = rng.standard_normal(d), rng.standard_normal(d)
    samples = np.sign(S @ e) * (S @ y)
    want = math.sqrt(2 / math.pi) * (e @ y) / np.linalg.norm(e)
    assert abs(samples.mean() - want) < 4 * samples.std() / math.sqrt(len(samples))
    # the generator is standard normal
    assert abs(S.mean()) < 0.005 and abs(S.std() - 1) < 0.005


def test_paged_encode_decode_reproduces_validated_mse(golden):
    g = golden("validated_mse.json")
    d, N = 128, g["num_vectors"]
    rng = np.random.default_rng(2024)
    x = rng.standard_normal((N, 1, d)).astype(np.float16)
    xd = x.astype(np.float64)[:, 0]
    slots = np.arange(N, dtype=np.int32)
    s = ti.sign_bits(ti.SEED_SIGNS_V, d)
    for b in (2, 3, 4):
        f = ti.Format(128, b, b, 0, 128, 64, 1)
        lay = oracle.page_layout(f)
        npages = (N + 63) // 64
        pool = np.zeros(npages * lay["page_bytes"], np.uint8)
        c, t = oracle.make_codebook(b)
        assert oracle.encode(f, 1, x, slots, pool, npages, s, c, t) == 0
        rc, xh = oracle.decode(f, 1, pool, npages, slots, s, c)
        assert rc == 0
        mse = (((xh[:, 0] - xd) ** 2).sum(1) / (xd ** 2).sum(1)).mean()
        want = g["mse"][str(b)]
        assert abs(mse - want) / want < 0.05, (b, mse)
        assert mse > g["theory_lower"][str(b)] > 4.0 ** (-b) - 1e-4


def test_rotation_gaussianizes_heavy_tailed_vectors(golden):
    """Excess kurtosis per vector, before and after the structured rotation.

    The page measured real activations (mean 50.98 -> -0.13).  On the synthetic
    recipe the energy sits in a handful of outlier channels, so a rotated vector
    is close to a mix of a few Hadamard rows, whose kurtosis is mildly negative;
    "toward 0" is pinned as a collapse by more than an order of magnitude.  An
    i.i.d. light-tailed input must land on the Gaussian reference -6/(n+1)."""
    g = golden("kurtosis.json")

    def kurt(x):
        c = x - x.mean(1, keepdims=True)
        return (c ** 4).mean(1) / (c ** 2).mean(1) ** 2 - 3

    d = 128
    s = ti.sign_bits(ti.SEED_SIGNS_K, d)
    k = ti.kv_history(1, 512, 8, d, 0, 0).float().numpy().reshape(-1, d).astype(np.float64)
    before = kurt(k)
    after = kurt(np.stack([oracle.rotate(v, s) for v in k]))
    assert before.mean() > 10 and before.max() > g["before"]["max"] * 0.5
    assert abs(after.mean()) < 1.0 and after.max() < 3.0
    assert abs(after.mean()) < before.mean() / 20
    rng = np.random.default_rng(3)
    lap = rng.laplace(size=(2000, d))  # excess kurtosis 3 per coordinate
    ka = kurt(np.stack([oracle.rotate(v, s) for v in lap]))
    assert kurt(lap).mean() > 2.0 and abs(ka.mean()) < 0.15
    # an orthogonal map sends an i.i.d. Gaussian vector to an i.i.d. Gaussian
    # vector: the sample excess kurtosis keeps its textbook mean -6/(n+1)
    gs = rng.standard_normal((4000, d))
    kg = kurt(np.stack([oracle.rotate(v, s) for v in gs]))
    assert abs(kg.mean() + 6.0 / (d + 1)) < 4 * kg.std() / math.sqrt(len(kg))


@pytest.mark.parametrize("vb", [2, 3, 4])
def test_value_code_placement_by_hand(vb):
    """Where the oracle puts value codes, written out byte by byte.  Section
    rows of 16 coordinates hold 16 tokens of a group in the order 0,1,8,9,
    2,3,10,11,...; 2- and 4-bit codes of an offset pair (2p, 2p+1) are
    interleaved coordinate by coordinate, even coordinates first; 3-bit codes
    keep each token's chunk as its own LSB-first stream.  Tokens at offsets 2
    and 3 (a pair) and 9 (its partner 8 never written: zeros stay)."""
    f = ti.Format(128, 4, vb, 0, 128, 16, 1)
    lay = oracle.page_layout(f)
    signs = ti.sign_bits(11, 128)
    cen, mid = oracle.kind_codebook(f, 1)
    X = ti.kv_history(1, 3, 1, 128, 0, 1).numpy()[0]
    offs = [2, 3, 9]
    pool = np.zeros(lay["page_bytes"], np.uint8)
    assert oracle.encode(f, 1, X, np.array(offs, np.int32), pool, 1, signs, cen, mid) == 0
    idx = [oracle.encode_vector(X[n, 0].astype(np.float64), vb, signs, cen, mid)["idx"] for n in range(3)]
    sec = pool[lay["v_codes"]:lay["v_codes"] + 16 * 128 * vb // 8]
    row = 16 * 2 * vb  # bytes of one 16-coordinate row of a token group
    want = np.zeros_like(sec)
    for r in range(8):
        for c in range(16):
            a, b, z = (int(idx[n][16 * r + c]) for n in range(3))
            if vb == 4:
                # tokens 2, 3 at slots 4, 5 (bytes 32..47 of the row): 8 bytes of
                # even coordinates, then 8 of odd ones, one coordinate per byte,
                # offset 2 in the low nibble; token 9 at slots 2, 3 (bytes 16..31)
                # in the high nibbles
                want[r * row + 32 + 8 * (c % 2) + c // 2] = a | (b << 4)
                want[r * row + 16 + 8 * (c % 2) + c // 2] = z << 4
            elif vb == 2:
                # 4 bytes of even coordinates, then 4 of odd ones; a byte holds
                # two coordinates, each as (even offset, odd offset) 2-bit codes
                sh = 4 * ((c // 2) % 2)
                want[r * row + 16 + 4 * (c % 2) + c // 4] |= (a | (b << 2)) << sh
                want[r * row + 8 + 4 * (c % 2) + c // 4] |= (z << 2) << sh
            else:
                # 6-byte chunks: token 2 at slot 4, token 3 at 5, token 9 at 3
                for tok, slot in ((a, 4), (b, 5), (z, 3)):
                    for k in range(3):
                        bit = 8 * (r * row + 6 * slot) + 3 * c + k
                        want[bit // 8] |= ((tok >> k) & 1) << (bit % 8)
    assert np.array_equal(sec, want)
