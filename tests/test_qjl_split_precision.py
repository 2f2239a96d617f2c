"""Precision of the QJL projection as the kernels compute it, against the
sign-bit exemption of the parity tests (no GPU).

Both key-encode paths compute (S e)_l from fp16 hi/lo parts of S and of the
residual e with three products, hi.hi + lo.hi + hi.lo, accumulated in fp32
(the lo.lo term is left out).  The parity tests allow a sign bit to differ
from the fp64 oracle only where |(S e)_l| / gamma < 1e-4 (gamma = ||e||, the
oracle's sign margin).  This emulates that arithmetic in numpy (fp16 rounding
to nearest, fp32 accumulation in two different orders) on residuals of the
encode's scale and checks that its error stays an order of magnitude inside
the band, so that every sign outside the band is the oracle's.
"""
import numpy as np
import pytest

import tq_inputs as ti
from tq_testlib import EXEMPT


def _split(x):
    hi = x.astype(np.float16)
    lo = (x.astype(np.float32) - hi.astype(np.float32)).astype(np.float16)
    return hi.astype(np.float32), lo.astype(np.float32)


def _three_products(S, E, order):
    """(S e) for the rows of E from the hi/lo parts, fp32 accumulation:
    'k' sums over coordinates one product kind after the other (the tcgen05
    order: all K steps of hi.hi, then lo.hi, then hi.lo), 'c' sums the three
    kinds per coordinate block of 16 (the register path's order)."""
    sh, sl = _split(S)
    eh, el = _split(E)
    n, d = E.shape
    acc = np.zeros((n, S.shape[0]), np.float32)
    if order == "k":
        for a, b in ((eh, sh), (el, sh), (eh, sl)):
            for k0 in range(0, d, 16):
                acc += (a[:, k0:k0 + 16] @ b[:, k0:k0 + 16].T).astype(np.float32)
    else:
        for k0 in range(0, d, 16):
            for a, b in ((eh, sh), (el, sh), (eh, sl)):
                acc += (a[:, k0:k0 + 16] @ b[:, k0:k0 + 16].T).astype(np.float32)
    return acc


@pytest.mark.parametrize("scale", [0.02, 0.1, 0.3])
@pytest.mark.parametrize("order", ["k", "c"])
def test_three_product_split_stays_inside_the_sign_exemption(scale, order):
    d = m = 128
    S = ti.gaussian_matrix(ti.SEED_QJL, m, d).astype(np.float32)
    rng = np.random.default_rng(7)
    E = (rng.standard_normal((512, d)) * scale).astype(np.float32)
    exact = E.astype(np.float64) @ S.astype(np.float64).T
    got = _three_products(S, E, order).astype(np.float64)
    gamma = np.linalg.norm(E.astype(np.float64), axis=1, keepdims=True)
    err = np.abs(got - exact) / gamma
    assert err.max() < EXEMPT / 10, err.max()
    margin = np.abs(exact) / gamma
    outside = margin >= EXEMPT
    assert np.array_equal((got >= 0)[outside], (exact >= 0)[outside])


def test_hi_part_alone_would_not_stay_inside_the_exemption():
    """The reason for the lo products: hi.hi alone errs by more than the band."""
    d = m = 128
    S = ti.gaussian_matrix(ti.SEED_QJL, m, d).astype(np.float32)
    rng = np.random.default_rng(8)
    E = (rng.standard_normal((512, d)) * 0.1).astype(np.float32)
    sh, _ = _split(S)
    eh, _ = _split(E)
    exact = E.astype(np.float64) @ S.astype(np.float64).T
    gamma = np.linalg.norm(E.astype(np.float64), axis=1, keepdims=True)
    err = np.abs((eh @ sh.T).astype(np.float64) - exact) / gamma
    assert err.max() > EXEMPT
