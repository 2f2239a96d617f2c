"""The synthetic input recipe (the seeded generators both sides draw from).

Checks that the draws have the structure the workloads state:

- draws are deterministic per seed, layer and kind;
- coordinates are heavy-tailed (Student-t, nu = 3);
- four fixed outlier channels are about 20x the others;
- keys carry RoPE with theta_i = 500000^(-2i/d) on the interleaved pairs
  (2i, 2i+1);
- values are finite fp16 inside the clamp;
- the sign vectors are balanced bits;
- the QJL matrix is standard normal;
- the page table is a permutation.
"""
import math

import numpy as np
import torch

import tq_inputs as ti


def test_draws_are_deterministic_per_seed_layer_and_kind():
    a = ti.kv_history(2, 64, 2, 128, layer=3, kind=1)
    b = ti.kv_history(2, 64, 2, 128, layer=3, kind=1)
    assert torch.equal(a, b)
    assert not torch.equal(a, ti.kv_history(2, 64, 2, 128, layer=4, kind=1))
    assert not torch.equal(a, ti.kv_history(2, 64, 2, 128, layer=3, kind=0))
    assert torch.equal(ti.query(2, 8, 128), ti.query(2, 8, 128))


def test_heavy_tails_and_outlier_channels():
    v = ti.kv_history(4, 2048, 2, 128, layer=0, kind=1).double().numpy()  # values: no RoPE
    assert v.dtype == np.float64 and np.isfinite(v).all() and np.abs(v).max() <= 6.0e4
    flat = v.reshape(-1, 128)
    med = np.median(np.abs(flat), axis=0)
    out = list(ti.OUTLIER_CHANNELS)
    rest = [j for j in range(128) if j not in out]
    ratio = med[out] / np.median(med[rest])
    assert np.all(np.abs(ratio / ti.OUTLIER_SCALE - 1.0) < 0.15), ratio
    # Student-t with 3 degrees of freedom: far heavier tails than a Gaussian
    # (the sample excess kurtosis of a Gaussian is about 0)
    x = flat[:, rest].ravel()
    x = (x - x.mean()) / x.std()
    assert (x ** 4).mean() - 3.0 > 3.0
    # median |t_3| is 0.765 (a Gaussian's is 0.674)
    assert abs(np.median(np.abs(flat[:, rest])) - 0.765) < 0.05


def test_rope_rotates_interleaved_pairs():
    d = 128
    x = torch.randn(1, 5, 1, d, generator=torch.Generator().manual_seed(3))
    pos = torch.arange(5)
    y = ti.apply_rope(x, pos)
    assert torch.allclose(y[:, 0], x[:, 0])  # position 0 is the identity
    xp = x.double().reshape(1, 5, 1, d // 2, 2)
    yp = y.double().reshape(1, 5, 1, d // 2, 2)
    # pair norms are kept, and pair i turns by p * theta_i
    assert torch.allclose(xp.norm(dim=-1), yp.norm(dim=-1), rtol=1e-5)
    for p in range(5):
        for i in (0, 1, 17, 63):
            theta = p * 500000.0 ** (-2.0 * i / d)
            a = complex(float(xp[0, p, 0, i, 0]), float(xp[0, p, 0, i, 1]))
            b = complex(float(yp[0, p, 0, i, 0]), float(yp[0, p, 0, i, 1]))
            assert abs(b - a * complex(math.cos(theta), math.sin(theta))) < 1e-5 * max(1.0, abs(a))


def test_signs_matrix_and_page_table():
    for seed in (ti.SEED_SIGNS_K, ti.SEED_SIGNS_V):
        s = ti.sign_bits(seed, 4096)
        assert set(np.unique(s)) <= {0, 1} and abs(s.mean() - 0.5) < 0.03
    assert not np.array_equal(ti.sign_bits(ti.SEED_SIGNS_K, 128), ti.sign_bits(ti.SEED_SIGNS_V, 128))
    S = ti.gaussian_matrix(ti.SEED_QJL, 128, 128).astype(np.float64)
    assert S.shape == (128, 128)
    assert abs(S.mean()) < 0.02 and abs(S.var() - 1.0) < 0.03
    n = 1000
    perm = ti.page_permutation(n).numpy()
    assert np.array_equal(np.sort(perm), np.arange(n)) and not np.array_equal(perm, np.arange(n))
