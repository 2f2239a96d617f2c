"""Pins of the oracle's per-step append with an fp16 ring window.

The append of "TurboQuant Family Design Study for CPU and Browser WASM KV
Caches" ('Append cost and memory-bandwidth tradeoffs', 'Packed format and
complete bit accounting': the last W tokens stay fp16, 'Paging, lifecycle,
and cache identity': fixed pages filled in order) is checked against its
closed form after n steps from an empty cache: the window holds tokens
n-W .. n-1 with token t in ring slot t mod W, and the pages hold tokens
0 .. n-W-1 exactly as one direct encode of that token list at the slots of
compressed positions 0 .. n-W-1 writes them.
"""
import numpy as np
import pytest

import oracle
import tq_inputs as ti


def _setup(fmt, B, n, W, seed):
    H, d, P = fmt.num_kv_heads, fmt.head_dim, fmt.page_size
    rng = np.random.default_rng(seed)
    K = (rng.standard_normal((n, B, H, d)) * 2).astype(np.float16)
    V = (rng.standard_normal((n, B, H, d)) * 2).astype(np.float16)
    pages_per_seq = max(1, (n + P - 1) // P)
    num_pages = B * pages_per_seq + 1
    bt = rng.permutation(num_pages)[: B * pages_per_seq].astype(np.int32).reshape(B, pages_per_seq)
    lay = oracle.page_layout(fmt)
    pool = np.full(num_pages * lay["page_bytes"], 0x33, np.uint8)
    kcb, vcb = oracle.make_codebook(fmt.k_bits), oracle.make_codebook(fmt.v_bits)
    ks = ti.sign_bits(ti.SEED_SIGNS_K, d)
    vs = ti.sign_bits(ti.SEED_SIGNS_V, d)
    S = ti.gaussian_matrix(ti.SEED_QJL, fmt.qjl_m, d) if fmt.k_qjl else None
    return K, V, bt, num_pages, pool, kcb, vcb, ks, vs, S


@pytest.mark.parametrize("W,n,qjl", [(4, 40, 0), (4, 3, 0), (4, 4, 1), (5, 37, 1), (0, 21, 0), (1, 18, 0)])
def test_append_matches_closed_form(W, n, qjl):
    fmt = ti.Format(32, 3, 2, qjl, 32, 16, 2)
    B, H, d, P = 3, fmt.num_kv_heads, fmt.head_dim, fmt.page_size
    K, V, bt, num_pages, pool, kcb, vcb, ks, vs, S = _setup(fmt, B, n, W, seed=W * 100 + n)
    kw = np.zeros((B, H, W, d), np.float16) if W else None
    vw = np.zeros((B, H, W, d), np.float16) if W else None
    wl = np.zeros(B, np.int32)
    wh = np.zeros(B, np.int32)
    cl = np.zeros(B, np.int32)
    for t in range(n):
        skipped = oracle.append_window(fmt, K[t], V[t], kw, vw, wl, wh, cl, bt, pool, num_pages, ks, vs, kcb, vcb, S)
        assert skipped == []

    ncomp = max(0, n - W)
    assert list(wl) == [min(n, W)] * B
    assert list(wh) == [((n - W) % W if n >= W else 0) if W else 0] * B
    assert list(cl) == [ncomp] * B
    for t in range(max(0, n - W), n):
        np.testing.assert_array_equal(kw[:, :, t % W], K[t])
        np.testing.assert_array_equal(vw[:, :, t % W], V[t])

    # the pages: one direct encode of tokens 0 .. ncomp-1 per sequence
    ref = np.full_like(pool, 0x33)
    for b in range(B):
        slots = np.array([bt[b, c // P] * P + c % P for c in range(ncomp)], np.int32)
        if ncomp:
            assert oracle.encode(fmt, 0, K[:ncomp, b], slots, ref, num_pages, ks, *kcb, S) == 0
            assert oracle.encode(fmt, 1, V[:ncomp, b], slots, ref, num_pages, vs, *vcb) == 0
    np.testing.assert_array_equal(pool, ref)


def test_append_missing_page_leaves_sequence_untouched():
    fmt = ti.Format(32, 4, 4, 0, 32, 16, 2)
    B, W, n = 2, 4, 30
    K, V, bt, num_pages, pool, kcb, vcb, ks, vs, S = _setup(fmt, B, n, W, seed=5)
    H, d = fmt.num_kv_heads, fmt.head_dim
    kw = np.zeros((B, H, W, d), np.float16)
    vw = np.zeros((B, H, W, d), np.float16)
    wl, wh, cl = np.zeros(B, np.int32), np.zeros(B, np.int32), np.zeros(B, np.int32)
    bt[1, 1] = -1  # sequence 1 has no page for compressed positions 16..31
    for t in range(n):
        before = (kw[1].copy(), wl[1], wh[1], cl[1], pool.copy())
        skipped = oracle.append_window(fmt, K[t], V[t], kw, vw, wl, wh, cl, bt, pool, num_pages, ks, vs, kcb, vcb, S)
        if t >= W + 16:  # the 17th eviction needs the missing page
            assert skipped == [1]
            np.testing.assert_array_equal(kw[1], before[0])
            assert (wl[1], wh[1], cl[1]) == before[1:4]
        else:
            assert skipped == []
    assert cl[0] == n - W and cl[1] == 16
