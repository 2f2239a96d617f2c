"""GPU parity of the KIVI-style control arm against its fp64 oracle.

* encode: the pool the GPU writes equals, byte for byte, the pool the oracle
  writes from the same inputs (fp16 scales and zeros, codes, and every byte
  the encode must not touch); the codes are decided in fp32 on both sides;
* decode: the GPU reconstruction z + s * code within fp32 rounding;
* decode attention: max |o - o_ref| / max |o_ref| <= 2e-3 per (sequence,
  query head) over ragged lengths, partial pages, windows and GQA 1..8.
"""
import numpy as np
import pytest
import torch

import oracle
import tq_inputs as ti
from tq_testlib import REL_ATTN, rel_err

pytestmark = pytest.mark.gpu


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("kb,vb,P", [(2, 2, 64), (4, 4, 64), (4, 2, 16), (2, 4, 128)])
def test_kivi_encode_matches_oracle_bytes(kb, vb, P):
    import decode_attention_tq_gb300 as tq

    f = ti.KiviFormat(128, kb, vb, P, 3)
    N = 3 * P + P // 2 + 5  # three full pages and a partial one
    K = ti.kv_history(1, N, 3, 128, 2, 0).numpy()[0]
    V = ti.kv_history(1, N, 3, 128, 2, 1).numpy()[0]
    V[5] = 0  # an all-zero token (zero scale)
    K[:, :, 9] = np.float16(1.5)  # a constant channel
    num_pages = 9
    lay = oracle.kivi_layout(f)
    pages = ti.page_permutation(num_pages).numpy()[:4].astype(np.int32)
    slots = (pages[np.arange(N) // P] * P + np.arange(N) % P).astype(np.int32)
    slots[7] = -1  # skipped
    ref = np.full(num_pages * lay["page_bytes"], 0x5A, np.uint8)
    assert oracle.kivi_encode_keys(f, K, pages, ref, num_pages) == 0
    assert oracle.kivi_encode_values(f, V, slots, ref, num_pages) == 0
    pool = torch.full((num_pages * lay["page_bytes"],), 0x5A, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.tq_kivi_encode_keys(f, _t(K), _t(pages), pool, num_pages, err_word=err)
    tq.tq_kivi_encode_values(f, _t(V), _t(slots), pool, num_pages, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = pool.cpu().numpy()
    diff = np.flatnonzero(got != ref)
    assert diff.size == 0, (diff[:10], got[diff[:10]], ref[diff[:10]])


def test_kivi_encode_range_errors():
    import decode_attention_tq_gb300 as tq

    f = ti.KiviFormat(128, 2, 2, 16, 1)
    N = 40
    K = ti.kv_history(1, N, 1, 128, 0, 0).numpy()[0]
    pages = np.array([0, 7, 1], np.int32)  # page 7 is outside a 4-page pool
    lay = oracle.kivi_layout(f)
    pool = torch.zeros(4 * lay["page_bytes"], dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.tq_kivi_encode_keys(f, _t(K), _t(pages), pool, 4, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == tq.TQ_DEVERR_PAGE_RANGE
    err.zero_()
    tq.tq_kivi_encode_values(f, _t(K), _t(np.arange(N, dtype=np.int32) + 60), pool, 4, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == tq.TQ_DEVERR_SLOT_RANGE


@pytest.mark.parametrize("kind,bits", [(0, 2), (0, 4), (1, 2), (1, 4)])
def test_kivi_decode_matches_oracle(kind, bits):
    import decode_attention_tq_gb300 as tq

    f = ti.KiviFormat(128, bits, bits, 32, 2)
    N = 100
    X = ti.kv_history(1, N, 2, 128, 1, kind).numpy()[0]
    num_pages = 5
    lay = oracle.kivi_layout(f)
    pages = np.arange(4, dtype=np.int32)
    slots = (pages[np.arange(N) // 32] * 32 + np.arange(N) % 32).astype(np.int32)
    pool = np.zeros(num_pages * lay["page_bytes"], np.uint8)
    if kind == 0:
        assert oracle.kivi_encode_keys(f, X, pages, pool, num_pages) == 0
    else:
        assert oracle.kivi_encode_values(f, X, slots, pool, num_pages) == 0
    rc, ref = oracle.kivi_decode(f, kind, pool, num_pages, slots)
    assert rc == 0
    out = tq.tq_kivi_decode(f, kind, _t(pool), num_pages, _t(slots))
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    # z + s * code in fp32 (one fma) against fp64
    assert np.all(np.abs(got - ref) <= 2.0 ** -23 * np.maximum(np.abs(ref), 1e-30) + 1e-30)


class KiviScenario:
    """A KIVI decode-attention case: K/V from the seeded recipe, encoded by the
    oracle into permuted pages (keys a page group at a time), query and window."""

    def __init__(self, f, B, Hq, comp, W, wl, layer=0, extra_pages=3):
        d, H, P = f.head_dim, f.num_kv_heads, f.page_size
        self.f, self.B, self.Hq, self.W = f, B, Hq, W
        self.comp = np.array(comp, np.int32)
        self.wl = np.array(wl, np.int32)
        self.max_pages = max(1, max(-(-c // P) for c in comp))
        self.num_pages = B * self.max_pages + extra_pages
        perm = ti.page_permutation(self.num_pages).numpy()
        self.bt = perm[: B * self.max_pages].reshape(B, self.max_pages).astype(np.int32)
        self.lay = oracle.kivi_layout(f)
        self.pool = np.full(self.num_pages * self.lay["page_bytes"], 0xA5, np.uint8)
        T = max(int(self.comp.max()) + W, 1)
        K = ti.kv_history(B, T, H, d, layer, 0).numpy()
        V = ti.kv_history(B, T, H, d, layer, 1).numpy()
        self.kwin = np.zeros((B, H, max(W, 1), d), np.float16)
        self.vwin = np.zeros((B, H, max(W, 1), d), np.float16)
        for b in range(B):
            c = int(self.comp[b])
            if c:
                npg = -(-c // P)
                assert oracle.kivi_encode_keys(f, K[b, :c], self.bt[b, :npg], self.pool, self.num_pages) == 0
                sl = (self.bt[b, np.arange(c) // P] * P + np.arange(c) % P).astype(np.int32)
                assert oracle.kivi_encode_values(f, V[b, :c], sl, self.pool, self.num_pages) == 0
            n = int(self.wl[b]) if W else 0
            self.kwin[b, :, :n] = K[b, c:c + n].transpose(1, 0, 2)
            self.vwin[b, :, :n] = V[b, c:c + n].transpose(1, 0, 2)
        self.q = ti.query(B, Hq, d).numpy()

    def oracle_attention(self, bt=None):
        return oracle.kivi_attention(self.f, self.q, self.pool, self.num_pages, self.bt if bt is None else bt, self.comp,
                                     self.kwin if self.W else None, self.vwin if self.W else None, self.wl)

    def gpu_attention(self, bt=None, err=None):
        import decode_attention_tq_gb300 as tq

        out = torch.full((self.B, self.Hq, self.f.head_dim), float("nan"), dtype=torch.float32, device="cuda")
        ws = torch.empty(tq.tq_kivi_decode_attn_workspace_size(self.f, self.B, self.Hq, self.max_pages, self.W), dtype=torch.uint8,
                         device="cuda")
        tq.tq_kivi_decode_attn(self.f, _t(self.q), _t(self.pool), self.num_pages, _t(self.bt if bt is None else bt), _t(self.comp),
                               _t(self.kwin) if self.W else None, _t(self.vwin) if self.W else None,
                               _t(self.wl) if self.W else None, out, ws, err_word=err)
        torch.cuda.synchronize()
        return out.cpu().numpy()


ATTN_CASES = {
    # name: (k_bits, v_bits, P, H, B, Hq, comp lens, W, win lens)
    "k2v2_g4": (2, 2, 64, 2, 2, 8, [1000, 333], 32, [32, 7]),
    "k4v4_g4": (4, 4, 64, 2, 2, 8, [640, 77], 0, [0, 0]),
    "k4v2_g1_p16": (4, 2, 16, 4, 3, 4, [129, 16, 1], 8, [8, 0, 5]),
    "k2v4_g8_p128": (2, 4, 128, 1, 2, 8, [300, 900], 16, [16, 16]),
    "k2v2_g2_window_only": (2, 2, 32, 2, 2, 4, [0, 0], 24, [24, 11]),
    "k4v4_g3_w300": (4, 4, 32, 2, 2, 6, [95, 257], 300, [300, 130]),
    "k2v2_g6_short": (2, 2, 16, 1, 4, 6, [5, 17, 33, 250], 4, [4, 4, 1, 0]),
}


@pytest.mark.parametrize("name", list(ATTN_CASES))
def test_kivi_attention_matches_oracle(name):
    kb, vb, P, H, B, Hq, comp, W, wl = ATTN_CASES[name]
    sc = KiviScenario(ti.KiviFormat(128, kb, vb, P, H), B, Hq, comp, W, wl)
    rc, ref = sc.oracle_attention()
    assert rc == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = sc.gpu_attention(err=err)
    assert int(err.item()) == 0
    assert np.isfinite(got).all()
    e = rel_err(got, ref)
    print(name, "max rel err", e.max())
    assert e.max() <= REL_ATTN, (name, e.max())


def test_kivi_attention_page_outside_pool():
    import decode_attention_tq_gb300 as tq

    sc = KiviScenario(ti.KiviFormat(128, 4, 4, 16, 1), 1, 2, [64], 0, [0])
    bt = sc.bt.copy()
    bt[0, 2] = sc.num_pages + 4
    rc, ref = sc.oracle_attention(bt=bt)
    assert rc == -2  # the oracle skips that page too
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = sc.gpu_attention(bt=bt, err=err)
    assert int(err.item()) & tq.TQ_DEVERR_PAGE_RANGE
    assert rel_err(got, ref).max() <= REL_ATTN
