"""GPU parity of libtq against the fp64 oracle, through the C ABI.

Encode: codes and sign bits bit-exact except where the oracle's fp64
coordinate lies within 1e-4 of a decision boundary; fp32 norms / gammas to
1e-6 relative; untouched bytes identical.  Decode: fp32 reconstruction to
1e-5 of the vector's max.  Attention: max |o - o_ref| / max |o_ref| <= 2e-3
per (sequence, query head), the tolerance the benchmark spec's target states.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tq_inputs as ti
from tq_testlib import REL_ATTN, Scenario, check_exemption_reach, compare_encoded, gpu_attention, rel_err

pytestmark = pytest.mark.gpu

tq = pytest.importorskip("decode_attention_tq_gb300")


def _encode_case(fmt, kind, N, seed, zero_rows=(), neg_slots=()):
    d, H, P = fmt.head_dim, fmt.num_kv_heads, fmt.page_size
    num_pages = (N + P - 1) // P + 2
    lay = oracle.page_layout(fmt)
    x = ti.kv_history(1, N, H, d, seed, kind)[0].numpy()  # [N, H, d]
    for zr in zero_rows:
        x[zr] = 0
    perm = np.random.default_rng(seed).permutation(num_pages * P)[:N].astype(np.int32)
    for ns in neg_slots:
        perm[ns] = -1
    signs = ti.sign_bits(ti.SEED_SIGNS_K if kind == 0 else ti.SEED_SIGNS_V, d)
    bits = fmt.k_bits if kind == 0 else fmt.v_bits
    c, t = oracle.kind_codebook(fmt, kind)
    S = None
    if kind == 0 and fmt.k_qjl:
        S = (ti.orthogonal_matrix if fmt.qjl_scale > 0 else ti.gaussian_matrix)(ti.SEED_QJL, fmt.qjl_m, d)
    pool_ref = np.full(num_pages * lay["page_bytes"], 0x5A, np.uint8)
    rc, u, cm, sm = oracle.encode(fmt, kind, x, perm, pool_ref, num_pages, signs, c, t, S, diagnostics=True)
    assert rc == 0
    pool = torch.full((num_pages * lay["page_bytes"],), 0x5A, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.tq_encode(fmt, kind, torch.from_numpy(x).cuda(), torch.from_numpy(perm).cuda(), pool, num_pages,
                 torch.from_numpy(signs).cuda(), tq.kind_codebook(fmt, kind), None if S is None else torch.from_numpy(S).cuda(), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return pool.cpu().numpy(), pool_ref, lay, perm, cm, sm, x, signs, c, S, num_pages


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("kind,qjl", [(0, 0), (0, 1), (1, 0)])
def test_encode_matches_oracle(bits, kind, qjl):
    fmt = ti.Format(128, bits, bits, qjl, 128, 64, 4)
    N = 333  # several pages and a ragged tail
    pool, pool_ref, lay, slots, cm, sm, *_ = _encode_case(fmt, kind, N, seed=bits + 10 * kind + 100 * qjl,
                                                          zero_rows=(5, 200), neg_slots=(17,))
    st = compare_encoded(pool, pool_ref, lay, fmt, kind, slots, cm, sm)
    print("encode", bits, kind, qjl, st)


@pytest.mark.parametrize("bits,kind,qjl", [(2, 0, 1), (3, 1, 0), (4, 0, 0), (4, 0, 1), (2, 1, 0), (4, 1, 0)])
def test_decode_matches_oracle(bits, kind, qjl):
    fmt = ti.Format(128, bits, bits, qjl, 128, 32, 2)
    N = 150
    pool, pool_ref, lay, slots, cm, sm, x, signs, c, S, num_pages = _encode_case(fmt, kind, N, seed=7)
    # the GPU decodes the oracle's pages
    out = tq.tq_decode(fmt, kind, torch.from_numpy(pool_ref).cuda(), num_pages, torch.from_numpy(slots).cuda(),
                       torch.from_numpy(signs).cuda(), tq.kind_codebook(fmt, kind), None if S is None else torch.from_numpy(S).cuda())
    torch.cuda.synchronize()
    rc, ref = oracle.decode(fmt, kind, pool_ref, num_pages, slots, signs, c, S)
    assert rc == 0
    e = rel_err(out.cpu().numpy(), ref)
    assert e.max() < 1e-5, e.max()
    # the zero vector decodes to exact zeros on both sides
    z = np.all(x == 0, axis=-1)
    assert np.all(out.cpu().numpy()[z] == 0)


ORTH_SHRINK = 0.7 * math.sqrt(math.pi / 2) / math.sqrt(128)  # orthogonal S, 0.7 damping


@pytest.mark.parametrize("bits,kmix", [(2, 0), (4, 0), (3, 1)])
def test_encode_qjl_many_batches_matches_oracle(bits, kmix):
    """Keys with QJL over more 128-vector batches than the grid has blocks
    (40,024 vectors: every block runs two or three batches through both
    residual/accumulator buffers, the last batch ragged), with zero vectors
    and skipped tokens; every field against the oracle."""
    fmt = ti.Format(128, bits, 4, 1, 128, 64, 8, k_mixed=kmix)
    N = 5003
    pool, pool_ref, lay, slots, cm, sm, *_ = _encode_case(fmt, 0, N, seed=40 + bits + 5 * kmix,
                                                          zero_rows=(0, 2500, N - 1), neg_slots=(7, 4099))
    st = compare_encoded(pool, pool_ref, lay, fmt, 0, slots, cm, sm)
    check_exemption_reach(st, f"qjl many batches b{bits} mixed {kmix}")
    print("qjl many batches", bits, kmix, st)


@pytest.mark.parametrize("b,qjl,nc", [(3, 0, 0), (2, 0, 0), (3, 1, 0), (2, 1, 0), (3, 0, 1)])
def test_encode_mixed_keys_matches_oracle(b, qjl, nc):
    """Keys at 3.5 / 2.5 bits per channel (b+1 bits on j mod 16 < 8, b on the rest)."""
    fmt = ti.Format(128, b, 4, qjl, 128, 64, 4, norm_correct=nc, k_mixed=1)
    pool, pool_ref, lay, slots, cm, sm, *_ = _encode_case(fmt, 0, 300, seed=b + 20 * qjl + 7 * nc, zero_rows=(4,), neg_slots=(11,))
    st = compare_encoded(pool, pool_ref, lay, fmt, 0, slots, cm, sm)
    print("mixed encode", b, qjl, nc, st)


@pytest.mark.parametrize("b,qjl", [(3, 1), (2, 0)])
def test_decode_mixed_keys_matches_oracle(b, qjl):
    fmt = ti.Format(128, b, 4, qjl, 128, 32, 2, k_mixed=1)
    pool, pool_ref, lay, slots, cm, sm, x, signs, c, S, num_pages = _encode_case(fmt, 0, 100, seed=b + 90)
    out = tq.tq_decode(fmt, 0, torch.from_numpy(pool_ref).cuda(), num_pages, torch.from_numpy(slots).cuda(),
                       torch.from_numpy(signs).cuda(), tq.kind_codebook(fmt, 0), None if S is None else torch.from_numpy(S).cuda())
    torch.cuda.synchronize()
    rc, ref = oracle.decode(fmt, 0, pool_ref, num_pages, slots, signs, c, S)
    assert rc == 0
    e = rel_err(out.cpu().numpy(), ref)
    assert e.max() < 1e-5, e.max()


@pytest.mark.parametrize("bits,kind", [(4, 0), (3, 1), (2, 0)])
def test_encode_norm_correction_matches_oracle(bits, kind):
    fmt = ti.Format(128, bits, bits, 0, 128, 64, 4, norm_correct=1)
    pool, pool_ref, lay, slots, cm, sm, *_ = _encode_case(fmt, kind, 200, seed=bits + 50, zero_rows=(9,), neg_slots=(3,))
    st = compare_encoded(pool, pool_ref, lay, fmt, kind, slots, cm, sm)
    print("norm-corrected encode", bits, kind, st)


@pytest.mark.parametrize("bits", [2, 4])
def test_decode_orthogonal_qjl_factor_matches_oracle(bits):
    fmt = ti.Format(128, bits, bits, 1, 128, 32, 2, qjl_scale=ORTH_SHRINK)
    pool, pool_ref, lay, slots, cm, sm, x, signs, c, S, num_pages = _encode_case(fmt, 0, 120, seed=bits + 70)
    out = tq.tq_decode(fmt, 0, torch.from_numpy(pool_ref).cuda(), num_pages, torch.from_numpy(slots).cuda(),
                       torch.from_numpy(signs).cuda(), tq.device_codebook(bits), torch.from_numpy(S).cuda())
    torch.cuda.synchronize()
    rc, ref = oracle.decode(fmt, 0, pool_ref, num_pages, slots, signs, c, S)
    assert rc == 0
    e = rel_err(out.cpu().numpy(), ref)
    assert e.max() < 1e-5, e.max()


ATTN_CASES = {
    # name: (fmt, B, Hq, comp_lens, W, win_lens)
    "k4v4_g4_t2048": (ti.Format(128, 4, 4, 0, 128, 64, 8), 1, 32, [2048], 0, [0]),
    "k3qjl_v4_g8_w": (ti.Format(128, 3, 4, 1, 128, 64, 2), 2, 16, [1000, 333], 128, [128, 77]),
    "k2qjl_v2_p128_w": (ti.Format(128, 2, 2, 1, 128, 128, 2), 2, 8, [700, 129], 64, [64, 64]),
    "k4v4_ragged_w": (ti.Format(128, 4, 4, 0, 128, 64, 4), 3, 16, [1, 640, 97], 16, [16, 5, 0]),
    "k4v3_g2": (ti.Format(128, 4, 3, 0, 128, 32, 3), 2, 6, [300, 47], 0, [0, 0]),
    "k2v4_g1": (ti.Format(128, 2, 4, 0, 128, 16, 4), 1, 4, [175], 8, [3]),
    "window_only": (ti.Format(128, 4, 4, 0, 128, 64, 2), 2, 8, [0, 0], 40, [40, 13]),
    "empty_seq": (ti.Format(128, 3, 3, 1, 128, 64, 2), 3, 8, [0, 200, 0], 8, [0, 8, 5]),
    "k3qjl_orth_shrink_v4_w": (ti.Format(128, 3, 4, 1, 128, 64, 2, qjl_scale=ORTH_SHRINK), 2, 8, [900, 257], 32, [32, 9]),
    "k4v4_norm_corrected": (ti.Format(128, 4, 4, 0, 128, 64, 4, norm_correct=1), 2, 16, [500, 64], 16, [16, 3]),
    "k35v4_w": (ti.Format(128, 3, 4, 0, 128, 64, 4, k_mixed=1), 2, 16, [777, 130], 32, [32, 11]),
    "k25qjl_v2_g8": (ti.Format(128, 2, 2, 1, 128, 64, 2, k_mixed=1), 2, 16, [600, 97], 16, [16, 16]),
    "k35qjl_v3_ragged": (ti.Format(128, 3, 3, 1, 128, 32, 4, k_mixed=1), 3, 16, [1, 333, 64], 8, [0, 8, 2]),
    "k25v4_p16": (ti.Format(128, 2, 4, 0, 128, 16, 8, k_mixed=1), 1, 32, [250], 0, [0]),
    # windows longer than 8 chunks of 32 (the merge's second window path)
    "k4v4_w300": (ti.Format(128, 4, 4, 0, 128, 64, 2), 2, 8, [410, 0], 300, [300, 259]),
    # GQA groups that are not powers of two (partly filled MMA columns)
    "k3v4_g3": (ti.Format(128, 3, 4, 0, 128, 64, 3), 2, 9, [333, 700], 16, [16, 1]),
    "k4qjl_v2_g7": (ti.Format(128, 4, 2, 1, 128, 64, 2), 1, 14, [515], 32, [20]),
    # 4-bit keys without QJL (centroid tables shifted to 64 KB shared-window
    # boundaries) with every value width and both column-tile counts
    "k4v4_g8_w": (ti.Format(128, 4, 4, 0, 128, 64, 2), 2, 16, [800, 310], 24, [24, 7]),
    "k4v3_g6": (ti.Format(128, 4, 3, 0, 128, 32, 2), 2, 12, [450, 1], 0, [0, 0]),
    "k4v2_g4_w": (ti.Format(128, 4, 2, 0, 128, 64, 4), 2, 16, [390, 1025], 40, [40, 33]),
    # a page of 48 tokens (three tiles per page) and many short sequences
    "k4v4_p48_b24": (ti.Format(128, 4, 4, 0, 128, 48, 2), 24, 4, [int(x) for x in (np.arange(24) * 37) % 211], 8, [int(x) for x in np.arange(24) % 9]),
    # batch-1 shapes with one or two kv heads and long sequences: hundreds to
    # over a thousand partials per (b, h), so the merge cuts a row into
    # several slices (the block finishing a row's last slice merges them);
    # the window partials come from their own kernel; the main kernel takes
    # ready-made query operands
    "k4v4_h1_g8_t24k_w": (ti.Format(128, 4, 4, 0, 128, 64, 1), 1, 8, [24000], 48, [48]),
    "k3qjl_v4_h2_g8_t16k_w": (ti.Format(128, 3, 4, 1, 128, 64, 2), 1, 16, [16000], 128, [128]),
    # rows with many partials beside rows with few (one slice, one chunk)
    "k4v4_h1_g4_ragged": (ti.Format(128, 4, 4, 0, 128, 64, 1), 2, 4, [20000, 300], 16, [16, 5]),
    # more than 31 short sequences (the first tile located by a binary search
    # over the tile prefix sums, not by a lane ballot)
    "k4v4_b40_short": (ti.Format(128, 4, 4, 0, 128, 16, 2), 40, 4, [int(x) for x in (np.arange(40) * 13) % 90 + 1], 8,
                       [int(x) for x in np.arange(40) % 8]),
}


@pytest.mark.parametrize("name", list(ATTN_CASES))
def test_attention_matches_oracle(name):
    fmt, B, Hq, comp, W, wl = ATTN_CASES[name]
    sc = Scenario(fmt, B, Hq, comp, W, wl, layer=3)
    dev = sc.device_inputs()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_attention(sc, dev, err=err)
    rc, ref = sc.oracle_attention()
    assert rc == 0 and int(err.item()) == 0
    e = rel_err(out, ref)
    print(name, "max rel err", float(e.max()))
    # heads with no token at all are exactly zero on both sides
    assert np.all(np.isfinite(out))
    assert e.max() <= REL_ATTN, e.max()


def test_attention_end_to_end_gpu_encode():
    """GPU encode -> GPU attention against oracle encode -> oracle attention."""
    fmt = ti.Format(128, 3, 4, 1, 128, 64, 4)
    B, Hq, comp, W, wl = 2, 16, [900, 450], 32, [32, 20]
    sc = Scenario(fmt, B, Hq, comp, W, wl, layer=5)
    dev = sc.device_inputs()
    pool = torch.full_like(dev["pool"], 0xA5)
    for b in range(B):
        c = comp[b]
        sl = torch.from_numpy(sc.slots[b]).cuda()
        tq.tq_encode(fmt, 0, torch.from_numpy(np.ascontiguousarray(sc.K[b, :c])).cuda(), sl, pool, sc.num_pages, dev["ks"], dev["kcb"], dev["S"])
        tq.tq_encode(fmt, 1, torch.from_numpy(np.ascontiguousarray(sc.V[b, :c])).cuda(), sl, pool, sc.num_pages, dev["vs"], dev["vcb"])
    dev["pool"] = pool
    out = gpu_attention(sc, dev)
    rc, ref = sc.oracle_attention()
    e = rel_err(out, ref)
    print("end-to-end max rel err", float(e.max()))
    assert e.max() <= REL_ATTN


@pytest.mark.parametrize("kb,vb,qjl", [(2, 2, 0), (3, 3, 0), (4, 4, 0), (4, 4, 1), (3, 4, 1), (2, 4, 0)])
def test_encode_kv_matches_two_encodes(kb, vb, qjl):
    """The joint K+V append writes exactly the bytes of two single-kind appends."""
    fmt = ti.Format(128, kb, vb, qjl, 128, 64, 4)
    d, H, P = fmt.head_dim, fmt.num_kv_heads, fmt.page_size
    N = 301
    num_pages = (N + P - 1) // P + 2
    lay = oracle.page_layout(fmt)
    k = ti.kv_history(1, N, H, d, 7 + kb, 0)[0].cuda()
    v = ti.kv_history(1, N, H, d, 7 + vb, 1)[0].cuda()
    k[3] = 0
    v[250] = 0
    perm = np.random.default_rng(kb * 10 + vb).permutation(num_pages * P)[:N].astype(np.int32)
    perm[40] = -1
    sl = torch.from_numpy(perm).cuda()
    ks = torch.from_numpy(ti.sign_bits(ti.SEED_SIGNS_K, d)).cuda()
    vs = torch.from_numpy(ti.sign_bits(ti.SEED_SIGNS_V, d)).cuda()
    S = torch.from_numpy(ti.gaussian_matrix(ti.SEED_QJL, fmt.qjl_m, d)).cuda() if qjl else None
    kcb, vcb = tq.device_codebook(kb), tq.device_codebook(vb)
    two = torch.full((num_pages * lay["page_bytes"],), 0x3C, dtype=torch.uint8, device="cuda")
    one = two.clone()
    tq.tq_encode(fmt, 0, k, sl, two, num_pages, ks, kcb, S)
    tq.tq_encode(fmt, 1, v, sl, two, num_pages, vs, vcb)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.tq_encode_kv(fmt, k, v, sl, one, num_pages, ks, vs, kcb, vcb, S, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(one, two)
    # an out-of-range slot is skipped and flagged, the other tokens still land
    bad = sl.clone()
    bad[0] = num_pages * P
    three = torch.full_like(one, 0x3C)
    tq.tq_encode_kv(fmt, k, v, bad, three, num_pages, ks, vs, kcb, vcb, S, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == tq.TQ_DEVERR_SLOT_RANGE
    page, off = int(perm[0]) // P, int(perm[0]) % P
    assert not torch.equal(three, one)
    mask = torch.ones_like(one, dtype=torch.bool)
    mask[page * lay["page_bytes"]:(page + 1) * lay["page_bytes"]] = False
    assert torch.equal(three[mask], one[mask])


def test_bad_page_is_skipped_and_flagged():
    fmt = ti.Format(128, 4, 4, 0, 128, 64, 2)
    sc = Scenario(fmt, 2, 4, [300, 130], 0, [0, 0], layer=1)
    dev = sc.device_inputs()
    bt = sc.bt.copy()
    bt[0, 2] = sc.num_pages + 7
    bt[1, 0] = -3
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_attention(sc, dev, err=err, bt=torch.from_numpy(bt).cuda())
    assert int(err.item()) & tq.TQ_DEVERR_PAGE_RANGE
    rc, ref = sc.oracle_attention(bt=bt)
    assert rc == -2  # the oracle skips the same pages
    assert rel_err(out, ref).max() <= REL_ATTN


def test_length_errors_are_clamped_and_flagged():
    fmt = ti.Format(128, 4, 4, 0, 128, 64, 2)
    sc = Scenario(fmt, 2, 4, [128, 64], 8, [8, 4], layer=2)
    dev = sc.device_inputs()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    comp = torch.tensor([10_000, 64], dtype=torch.int32, device="cuda")  # beyond max_pages * P
    out = gpu_attention(sc, dev, err=err, comp=comp)
    assert int(err.item()) & tq.TQ_DEVERR_LENGTH
    rc, ref = sc.oracle_attention(comp=np.array([sc.max_pages * 64, 64], np.int32))
    assert rel_err(out, ref).max() <= REL_ATTN


def test_encode_slot_out_of_range_flagged():
    fmt = ti.Format(128, 4, 4, 0, 128, 64, 1)
    x = torch.randn(4, 1, 128, device="cuda").half()
    pool = torch.zeros(2 * tq.tq_page_layout(fmt)["page_bytes"], dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.tensor([0, 1, 128, 5], dtype=torch.int32, device="cuda")
    tq.tq_encode(fmt, 1, x, slots, pool, 2, torch.zeros(128, dtype=torch.uint8, device="cuda"), tq.device_codebook(4), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == tq.TQ_DEVERR_SLOT_RANGE


def test_host_argument_errors():
    fmt = ti.Format(128, 4, 4, 0, 128, 64, 2)
    q = torch.zeros(1, 4, 128, dtype=torch.float16, device="cuda")
    with pytest.raises(tq.TQError) as ei:
        tq.tq_decode_attn_workspace_size(ti.Format(64, 4, 4, 0, 128, 64, 2), 1, 4, 4, 0)
    assert ei.value.status == 2
    with pytest.raises(tq.TQError) as ei:
        tq.tq_decode_attn_workspace_size(fmt, 1, 3, 4, 0)  # Hq not a multiple of H
    assert ei.value.status == 1
    ws_need = tq.tq_decode_attn_workspace_size(fmt, 1, 4, 4, 0)
    small = torch.empty(ws_need - 256, dtype=torch.uint8, device="cuda")
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    cb = tq.device_codebook(4)
    s = torch.zeros(128, dtype=torch.uint8, device="cuda")
    pool = torch.zeros(4 * tq.tq_page_layout(fmt)["page_bytes"], dtype=torch.uint8, device="cuda")
    out = torch.empty(1, 4, 128, device="cuda")
    bt = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    with pytest.raises(tq.TQError) as ei:
        tq.tq_decode_attn(fmt, q, pool, 4, bt, z, None, None, None, s, s, cb, cb, None, out, small)
    assert ei.value.status == 6


@pytest.mark.parametrize("kb,vb,qjl,W,kmix", [(4, 4, 0, 8, 0), (3, 4, 1, 8, 0), (2, 2, 1, 5, 0), (4, 4, 0, 0, 0), (3, 4, 0, 8, 1)])
def test_append_window_matches_oracle(kb, vb, qjl, W, kmix):
    """Window roll plus encode of the leaving token, from mixed initial states
    (empty, partial, full at several ring heads, a missing page), stepped on
    both sides: windows and counters identical, pages field by field."""
    fmt = ti.Format(128, kb, vb, qjl, 128, 16, 4, k_mixed=kmix)
    d, H, P = fmt.head_dim, fmt.num_kv_heads, fmt.page_size
    B, steps = 5, 30
    rng = np.random.default_rng(kb * 100 + vb * 10 + W)
    max_pages = 8
    num_pages = B * max_pages + 2
    bt = rng.permutation(num_pages)[: B * max_pages].astype(np.int32).reshape(B, max_pages)
    bt[4, 2] = -1  # sequence 4 runs out of pages at compressed position 32
    comp = np.array([0, 5, 7, 16, 20], np.int32)
    lens = np.array([0, 3, W, W, W], np.int32) if W else None
    head = np.array([0, 0, 5 % max(W, 1), 0, 2 % max(W, 1)], np.int32) if W else None
    kw = (rng.standard_normal((B, H, W, d)) * 3).astype(np.float16) if W else None
    vw = (rng.standard_normal((B, H, W, d)) * 3).astype(np.float16) if W else None
    K = ti.kv_history(steps, B, H, d, 3, 0).numpy()  # [steps, B, H, d]
    V = ti.kv_history(steps, B, H, d, 3, 1).numpy()
    lay = oracle.page_layout(fmt)
    pool_ref = np.full(num_pages * lay["page_bytes"], 0x5A, np.uint8)
    kcb, vcb = oracle.kind_codebook(fmt, 0), oracle.kind_codebook(fmt, 1)
    ks, vs = ti.sign_bits(ti.SEED_SIGNS_K, d), ti.sign_bits(ti.SEED_SIGNS_V, d)
    S = ti.gaussian_matrix(ti.SEED_QJL, fmt.qjl_m, d) if qjl else None

    dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    g_kw, g_vw, g_lens, g_head, g_comp, g_bt = dev(kw), dev(vw), dev(lens), dev(head), dev(comp), dev(bt)
    g_pool = torch.full((pool_ref.size,), 0x5A, dtype=torch.uint8, device="cuda")
    g_ks, g_vs, g_S = dev(ks), dev(vs), dev(S)
    ws = torch.empty(tq.tq_append_window_workspace_size(fmt, B), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    evicted, skipped_any = [], set()
    for t in range(steps):
        tq.tq_append_window(fmt, dev(K[t]), dev(V[t]), g_kw, g_vw, g_lens, g_head, g_comp, g_bt, g_pool, num_pages, g_ks, g_vs,
                            tq.kind_codebook(fmt, 0), tq.kind_codebook(fmt, 1), g_S, workspace=ws, err_word=err)
        sk = oracle.append_window(fmt, K[t], V[t], kw, vw, lens, head, comp, bt, pool_ref, num_pages, ks, vs, kcb, vcb, S,
                                  evicted=evicted)
        skipped_any |= set(sk)
    torch.cuda.synchronize()
    assert skipped_any == {4}
    assert int(err.item()) == tq.TQ_DEVERR_PAGE_RANGE
    assert np.array_equal(g_comp.cpu().numpy(), comp)
    if W:
        assert np.array_equal(g_lens.cpu().numpy(), lens) and np.array_equal(g_head.cpu().numpy(), head)
        assert np.array_equal(g_kw.cpu().numpy(), kw) and np.array_equal(g_vw.cpu().numpy(), vw)
    _check_append_pages(fmt, g_pool.cpu().numpy(), pool_ref, lay, evicted, num_pages, ks, vs, kcb, vcb, S)


def _check_append_pages(fmt, pool, pool_ref, lay, evicted, num_pages, ks, vs, kcb, vcb, S):
    """Pages after appends: the evicted tokens, field by field against a direct
    oracle encode of them (each kind in its own pass)."""
    from tq_testlib import merge_bits, written_mask
    slots = np.array([e[1] for e in evicted], np.int32)
    assert len(slots) > 0
    for kind in (0, 1):
        X = np.stack([e[2 + kind] for e in evicted])
        scratch = np.zeros_like(pool_ref)
        rc, _, cm, sm = oracle.encode(fmt, kind, X, slots, scratch, num_pages, ks if kind == 0 else vs,
                                      *(kcb if kind == 0 else vcb), S if kind == 0 else None, diagnostics=True)
        assert rc == 0
        other = written_mask(len(pool_ref), lay, fmt, 1 - kind, slots)
        pg = merge_bits(pool, pool_ref, other)  # the other kind is checked in its own pass
        compare_encoded(pg, pool_ref, lay, fmt, kind, slots, cm, sm)


@pytest.mark.parametrize("B,H,W,kb,vb,qjl", [(400, 4, 8, 4, 4, 0), (301, 2, 0, 3, 2, 1), (3, 128, 4, 4, 3, 1), (2, 64, 6, 2, 4, 0)])
def test_append_window_block_shapes(B, H, W, kb, vb, qjl):
    """The append's block shapes: several sequences per block (more sequences
    than SMs), a shorter last block, and the largest head counts (one
    sequence of 64 or 128 heads per block, QJL matrix and both token buffers
    in shared memory).  Random initial states; all pages valid."""
    fmt = ti.Format(128, kb, vb, qjl, 128, 16, H)
    d, P = fmt.head_dim, fmt.page_size
    steps = 6
    rng = np.random.default_rng(B * 7 + H)
    max_pages = 4
    num_pages = B * max_pages
    bt = rng.permutation(num_pages).astype(np.int32).reshape(B, max_pages)
    comp = rng.integers(0, max_pages * P - steps, B).astype(np.int32)
    lens = np.where(rng.random(B) < 0.6, W, rng.integers(0, W + 1, B)).astype(np.int32) if W else None
    head = (rng.integers(0, W, B) * (lens == W)).astype(np.int32) if W else None
    kw = (rng.standard_normal((B, H, W, d)) * 3).astype(np.float16) if W else None
    vw = (rng.standard_normal((B, H, W, d)) * 3).astype(np.float16) if W else None
    K = ti.kv_history(steps, B, H, d, 3, 0).numpy()
    V = ti.kv_history(steps, B, H, d, 3, 1).numpy()
    lay = oracle.page_layout(fmt)
    pool_ref = np.full(num_pages * lay["page_bytes"], 0x5A, np.uint8)
    kcb, vcb = oracle.kind_codebook(fmt, 0), oracle.kind_codebook(fmt, 1)
    ks, vs = ti.sign_bits(ti.SEED_SIGNS_K, d), ti.sign_bits(ti.SEED_SIGNS_V, d)
    S = ti.gaussian_matrix(ti.SEED_QJL, fmt.qjl_m, d) if qjl else None
    dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    g_kw, g_vw, g_lens, g_head, g_comp, g_bt = dev(kw), dev(vw), dev(lens), dev(head), dev(comp), dev(bt)
    g_pool = torch.full((pool_ref.size,), 0x5A, dtype=torch.uint8, device="cuda")
    g_ks, g_vs, g_S = dev(ks), dev(vs), dev(S)
    assert tq.tq_append_window_workspace_size(fmt, B) == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    evicted = []
    for t in range(steps):
        tq.tq_append_window(fmt, dev(K[t]), dev(V[t]), g_kw, g_vw, g_lens, g_head, g_comp, g_bt, g_pool, num_pages, g_ks, g_vs,
                            tq.kind_codebook(fmt, 0), tq.kind_codebook(fmt, 1), g_S, err_word=err)
        assert oracle.append_window(fmt, K[t], V[t], kw, vw, lens, head, comp, bt, pool_ref, num_pages, ks, vs, kcb, vcb, S,
                                    evicted=evicted) == []
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(g_comp.cpu().numpy(), comp)
    if W:
        assert np.array_equal(g_lens.cpu().numpy(), lens) and np.array_equal(g_head.cpu().numpy(), head)
        assert np.array_equal(g_kw.cpu().numpy(), kw) and np.array_equal(g_vw.cpu().numpy(), vw)
    _check_append_pages(fmt, g_pool.cpu().numpy(), pool_ref, lay, evicted, num_pages, ks, vs, kcb, vcb, S)


@pytest.mark.parametrize("kind,qjl", [(0, 1), (1, 0)])
def test_encode_non_finite_vector_is_a_zero_block(kind, qjl):
    """A head vector with an infinite or NaN coordinate is stored as a zero
    block (codes, signs and gamma 0) with its non-finite norm; the other
    vectors are unaffected."""
    from tq_testlib import unpack_field
    fmt = ti.Format(128, 4, 4, qjl, 128, 64, 4)
    d, H = fmt.head_dim, fmt.num_kv_heads
    N = 24
    lay = oracle.page_layout(fmt)
    x = ti.kv_history(1, N, H, d, 2, kind)[0].clone()
    bad = [(3, 1), (7, 2), (9, 0)]
    x[3, 1, 5] = float("inf")
    x[7, 2, :] = float("nan")
    x[9, 0, 0] = float("-inf")
    slots = torch.arange(N, dtype=torch.int32)
    signs = torch.from_numpy(ti.sign_bits(ti.SEED_SIGNS_K if kind == 0 else ti.SEED_SIGNS_V, d)).cuda()
    S = torch.from_numpy(ti.gaussian_matrix(ti.SEED_QJL, 128, d)).cuda() if qjl else None
    pools = []
    for xs in (x, torch.where(torch.isfinite(x), x, torch.zeros_like(x))):
        pool = torch.full((2 * lay["page_bytes"],), 0x77, dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        tq.tq_encode(fmt, kind, xs.cuda(), slots.cuda(), pool, 2, signs, tq.device_codebook(4), S, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        pools.append(pool.cpu().numpy())
    n, g, c, s = unpack_field(pools[0], lay, fmt, kind, slots.numpy())
    n2, g2, c2, s2 = unpack_field(pools[1], lay, fmt, kind, slots.numpy())
    good = np.ones((N, H), bool)
    for t, h in bad:
        good[t, h] = False
        assert not np.isfinite(n[t, h])
        assert np.all(c[t, h] == 0)
        if qjl:
            assert g[t, h] == 0 and np.all(s[t, h] == 0)
    assert np.array_equal(n[good], n2[good]) and np.array_equal(c[good], c2[good])
    if qjl:
        assert np.array_equal(g[good], g2[good]) and np.array_equal(s[good], s2[good])


def _random_attention_cases(n=24, seed=2024):
    """Seeded random formats and shapes: every key width (uniform and mixed),
    value width, QJL on/off, page sizes, GQA groups 1..8, ragged lengths,
    windows from none to several chunks."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        kmix = int(rng.random() < 0.3)
        kb = int(rng.choice([2, 3])) if kmix else int(rng.choice([2, 3, 4]))
        vb = int(rng.choice([2, 3, 4]))
        qjl = int(rng.random() < 0.4)
        P = int(rng.choice([16, 32, 48, 64, 128]))
        H = int(rng.choice([1, 2, 4]))
        G = int(rng.integers(1, 9))
        B = int(rng.integers(1, 5))
        W = int(rng.choice([0, 8, 40, 100]))
        comp = [int(x) for x in rng.integers(0, 700, B)]
        wl = [int(rng.integers(0, W + 1)) for _ in range(B)]
        fmt = ti.Format(128, kb, vb, qjl, 128, P, H, k_mixed=kmix)
        cases.append((f"r{i}_k{kb}{'m' if kmix else ''}v{vb}q{qjl}_p{P}_h{H}g{G}_b{B}_w{W}", fmt, B, H * G, comp, W, wl))
    return cases


@pytest.mark.parametrize("case", _random_attention_cases(), ids=lambda c: c[0])
def test_attention_random_formats_match_oracle(case):
    name, fmt, B, Hq, comp, W, wl = case
    sc = Scenario(fmt, B, Hq, comp, W, wl, layer=7)
    dev = sc.device_inputs()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_attention(sc, dev, err=err)
    rc, ref = sc.oracle_attention()
    assert rc == 0 and int(err.item()) == 0
    e = rel_err(out, ref)
    assert np.all(np.isfinite(out))
    assert e.max() <= REL_ATTN, (name, e.max())


def _random_encode_cases(n=16, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        kind = int(rng.integers(0, 2))
        kmix = int(kind == 0 and rng.random() < 0.35)
        bits = int(rng.choice([2, 3])) if kmix else int(rng.choice([2, 3, 4]))
        qjl = int(kind == 0 and rng.random() < 0.5)
        nc = int(rng.random() < 0.25 and not qjl)
        P = int(rng.choice([16, 32, 48, 64, 128]))
        H = int(rng.choice([1, 2, 3, 8]))
        N = int(rng.integers(1, 400))
        fmt = ti.Format(128, bits, bits, qjl, 128, P, H, norm_correct=nc, k_mixed=kmix)
        out.append((f"e{i}_kind{kind}_b{bits}{'m' if kmix else ''}_q{qjl}_nc{nc}_p{P}_h{H}_n{N}", fmt, kind, N, 1000 + i))
    return out


@pytest.mark.parametrize("case", _random_encode_cases(), ids=lambda c: c[0])
def test_encode_random_formats_match_oracle(case):
    name, fmt, kind, N, seed = case
    zero = (N // 2,) if N > 2 else ()
    neg = (N - 1,) if N > 3 else ()
    pool, pool_ref, lay, slots, cm, sm, *_ = _encode_case(fmt, kind, N, seed=seed, zero_rows=zero, neg_slots=neg)
    compare_encoded(pool, pool_ref, lay, fmt, kind, slots, cm, sm)


@pytest.mark.parametrize("vb,H", [(4, 1), (4, 3), (2, 2)])
def test_encode_value_pairs_every_store_path(vb, H):
    """2- and 4-bit value codes share bytes between the tokens of an offset
    pair (2p, 2p+1).  Two calls whose slots take every store path: pairs in
    order (one store of both tokens' words), reversed and misaligned pairs,
    a pair split over two pages, a live token whose partner is skipped, a
    lone last token, partners that arrive in the second call, and tokens the
    second call overwrites.  The pool after both calls equals the oracle's
    after the same two calls (codes up to the boundary exemption), and no
    bit outside the written codes changes."""
    fmt = ti.Format(128, 4, vb, 0, 128, 64, H)
    d, P = 128, 64
    num_pages = 4
    A, Bp = 1 * P, 3 * P  # slot bases of pages 1 and 3
    s1 = ([A + i for i in range(20)]            # in order: pairs (0,1) .. (18,19)
          + [A + 33, A + 32]                    # a reversed pair
          + [A + 41, A + 42, A + 43, A + 44]    # misaligned: no two neighbours are partners
          + [Bp + 2, A + 3 + 60]                # neighbours on different pages
          + [A + 50, -1]                        # live token, skipped neighbour
          + [A + 52])                           # lone last token (odd count)
    s2 = [A + 51, A + 53, A + 0, A + 7, Bp + 3]  # partners of earlier tokens, overwrites of 0 and 7
    lay = oracle.page_layout(fmt)
    signs = ti.sign_bits(ti.SEED_SIGNS_V, d)
    c, t = oracle.kind_codebook(fmt, 1)
    x1 = ti.kv_history(1, len(s1), H, d, 3, 1)[0].numpy()
    x2 = ti.kv_history(1, len(s2), H, d, 4, 1)[0].numpy()
    s1, s2 = np.array(s1, np.int32), np.array(s2, np.int32)
    pool_ref = np.full(num_pages * lay["page_bytes"], 0xA5, np.uint8)
    r1 = oracle.encode(fmt, 1, x1, s1, pool_ref, num_pages, signs, c, t, diagnostics=True)
    r2 = oracle.encode(fmt, 1, x2, s2, pool_ref, num_pages, signs, c, t, diagnostics=True)
    assert r1[0] == 0 and r2[0] == 0
    pool = torch.full((num_pages * lay["page_bytes"],), 0xA5, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cb = tq.kind_codebook(fmt, 1)
    for x, s in ((x1, s1), (x2, s2)):
        tq.tq_encode(fmt, 1, torch.from_numpy(x).cuda(), torch.from_numpy(s).cuda(), pool, num_pages,
                     torch.from_numpy(signs).cuda(), cb, None, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    keep = ~np.isin(s1, s2)  # the final writer of each slot
    slots = np.concatenate([s1[keep], s2])
    cm = np.concatenate([r1[2][keep], r2[2]])
    st = compare_encoded(pool.cpu().numpy(), pool_ref, lay, fmt, 1, slots, cm, None)
    print("pairs", vb, H, st)
