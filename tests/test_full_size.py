"""Parity at the full sizes of the five workloads, in the launch
configuration the benchmark times (the benchmark's own cache builder and call
sequence, one layer), on sampled outputs the oracle computes one by one:

* decode attention: the GPU output of sampled (sequence, query head) rows
  against the oracle's exact-softmax attention over the same packed pool,
  window and query;
* encode: sampled tokens (first and last of pages and of the sequence,
  plus random ones) re-encoded by the oracle into a copy of the GPU pool and
  compared field by field.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import tq_inputs as ti
from tq_testlib import REL_ATTN, check_exemption_reach, compare_encoded, merge_stats, rel_err

pytestmark = pytest.mark.gpu


def _sample_positions(comp, P, rng, n_random=6):
    pos = {0, P - 1, P, comp - 2, comp - 1, comp // 2}
    pos |= set(int(x) for x in rng.integers(0, comp, n_random))
    return sorted(p for p in pos if 0 <= p < comp)


def _check_encode_samples(fmt, kind, x_dev, slots_dev, pool_host, num_pages, pick, rng_name):
    """x_dev [N, H, d] fp16 (device), slots [N]; re-encode rows `pick` with the oracle."""
    lay = oracle.page_layout(fmt)
    d = fmt.head_dim
    x = x_dev[pick].cpu().numpy()
    slots = slots_dev[pick].cpu().numpy().astype(np.int32)
    signs = ti.sign_bits(ti.SEED_SIGNS_K if kind == 0 else ti.SEED_SIGNS_V, d)
    c, t = oracle.kind_codebook(fmt, kind)
    S = ti.gaussian_matrix(ti.SEED_QJL, fmt.qjl_m, d) if (kind == 0 and fmt.k_qjl) else None
    ref = pool_host.copy()
    rc, _, cm, sm = oracle.encode(fmt, kind, x, slots, ref, num_pages, signs, c, t, S, diagnostics=True)
    assert rc == 0
    stats = compare_encoded(pool_host, ref, lay, fmt, kind, slots, cm, sm)
    assert stats["codes"] > 0, rng_name
    return stats


@pytest.mark.parametrize("wl", ti.DECODE_WORKLOADS, ids=[w.name for w in ti.DECODE_WORKLOADS])
def test_decode_workload_full_size(wl):
    import bench
    import decode_attention_tq_gb300 as tq

    two = dataclasses.replace(wl, layers=min(wl.layers, 2))  # at least two layers, as the benchmark builds them
    b = bench.DecodeBench(two, "cuda")
    f = b.fmt
    B, Hq, H, d = b.B, b.Hq, b.H, f.head_dim
    kc, _ = oracle.kind_codebook(f, 0)
    vc, _ = oracle.kind_codebook(f, 1)
    S = b.S.cpu().numpy() if b.S is not None else None
    for li, L in enumerate(b.layers):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
        tq.tq_decode_attn(f, L["q"], L["pool"], b.num_pages, b.bt, b.comp_lens, L["kwin"], L["vwin"], b.win_lens if b.W else None,
                          b.ks, b.vs, b.kcb, b.vcb, b.S, out, b.ws, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = out.cpu().numpy()
        assert np.isfinite(got).all()

        # sampled rows through the oracle, on the very same pool / window / query
        pool = L["pool"].cpu().numpy()
        rows = sorted({0, Hq - 1, (B - 1) * Hq, B * Hq - 1, (B // 2) * Hq + Hq // 2 + 1 + li})
        rc, ref = oracle.attention(f, L["q"].cpu().numpy(), pool, b.num_pages, b.bt.cpu().numpy(), b.comp_lens.cpu().numpy(),
                                   L["kwin"].cpu().numpy() if b.W else None, L["vwin"].cpu().numpy() if b.W else None,
                                   b.win_lens.cpu().numpy(), b.ks.cpu().numpy(), b.vs.cpu().numpy(), kc, vc, S, heads=rows)
        assert rc == 0
        e = rel_err(got.reshape(B * Hq, d)[rows], ref)
        assert e.max() <= REL_ATTN, (wl.name, li, e)

        # sampled tokens of this layer's cache, re-encoded by the oracle
        rng = np.random.default_rng(5 + li)
        comp, P = b.comp, f.page_size
        totals = {0: {}, 1: {}}
        slots_all = b.bt[:, torch.arange(comp, device="cuda") // P] * P + (torch.arange(comp, device="cuda") % P)[None, :]
        for kind in (0, 1):
            x = ti.kv_history(B, wl.context, H, d, li, kind, device="cuda")[:, :comp]  # [B, comp, H, d]
            for bb in sorted({0, B - 1}):
                pick = _sample_positions(comp, P, rng)
                merge_stats(totals[kind], _check_encode_samples(f, kind, x[bb], slots_all[bb].to(torch.int32), pool, b.num_pages,
                                                                pick, f"{wl.name} layer {li} b{bb}"))
            del x
            check_exemption_reach(totals[kind], f"{wl.name} layer {li} kind {kind}")
    del b
    torch.cuda.empty_cache()


@pytest.mark.parametrize("bits", (2, 3, 4))
@pytest.mark.parametrize("qjl", (0, 1))
def test_bulk_encode_full_size(bits, qjl):
    """One layer of the bulk-encode workload (65536 tokens x 8 heads, K and V)
    with the benchmark's slot mapping; sampled tokens against the oracle."""
    import decode_attention_tq_gb300 as tq

    wl = ti.BULK_ENCODE_64K
    H, d, N, P = wl.kv_heads, 128, wl.tokens, wl.page_size
    fmt = ti.Format(d, bits, bits, qjl, wl.qjl_m, P, H)
    num_pages = N // P
    perm = ti.page_permutation(num_pages).to("cuda")
    pos = torch.arange(N, device="cuda")
    slots = (perm[pos // P] * P + pos % P).to(torch.int32).contiguous()
    lay = tq.tq_page_layout(fmt)
    S = torch.from_numpy(ti.gaussian_matrix(ti.SEED_QJL, wl.qjl_m, d)).to("cuda")
    cb = tq.device_codebook(bits, "cuda")
    rng = np.random.default_rng(11)
    for kind in (0, 1):
        x = ti.kv_history(1, N, H, d, 0, kind, device="cuda")[0].contiguous()
        pool = torch.full((num_pages * lay["page_bytes"],), 0xA5, dtype=torch.uint8, device="cuda")
        signs = torch.from_numpy(ti.sign_bits(ti.SEED_SIGNS_K if kind == 0 else ti.SEED_SIGNS_V, d)).to("cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        tq.tq_encode(fmt, kind, x, slots, pool, num_pages, signs, cb, S if (kind == 0 and qjl) else None, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        pick = _sample_positions(N, P, rng, n_random=120)
        st = _check_encode_samples(fmt, kind, x, slots, pool.cpu().numpy(), num_pages, pick, f"b{bits} qjl{qjl} kind{kind}")
        check_exemption_reach(st, f"bulk encode b{bits} qjl{qjl} kind {kind}")


@pytest.mark.parametrize("wl", ti.KIVI_WORKLOADS, ids=[w.name for w in ti.KIVI_WORKLOADS])
def test_kivi_workload_full_size(wl):
    """The KIVI control arm at the Llama-3-8B decode shape (two layers, the
    benchmark's own cache builder): sampled attention rows against the
    oracle over the same pool, and sampled page groups / tokens re-encoded by
    the oracle byte for byte."""
    import bench
    import decode_attention_tq_gb300 as tq

    two = dataclasses.replace(wl, layers=2)
    b = bench.KiviDecodeBench(two, "cuda")
    f = b.fmt
    B, Hq, H, d, P = b.B, b.Hq, b.H, f.head_dim, f.page_size
    lay = oracle.kivi_layout(f)
    for li, L in enumerate(b.layers):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
        tq.tq_kivi_decode_attn(f, L["q"], L["pool"], b.num_pages, b.bt, b.comp_lens, L["kwin"], L["vwin"], b.win_lens, out, b.ws,
                               err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        pool = L["pool"].cpu().numpy()
        rows = sorted({0, Hq - 1, (B - 1) * Hq, B * Hq - 1, (B // 2) * Hq + 3 + li})
        rc, ref = oracle.kivi_attention(f, L["q"].cpu().numpy(), pool, b.num_pages, b.bt.cpu().numpy(), b.comp_lens.cpu().numpy(),
                                        L["kwin"].cpu().numpy(), L["vwin"].cpu().numpy(), b.win_lens.cpu().numpy(), heads=rows)
        assert rc == 0
        e = rel_err(got.reshape(B * Hq, d)[rows], ref)
        print(wl.name, li, "max rel err", e.max())
        assert e.max() <= REL_ATTN, (wl.name, li, e)
        # sampled page groups (keys) and tokens (values) re-encoded by the oracle
        rng = np.random.default_rng(7 + li)
        bt = b.bt.cpu().numpy()
        for kind in (0, 1):
            x = ti.kv_history(B, wl.context, H, d, li, kind, device="cuda")
            for bb in sorted({0, B - 1}):
                ref_pool = pool.copy()
                if kind == 0:
                    for g in sorted({0, b.pages_per_seq - 1, int(rng.integers(0, b.pages_per_seq))}):
                        xs = x[bb, g * P:(g + 1) * P].cpu().numpy()
                        assert oracle.kivi_encode_keys(f, xs, bt[bb, g:g + 1], ref_pool, b.num_pages) == 0
                else:
                    pick = _sample_positions(b.comp, P, rng)
                    xs = x[bb, pick].cpu().numpy()
                    sl = (bt[bb, np.array(pick) // P] * P + np.array(pick) % P).astype(np.int32)
                    assert oracle.kivi_encode_values(f, xs, sl, ref_pool, b.num_pages) == 0
                assert np.array_equal(ref_pool, pool), (wl.name, li, kind, bb)
            del x
    del b
    torch.cuda.empty_cache()
