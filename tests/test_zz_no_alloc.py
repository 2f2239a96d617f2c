"""tq_decode_attn_static: decode attention on the library's fixed scratch
buffer (no workspace, no allocation), for callers that cannot allocate.

Each case first runs a static call of a different shape, so the shared buffer
holds another call's finite leftovers, not the zeros a freshly loaded module
starts with.  Then two static calls in a row must give exactly the output of
tq_decode_attn with a torch workspace (the same kernels on the same plan,
with no atomics on the attention path, so bit for bit) and stay within the
attention tolerance of the fp64 oracle.

The file name sorts last so that a run which stops at the first failure has
already run every other test; it passes on its own too."""
import numpy as np
import pytest
import torch

import tq_inputs as ti
from tq_testlib import REL_ATTN, Scenario, gpu_attention, rel_err

pytestmark = pytest.mark.gpu

CASES = {
    "k4v4_g4_w": (ti.Format(128, 4, 4, 0, 128, 64, 4), 2, 16, [1000, 333], 32, [32, 7]),
    "k3qjl_v4_g8": (ti.Format(128, 3, 4, 1, 128, 64, 2), 2, 16, [640, 77], 0, [0, 0]),
}
# the shape whose leftovers each case starts from: other batch, lengths,
# heads and window, so every workspace section sits elsewhere
DIRTY = (ti.Format(128, 2, 3, 0, 128, 32, 3), 3, 6, [700, 41, 259], 48, [48, 3, 20])


def _static(sc, dev_in, err):
    import decode_attention_tq_gb300 as tq

    out = torch.full((sc.B, sc.Hq, sc.fmt.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    tq.tq_decode_attn_static(sc.fmt, dev_in["q"], dev_in["pool"], sc.num_pages, dev_in["bt"], dev_in["comp"], dev_in["kwin"],
                             dev_in["vwin"], dev_in["wl"], dev_in["ks"], dev_in["vs"], dev_in["kcb"], dev_in["vcb"], dev_in["S"],
                             out, err_word=err)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("name", list(CASES))
def test_static_scratch_matches_workspace_entry(name):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dirty = Scenario(*DIRTY)
    dirty_in = dirty.device_inputs()
    first = _static(dirty, dirty_in, err)
    assert int(err.item()) == 0 and np.isfinite(first).all()
    assert np.array_equal(first, gpu_attention(dirty, dirty_in))

    fmt, B, Hq, comp, W, wl = CASES[name]
    sc = Scenario(fmt, B, Hq, comp, W, wl)
    dev_in = sc.device_inputs()
    want = gpu_attention(sc, dev_in)  # tq_decode_attn with a torch workspace
    rc, ref = sc.oracle_attention()
    assert rc == 0
    for _ in range(2):  # two calls in a row on the same scratch
        got = _static(sc, dev_in, err)
        assert int(err.item()) == 0
        assert np.array_equal(got, want)
        assert rel_err(got, ref).max() <= REL_ATTN


def test_static_scratch_rejects_oversized_shapes():
    import decode_attention_tq_gb300 as tq

    fmt = ti.Format(128, 4, 4, 0, 128, 64, 8)
    B, Hq, max_pages, W = 512, 64, 64, 128
    assert tq.tq_decode_attn_workspace_size(fmt, B, Hq, max_pages, W) > tq.TQ_STATIC_SCRATCH_BYTES
    q = torch.zeros(B, Hq, 128, dtype=torch.float16, device="cuda")
    pool = torch.zeros(69632, dtype=torch.uint8, device="cuda")
    bt = torch.zeros(B, max_pages, dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    win = torch.zeros(B, 8, W, 128, dtype=torch.float16, device="cuda")
    signs = torch.zeros(128, dtype=torch.uint8, device="cuda")
    cb = tq.device_codebook(4, "cuda")
    out = torch.zeros(B, Hq, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attn_static(fmt, q, pool, 1, bt, lens, win, win, lens, signs, signs, cb, cb, None, out)
    assert e.value.status == 7  # TQ_ERR_SCRATCH_LIMIT, before any launch
