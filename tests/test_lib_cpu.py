"""CPU-side checks of libtq.so: it builds, loads, exports every entry point the
header declares, and its host-only functions agree with the oracle.  No CUDA
device is needed; nothing here launches a kernel."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
import tq_inputs as ti

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from decode_attention_tq_gb300 import build, tq

    build.build()
    return tq.load_library()


def header_functions():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert {"tq_make_codebook", "tq_encode", "tq_decode", "tq_decode_attn", "tq_decode_attn_workspace_size",
            "tq_page_layout", "tq_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5])
def test_codebook_equals_oracle(lib, bits):
    from decode_attention_tq_gb300 import tq_make_codebook

    c, t = tq_make_codebook(bits)
    c2, t2 = oracle.make_codebook(bits)
    assert np.array_equal(c, c2) and np.array_equal(t, t2)


@pytest.mark.parametrize("fmt", [ti.Format(128, b, v, q, 128, P, H) for b in (2, 3, 4) for v in (2, 4) for q in (0, 1) for P in (16, 64, 128)
                                 for H in (1, 8)] + [ti.Format(64, 3, 5, 1, 24, 48, 3), ti.Format(16, 1, 2, 0, 8, 16, 1)]
                         + [ti.Format(128, b, 4, q, 128, 64, 8, k_mixed=1) for b in (1, 2, 3, 7) for q in (0, 1)])
def test_layout_equals_oracle(lib, fmt):
    from decode_attention_tq_gb300 import tq_page_layout

    assert tq_page_layout(fmt) == oracle.page_layout(fmt)


def test_status_strings(lib):
    from decode_attention_tq_gb300 import tq_status_string

    for s in range(7):
        assert len(tq_status_string(s)) >= 2
    assert tq_status_string(99) == "unknown status"


def _F(**kw):
    from decode_attention_tq_gb300.tq import tq_format

    f = dict(head_dim=128, k_bits=4, v_bits=4, k_qjl=0, qjl_m=128, page_size=64, num_kv_heads=8)
    f.update(kw)
    return tq_format(**f)


def test_host_validation_before_any_launch(lib):
    P = C.c_void_p
    dummy = P(4096)  # never dereferenced: every call below fails its host checks first
    f = _F()
    # null / malformed format
    assert lib.tq_encode(None, 0, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    assert lib.tq_encode(C.byref(_F(head_dim=100)), 0, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    # a valid format the kernels do not implement
    assert lib.tq_encode(C.byref(_F(head_dim=64)), 0, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 2
    assert lib.tq_encode(C.byref(_F(k_bits=5)), 0, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 2
    assert lib.tq_encode(C.byref(_F(qjl_m=64, k_qjl=1)), 0, dummy, 1, dummy, dummy, 1, dummy, dummy, dummy, None, None) == 2
    # pages are whole 16-token groups
    assert lib.tq_encode(C.byref(_F(page_size=24)), 0, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    # bad kind, negative count, missing S for QJL keys, misaligned input
    assert lib.tq_encode(C.byref(f), 2, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    assert lib.tq_encode(C.byref(f), 0, dummy, -1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    assert lib.tq_encode(C.byref(_F(k_qjl=1)), 0, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    assert lib.tq_encode(C.byref(f), 0, P(4098), 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    # format variants: norm correction and the QJL factor are validated; the
    # GPU encode of QJL keys has no norm correction
    assert lib.tq_encode(C.byref(_F(norm_correct=2)), 1, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    assert lib.tq_encode(C.byref(_F(qjl_scale=-1.0)), 1, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    assert lib.tq_encode(C.byref(_F(qjl_scale=float("nan"))), 1, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    assert lib.tq_encode(C.byref(_F(k_qjl=1, norm_correct=1)), 0, dummy, 1, dummy, dummy, 1, dummy, dummy, dummy, None, None) == 2
    assert lib.tq_encode(C.byref(_F(k_qjl=1, norm_correct=1)), 1, dummy, 0, dummy, dummy, 1, dummy, dummy, None, None, None) == 0
    # mixed-rate keys: 3.5 and 2.5 bits run on the GPU, 4.5 does not; 8.5 is not a format
    assert lib.tq_encode(C.byref(_F(k_bits=4, k_mixed=1)), 0, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 2
    assert lib.tq_encode(C.byref(_F(k_bits=8, k_mixed=1)), 0, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    assert lib.tq_encode(C.byref(_F(k_mixed=3)), 0, dummy, 1, dummy, dummy, 1, dummy, dummy, None, None, None) == 1
    assert lib.tq_encode(C.byref(_F(k_bits=3, k_mixed=1)), 0, dummy, 0, dummy, dummy, 1, dummy, dummy, None, None, None) == 0
    # append: window buffers and counters are required with a window
    assert lib.tq_append_window(C.byref(f), 2, dummy, dummy, None, None, 8, None, None, dummy, dummy, 4, dummy, 4, dummy, dummy,
                                dummy, dummy, None, dummy, 1 << 20, None, None) == 1
    # a block holds one sequence's tokens: more than 128 kv heads are not supported
    assert lib.tq_append_window(C.byref(_F(num_kv_heads=129)), 2, dummy, dummy, None, None, 0, None, None, dummy, dummy, 4,
                                dummy, 4, dummy, dummy, dummy, dummy, None, None, 0, None, None) == 2
    # page slots are int32: a pool of more than 2^31 slots is not supported
    assert lib.tq_append_window(C.byref(f), 2, dummy, dummy, None, None, 0, None, None, dummy, dummy, 4, dummy,
                                (1 << 31) // 64 + 1, dummy, dummy, dummy, dummy, None, dummy, 1 << 20, None, None) == 2
    n_ws = C.c_size_t(0)
    assert lib.tq_append_window_workspace_size(C.byref(f), 2, C.byref(n_ws)) == 0 and n_ws.value == 0  # staged in shared memory
    # zero tokens is a no-op success without touching the device
    assert lib.tq_encode(C.byref(f), 1, dummy, 0, dummy, dummy, 1, dummy, dummy, None, None, None) == 0
    assert lib.tq_decode(C.byref(f), 1, dummy, 1, dummy, 0, dummy, dummy, None, dummy, None, None) == 0
    # attention shape checks
    n = C.c_size_t(0)
    assert lib.tq_decode_attn_workspace_size(C.byref(f), 1, 12, 4, 0, C.byref(n)) == 1   # Hq % H
    assert lib.tq_decode_attn_workspace_size(C.byref(f), 1, 8 * 16, 4, 0, C.byref(n)) == 2  # G = 16 > 8
    assert lib.tq_decode_attn_workspace_size(C.byref(f), 0, 8, 4, 0, C.byref(n)) == 1
    assert lib.tq_decode_attn_workspace_size(C.byref(f), 1, 8, 4, -1, C.byref(n)) == 1
    assert lib.tq_decode_attn(C.byref(f), 1, 8, None, dummy, 4, dummy, 4, dummy, None, None, None, 0, dummy, dummy, dummy, dummy,
                              None, dummy, dummy, 1 << 20, None, None) == 1
    # window > 0 needs the window buffers
    assert lib.tq_decode_attn(C.byref(f), 1, 8, dummy, dummy, 4, dummy, 4, dummy, None, None, None, 16, dummy, dummy, dummy, dummy,
                              None, dummy, dummy, 1 << 20, None, None) == 1


@pytest.mark.parametrize("fmt", [ti.KiviFormat(128, kb, vb, P, H) for kb in (2, 4) for vb in (2, 4) for P in (16, 64, 128) for H in (1, 8)]
                         + [ti.KiviFormat(64, 3, 2, 32, 2), ti.KiviFormat(16, 1, 8, 16, 3)])
def test_kivi_layout_equals_oracle(lib, fmt):
    from decode_attention_tq_gb300 import tq_kivi_page_layout

    assert tq_kivi_page_layout(fmt) == oracle.kivi_layout(fmt)


def test_kivi_host_validation_before_any_launch(lib):
    from decode_attention_tq_gb300.tq import tq_kivi_format

    P = C.c_void_p
    dummy = P(4096)  # never dereferenced
    f = tq_kivi_format(128, 2, 2, 64, 8)
    assert lib.tq_kivi_encode_keys(None, dummy, 1, dummy, dummy, 1, None, None) == 1
    assert lib.tq_kivi_encode_keys(C.byref(tq_kivi_format(128, 2, 2, 24, 8)), dummy, 1, dummy, dummy, 1, None, None) == 1
    assert lib.tq_kivi_encode_keys(C.byref(tq_kivi_format(128, 3, 2, 64, 8)), dummy, 1, dummy, dummy, 1, None, None) == 2
    assert lib.tq_kivi_encode_values(C.byref(tq_kivi_format(64, 2, 2, 64, 8)), dummy, 1, dummy, dummy, 1, None, None) == 2
    assert lib.tq_kivi_encode_values(C.byref(f), dummy, -1, dummy, dummy, 1, None, None) == 1
    assert lib.tq_kivi_encode_values(C.byref(f), P(4098), 1, dummy, dummy, 1, None, None) == 1
    assert lib.tq_kivi_encode_values(C.byref(f), dummy, 0, dummy, dummy, 1, None, None) == 0  # no-op
    assert lib.tq_kivi_decode(C.byref(f), 2, dummy, 1, dummy, 1, dummy, None, None) == 1
    n = C.c_size_t(0)
    assert lib.tq_kivi_decode_attn_workspace_size(C.byref(f), 1, 12, 4, 0, C.byref(n)) == 1   # Hq % H
    assert lib.tq_kivi_decode_attn_workspace_size(C.byref(f), 1, 8 * 16, 4, 0, C.byref(n)) == 2  # G = 16 > 8
    assert lib.tq_kivi_decode_attn(C.byref(f), 1, 8, None, dummy, 4, dummy, 4, dummy, None, None, None, 0, dummy, dummy,
                                   1 << 20, None, None) == 1
    assert lib.tq_kivi_decode_attn(C.byref(f), 1, 8, dummy, dummy, 4, dummy, 4, dummy, None, None, None, 16, dummy, dummy,
                                   1 << 20, None, None) == 1  # window buffers missing


def test_device_error_bits_match_header():
    from decode_attention_tq_gb300 import tq

    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    bits = {m.group(1): int(m.group(2), 16) for m in re.finditer(r"#define (TQ_DEVERR_[A-Z_]+) 0x([0-9a-fA-F]+)", src)}
    assert set(bits) == {"TQ_DEVERR_SLOT_RANGE", "TQ_DEVERR_PAGE_RANGE", "TQ_DEVERR_LENGTH", "TQ_DEVERR_TIMEOUT"}
    for name, v in bits.items():
        assert getattr(tq, name) == v, name
    assert len(set(bits.values())) == len(bits) and all(v & (v - 1) == 0 for v in bits.values())
