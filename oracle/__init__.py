"""fp64 CPU oracle for TurboQuant-style KV-cache compression (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package.  The
product path (``libtq.so`` and ``decode_attention_tq_gb300``) never imports it
and shares no code with it; this wrapper only marshals numpy arrays into the
plain C functions of ``oracle.c``, where every step of the method is written
out (see the header of ``oracle.c`` for the passages each function follows).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, library routines, brute force or values printed on the
pages; nothing in this oracle is "parity unpinned" except the conventions the
pages leave open (bit order, seeds), which are self-consistent by construction.
"""
from __future__ import annotations

import ctypes as C
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = (os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "kivi.c"))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c and kivi.c into liboracle.so with gcc (-O2, no
    fast-math, no floating-point contraction)."""
    newest = max(os.path.getmtime(p) for p in _SRCS)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, *_SRCS, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Format(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("head_dim", "k_bits", "v_bits", "k_qjl", "qjl_m", "page_size", "num_kv_heads",
                                         "norm_correct")] + [("qjl_scale", C.c_float), ("k_mixed", C.c_int32)]


class _Layout(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("slab_bytes", "page_bytes", "k_norm", "k_gamma", "k_codes", "k_signs", "v_norm", "v_codes")] + [
        (n, C.c_int32) for n in ("k_code_bytes", "k_sign_bytes", "v_code_bytes")
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = C.CDLL(_LIB_PATH)
            P = C.c_void_p
            i32, i64, dbl = C.c_int32, C.c_int64, C.c_double
            lib.orc_half_to_double.argtypes = [C.c_uint16]
            lib.orc_half_to_double.restype = dbl
            lib.orc_lloyd_max_f64.argtypes = [C.c_int, P, P]
            lib.orc_make_codebook.argtypes = [C.c_int, P, P]
            lib.orc_round_to_half.argtypes = [dbl]
            lib.orc_round_to_half.restype = dbl
            lib.orc_quantize_scalar.argtypes = [C.c_int, P, dbl]
            lib.orc_fwht.argtypes = [P, C.c_int]
            lib.orc_fwht.restype = None
            lib.orc_rotate.argtypes = [C.c_int, P, P, P]
            lib.orc_rotate.restype = None
            lib.orc_unrotate.argtypes = [C.c_int, P, P, P]
            lib.orc_unrotate.restype = None
            lib.orc_encode_vector.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int] + [P] * 12 + [C.c_int, dbl, C.c_int, P, P]
            lib.orc_decode_vector.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, dbl, dbl] + [P] * 6 + [dbl, C.c_int, P]
            lib.orc_pack_bits.argtypes = [C.c_int, C.c_int, P, P]
            lib.orc_pack_bits.restype = None
            lib.orc_unpack_bits.argtypes = [C.c_int, C.c_int, P, P]
            lib.orc_unpack_bits.restype = None
            lib.orc_page_layout.argtypes = [P, P]
            lib.orc_encode.argtypes = [P, C.c_int, P, i64, P, P, i64, P, P, P, P, P, P, P]
            lib.orc_decode.argtypes = [P, C.c_int, P, i64, P, i64, P, P, P, P]
            lib.orc_attention.argtypes = [P, C.c_int, C.c_int, P, P, i64, P, C.c_int, P, P, P, P, C.c_int, P, P, P, P, P, P, C.c_int, P]
            lib.orc_kivi_layout.argtypes = [P, P]
            lib.orc_kivi_quantize_group.argtypes = [C.c_int, P, i64, C.c_int, P, P, P]
            lib.orc_kivi_quantize_group.restype = None
            lib.orc_kivi_encode_keys.argtypes = [P, P, i64, P, P, i64]
            lib.orc_kivi_encode_values.argtypes = [P, P, i64, P, P, i64]
            lib.orc_kivi_decode.argtypes = [P, C.c_int, P, i64, P, i64, P]
            lib.orc_kivi_attention.argtypes = [P, C.c_int, C.c_int, P, P, i64, P, C.c_int, P, P, P, P, C.c_int, P, C.c_int, P]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else C.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _fmt(f) -> _Format:
    return _Format(int(f.head_dim), int(f.k_bits), int(f.v_bits), int(f.k_qjl), int(f.qjl_m), int(f.page_size), int(f.num_kv_heads),
                   int(getattr(f, "norm_correct", 0)), float(getattr(f, "qjl_scale", 0.0)), int(getattr(f, "k_mixed", 0)))


def _f16bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    if x.dtype == np.uint16:
        return x
    raise TypeError("expected float16 data")


# ------------------------------------------------------------------ scalar --
def half_to_double(bits: int) -> float:
    return _load().orc_half_to_double(int(bits))


def lloyd_max_f64(bits: int):
    """fp64 Lloyd-Max centroids [2^b] and midpoints [2^b-1] for N(0,1)."""
    c = np.zeros(256)
    t = np.zeros(256)
    it = _load().orc_lloyd_max_f64(bits, _ptr(c), _ptr(t))
    if it < 0:
        raise ValueError("bad bits")
    L = 1 << bits
    return c[:L].copy(), t[: L - 1].copy(), it


def kind_codebook(f, kind: int):
    """(centroids, midpoints) a kind of format f is encoded with: one
    codebook, or for mixed-rate keys the k_bits + 1 codebook followed by the
    k_bits one (the layout of the device codebooks)."""
    bits = int(f.k_bits if kind == 0 else f.v_bits)
    if kind == 0 and int(getattr(f, "k_mixed", 0)):
        ch, th = make_codebook(bits + 1)
        cl, tl = make_codebook(bits)
        return np.concatenate([ch, cl]).astype(np.float32), np.concatenate([th, tl]).astype(np.float32)
    return make_codebook(bits)


def round_to_half(x: float) -> float:
    """The nearest fp16 value of x (ties to even), as a float."""
    return _load().orc_round_to_half(float(x))


def make_codebook(bits: int):
    """The stored codebook as fp32 arrays: centroids [2^b] (the fp64 Lloyd-Max
    fixed point rounded to fp16) and thresholds [2^b-1] (exact midpoints of
    neighbouring stored centroids)."""
    L = 1 << bits
    c = np.zeros(L, np.float32)
    t = np.zeros(max(L - 1, 1), np.float32)
    it = _load().orc_make_codebook(bits, _ptr(c), _ptr(t))
    if it < 0:
        raise ValueError("bad bits")
    return c, t[: L - 1]


def quantize_scalar(bits: int, midpoints, u: float) -> int:
    m = _c(midpoints, np.float32)
    return _load().orc_quantize_scalar(bits, _ptr(m), float(u))


def fwht(x) -> np.ndarray:
    y = _c(x, np.float64).copy()
    _load().orc_fwht(_ptr(y), y.shape[-1])
    return y


def rotate(x, signs) -> np.ndarray:
    x = _c(x, np.float64)
    s = _c(signs, np.uint8)
    y = np.zeros_like(x)
    _load().orc_rotate(x.shape[-1], _ptr(s), _ptr(x), _ptr(y))
    return y


def unrotate(y, signs) -> np.ndarray:
    y = _c(y, np.float64)
    s = _c(signs, np.uint8)
    x = np.zeros_like(y)
    _load().orc_unrotate(y.shape[-1], _ptr(s), _ptr(y), _ptr(x))
    return x


# ------------------------------------------------------------------ vector --
def qjl_coef(qjl_m: int, qjl_scale: float = 0.0) -> float:
    """Factor of gamma S^T (2z - 1) in y_hat: qjl_scale, else the paper's sqrt(pi/2)/m."""
    return float(qjl_scale) if qjl_scale > 0 else math.sqrt(math.pi / 2) / qjl_m


def encode_vector(x, bits, signs, centroids, midpoints, S=None, qjl_m=0, norm_correct=0, qjl_scale=0.0, lo_codebook=None):
    """Encode one vector (fp64 values).  Returns a dict with norm, gamma, idx,
    z, u, code_margin, sign_margin.  With norm_correct the returned norm is
    ||x|| / ||y_hat|| (y_hat with the QJL factor of qjl_coef).  With
    lo_codebook = (centroids, midpoints) of bits - 1 the vector is mixed-rate:
    high channels ((j mod 16) < 8) use `bits`, the others bits - 1."""
    x = _c(x, np.float64)
    d = x.shape[0]
    qjl = S is not None
    m = int(qjl_m) if qjl else 0
    idx = np.zeros(d, np.int32)
    z = np.zeros(max(m, 1), np.uint8)
    u = np.zeros(d)
    cm = np.zeros(d)
    sm = np.zeros(max(m, 1))
    norm = C.c_double(0)
    gamma = C.c_double(0)
    Sa = _c(S, np.float32) if qjl else None
    rc = _load().orc_encode_vector(
        d, bits, int(qjl), m, _ptr(x), _ptr(_c(signs, np.uint8)), _ptr(_c(centroids, np.float32)),
        _ptr(_c(midpoints, np.float32)), _ptr(Sa), C.byref(norm), C.byref(gamma), _ptr(idx), _ptr(z), _ptr(u), _ptr(cm), _ptr(sm),
        int(norm_correct), qjl_coef(m, qjl_scale) if qjl else 0.0, int(lo_codebook is not None),
        _ptr(None if lo_codebook is None else _c(lo_codebook[0], np.float32)),
        _ptr(None if lo_codebook is None else _c(lo_codebook[1], np.float32)),
    )
    if rc != 0:
        raise ValueError(f"orc_encode_vector rc={rc}")
    return dict(norm=norm.value, gamma=gamma.value, idx=idx, z=z[:m], u=u, code_margin=cm, sign_margin=sm[:m])


def decode_vector(norm, idx, bits, signs, centroids, gamma=0.0, z=None, S=None, qjl_m=0, qjl_scale=0.0, lo_centroids=None):
    idx = _c(idx, np.int32)
    d = idx.shape[0]
    qjl = S is not None
    m = int(qjl_m) if qjl else 0
    out = np.zeros(d)
    za = _c(z, np.uint8) if qjl else None
    Sa = _c(S, np.float32) if qjl else None
    rc = _load().orc_decode_vector(
        d, bits, int(qjl), m, float(norm), float(gamma), _ptr(idx), _ptr(za), _ptr(_c(signs, np.uint8)),
        _ptr(_c(centroids, np.float32)), _ptr(Sa), _ptr(out), qjl_coef(m, qjl_scale) if qjl else 0.0,
        int(lo_centroids is not None), _ptr(None if lo_centroids is None else _c(lo_centroids, np.float32)),
    )
    if rc != 0:
        raise ValueError(f"orc_decode_vector rc={rc}")
    return out


def pack_bits(vals, b: int) -> np.ndarray:
    v = _c(vals, np.int32)
    out = np.zeros((v.shape[0] * b + 7) // 8, np.uint8)
    _load().orc_pack_bits(v.shape[0], b, _ptr(v), _ptr(out))
    return out


def unpack_bits(data, count: int, b: int) -> np.ndarray:
    d = _c(data, np.uint8)
    out = np.zeros(count, np.int32)
    _load().orc_unpack_bits(count, b, _ptr(d), _ptr(out))
    return out


# ------------------------------------------------------------------- paged --
def page_layout(f) -> dict:
    L = _Layout()
    F = _fmt(f)
    rc = _load().orc_page_layout(C.byref(F), C.byref(L))
    if rc != 0:
        raise ValueError("unsupported format for the oracle layout")
    return {n: getattr(L, n) for n, _ in _Layout._fields_}


def encode(f, kind: int, x, slot_mapping, pool, num_pages: int, signs, centroids, midpoints, S=None, diagnostics=False):
    """Encode x [N,H,d] fp16 into ``pool`` (uint8, modified in place).
    With ``diagnostics`` returns (rc, u, code_margin, sign_margin)."""
    xb = _f16bits(x)
    N = xb.shape[0]
    H, d = int(f.num_kv_heads), int(f.head_dim)
    m = int(f.qjl_m) if (kind == 0 and f.k_qjl) else 0
    u = cm = sm = None
    if diagnostics:
        u = np.zeros((N, H, d))
        cm = np.zeros((N, H, d))
        sm = np.zeros((N, H, max(m, 1)))
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"]
    F = _fmt(f)
    rc = _load().orc_encode(
        C.byref(F), kind, _ptr(xb), N, _ptr(_c(slot_mapping, np.int32)), _ptr(pool), int(num_pages), _ptr(_c(signs, np.uint8)),
        _ptr(_c(centroids, np.float32)), _ptr(_c(midpoints, np.float32)), _ptr(None if S is None else _c(S, np.float32)),
        _ptr(u), _ptr(cm), _ptr(sm),
    )
    if diagnostics:
        return rc, u, cm, (sm[..., :m] if m else None)
    return rc


def decode(f, kind: int, pool, num_pages: int, slot_mapping, signs, centroids, S=None):
    sl = _c(slot_mapping, np.int32)
    N = sl.shape[0]
    out = np.zeros((N, int(f.num_kv_heads), int(f.head_dim)))
    F = _fmt(f)
    rc = _load().orc_decode(
        C.byref(F), kind, _ptr(pool), int(num_pages), _ptr(sl), N, _ptr(_c(signs, np.uint8)), _ptr(_c(centroids, np.float32)),
        _ptr(None if S is None else _c(S, np.float32)), _ptr(out),
    )
    return rc, out


def attention(f, q, pool, num_pages, block_tables, comp_lens, k_win, v_win, win_lens, k_signs, v_signs, k_centroids, v_centroids,
              S=None, heads=None):
    """Exact-softmax decode attention over the compressed cache plus window.
    q [B,Hq,d] fp16; k_win/v_win [B,Hkv,W,d] fp16 or None.  ``heads``: optional
    list of b*Hq+qh; returns (rc, out) with out [B,Hq,d] or [len(heads),d]."""
    qb = _f16bits(q)
    B, Hq, d = qb.shape
    bt = _c(block_tables, np.int32)
    max_pages = bt.shape[1]
    if k_win is None:
        W = 0
        kw = vw = wl = None
    else:
        kw = _f16bits(k_win)
        vw = _f16bits(v_win)
        W = kw.shape[2]
        wl = _c(win_lens, np.int32)
    hs = None if heads is None else _c(heads, np.int32)
    n = B * Hq if hs is None else hs.shape[0]
    out = np.zeros((n, d))
    F = _fmt(f)
    rc = _load().orc_attention(
        C.byref(F), B, Hq, _ptr(qb), _ptr(pool), int(num_pages), _ptr(bt), max_pages, _ptr(_c(comp_lens, np.int32)), _ptr(kw), _ptr(vw),
        _ptr(wl), W, _ptr(_c(k_signs, np.uint8)), _ptr(_c(v_signs, np.uint8)), _ptr(_c(k_centroids, np.float32)),
        _ptr(_c(v_centroids, np.float32)), _ptr(None if S is None else _c(S, np.float32)), _ptr(hs), n, _ptr(out),
    )
    if hs is None:
        out = out.reshape(B, Hq, d)
    return rc, out


def append_window(f, k_new, v_new, k_win, v_win, win_lens, win_head, comp_lens, block_tables, pool, num_pages,
                  k_signs, v_signs, k_codebook, v_codebook, S=None, evicted=None):
    """One decode step's append into a cache made of compressed pages plus an
    fp16 recent window kept as a ring of W slots per sequence.

    Follows "TurboQuant Family Design Study for CPU and Browser WASM KV
    Caches": 'Packed format and complete bit accounting' (the most recent W
    tokens stay fp16 for K and V), 'Append cost and memory-bandwidth
    tradeoffs' (the append runs once per generated token, per layer and kv
    head: rotate, quantize, pack, store) and 'Paging, lifecycle, and cache
    identity' (fixed-size pages filled in order).  Per sequence b:

    * W == 0: the new token is encoded at compressed position comp_lens[b];
    * window not full (win_lens[b] < W): the new token goes to ring slot
      win_lens[b] and win_lens[b] grows by one (win_head stays 0);
    * window full: the oldest token, at ring slot win_head[b], is encoded at
      compressed position comp_lens[b], the new token takes its ring slot,
      win_head[b] advances by one modulo W.

    Compressed position c lives in physical page block_tables[b][c // P] at
    offset c % P; those pages are allocated by the caller.  A position whose
    page index reaches the table width or whose entry lies outside
    [0, num_pages) leaves that sequence untouched and is reported.

    k_new, v_new [B, H, d] fp16; k_win, v_win [B, H, W, d] fp16 (or None for
    W == 0); counters int32 [B]; all but the inputs are updated in place.
    Returns the list of sequences that were skipped.  With a list as
    ``evicted``, each token written to the pages is appended to it as
    (b, slot, k [H, d], v [H, d]).
    """
    B, H, d = k_new.shape
    P = int(f.page_size)
    W = 0 if k_win is None else int(k_win.shape[2])
    kc, kt = k_codebook
    vc, vt = v_codebook
    skipped = []
    for b in range(B):
        if W > 0 and win_lens[b] < W:
            k_win[b, :, win_lens[b]] = k_new[b]
            v_win[b, :, win_lens[b]] = v_new[b]
            win_lens[b] += 1
            continue
        c = int(comp_lens[b])
        pi = c // P
        page = int(block_tables[b, pi]) if pi < block_tables.shape[1] else -1
        if page < 0 or page >= num_pages:
            skipped.append(b)
            continue
        slot = np.array([page * P + c % P], np.int32)
        if W == 0:
            k_out, v_out = k_new[b], v_new[b]
        else:
            i = int(win_head[b])
            k_out, v_out = k_win[b, :, i].copy(), v_win[b, :, i].copy()
            k_win[b, :, i] = k_new[b]
            v_win[b, :, i] = v_new[b]
            win_head[b] = (i + 1) % W
        if evicted is not None:
            evicted.append((b, int(slot[0]), np.array(k_out), np.array(v_out)))
        rc = encode(f, 0, k_out[None], slot, pool, num_pages, k_signs, kc, kt, S)
        assert rc == 0
        rc = encode(f, 1, v_out[None], slot, pool, num_pages, v_signs, vc, vt, None)
        assert rc == 0
        comp_lens[b] += 1
    return skipped


# ------------------------------------------------------------------- KIVI --
class _KiviFormat(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("head_dim", "k_bits", "v_bits", "page_size", "num_kv_heads")]


class _KiviLayout(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("slab_bytes", "page_bytes", "k_params", "k_codes", "v_params", "v_codes")] + [
        (n, C.c_int32) for n in ("k_code_bytes", "v_code_bytes")
    ]


def _kfmt(f) -> _KiviFormat:
    return _KiviFormat(int(f.head_dim), int(f.k_bits), int(f.v_bits), int(f.page_size), int(f.num_kv_heads))


def kivi_layout(f) -> dict:
    """Page layout of the KIVI-style control arm (kivi.c)."""
    L = _KiviLayout()
    F = _kfmt(f)
    if _load().orc_kivi_layout(C.byref(F), C.byref(L)) != 0:
        raise ValueError("invalid KIVI format")
    return {n: getattr(L, n) for n, _ in _KiviLayout._fields_}


def kivi_quantize_group(x, bits: int):
    """Asymmetric quantization of one group of fp16 values: (scale, zero) as
    fp16 and the codes."""
    xb = _c(_f16bits(np.asarray(x, np.float16)), np.uint16)
    codes = np.zeros(len(xb), np.int32)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    _load().orc_kivi_quantize_group(len(xb), _ptr(xb), 1, int(bits), _ptr(s), _ptr(z), _ptr(codes))
    return s.view(np.float16)[0], z.view(np.float16)[0], codes


def kivi_encode_keys(f, x, page_ids, pool: np.ndarray, num_pages: int) -> int:
    """Keys x [N][H][d] fp16 in token order into pages page_ids[n // P]."""
    xb = _f16bits(x)
    pi = _c(page_ids, np.int32)
    F = _kfmt(f)
    return _load().orc_kivi_encode_keys(C.byref(F), _ptr(xb), int(xb.shape[0]), _ptr(pi), _ptr(pool), int(num_pages))


def kivi_encode_values(f, x, slot_mapping, pool: np.ndarray, num_pages: int) -> int:
    """Values x [N][H][d] fp16 into slots slot_mapping[n] (negative: skipped)."""
    xb = _f16bits(x)
    sl = _c(slot_mapping, np.int32)
    F = _kfmt(f)
    return _load().orc_kivi_encode_values(C.byref(F), _ptr(xb), int(xb.shape[0]), _ptr(sl), _ptr(pool), int(num_pages))


def kivi_decode(f, kind: int, pool, num_pages: int, slot_mapping):
    """Reconstructions [N][H][d] (fp64) of the given slots of one kind."""
    sl = _c(slot_mapping, np.int32)
    out = np.zeros((len(sl), int(f.num_kv_heads), int(f.head_dim)), np.float64)
    F = _kfmt(f)
    rc = _load().orc_kivi_decode(C.byref(F), int(kind), _ptr(_c(pool, np.uint8)), int(num_pages), _ptr(sl), len(sl), _ptr(out))
    return rc, out


def kivi_attention(f, q, pool, num_pages: int, block_tables, comp_lens, k_win, v_win, win_lens, heads=None):
    """Exact-softmax decode attention over a KIVI cache plus the fp16 window."""
    qb = _f16bits(q)
    B, Hq, d = qb.shape
    bt = _c(block_tables, np.int32)
    cl = _c(comp_lens, np.int32)
    W = 0 if k_win is None else int(k_win.shape[2])
    kw = None if k_win is None else _f16bits(k_win)
    vw = None if v_win is None else _f16bits(v_win)
    wl = None if win_lens is None else _c(win_lens, np.int32)
    hs = None if heads is None else _c(heads, np.int32)
    n = B * Hq if hs is None else len(hs)
    out = np.zeros((n, d), np.float64)
    F = _kfmt(f)
    rc = _load().orc_kivi_attention(C.byref(F), B, Hq, _ptr(qb), _ptr(_c(pool, np.uint8)), int(num_pages), _ptr(bt), int(bt.shape[1]),
                                    _ptr(cl), _ptr(kw), _ptr(vw), _ptr(wl), W, _ptr(hs), 0 if hs is None else len(hs), _ptr(out))
    return rc, (out.reshape(B, Hq, d) if hs is None else out)
