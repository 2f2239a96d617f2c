"""Python binding of libtq.so (ctypes): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks tensor dtypes/devices, turns tensors into raw
pointers and the current CUDA stream into a handle, calls the library and
raises ``TQError`` on a non-OK status.  If libtq.so has not been built the
first call raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtq.so")  # the in-tree build

TQ_KIND_K = 0
TQ_KIND_V = 1
TQ_DEVERR_SLOT_RANGE = 0x1
TQ_DEVERR_PAGE_RANGE = 0x2
TQ_DEVERR_LENGTH = 0x4
TQ_DEVERR_TIMEOUT = 0x8

STATUS = {0: "TQ_OK", 1: "TQ_ERR_INVALID_ARG", 2: "TQ_ERR_UNSUPPORTED", 3: "TQ_ERR_CUDA", 4: "TQ_ERR_DEVICE_FAULT",
          5: "TQ_ERR_TIMEOUT", 6: "TQ_ERR_WORKSPACE", 7: "TQ_ERR_SCRATCH_LIMIT"}
TQ_STATIC_SCRATCH_BYTES = 16 << 20


class TQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({tq_status_string(status)})")


class tq_format(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("head_dim", "k_bits", "v_bits", "k_qjl", "qjl_m", "page_size", "num_kv_heads",
                                         "norm_correct")] + [("qjl_scale", C.c_float), ("k_mixed", C.c_int32)]


class tq_kivi_format(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("head_dim", "k_bits", "v_bits", "page_size", "num_kv_heads")]


class tq_kivi_layout(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("slab_bytes", "page_bytes", "k_params", "k_codes", "v_params", "v_codes")] + [
        (n, C.c_int32) for n in ("k_code_bytes", "v_code_bytes")
    ]


class tq_layout(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("slab_bytes", "page_bytes", "k_norm", "k_gamma", "k_codes", "k_signs", "v_norm", "v_codes")] + [
        (n, C.c_int32) for n in ("k_code_bytes", "k_sign_bytes", "v_code_bytes")
    ]


_lock = threading.Lock()
_lib = None


def load_library():
    """Load libtq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libtq.so not found at {LIB_PATH}: build it with decode_attention_tq_gb300.build.build()")
            lib = C.CDLL(LIB_PATH)
            P, i32, i64, sz = C.c_void_p, C.c_int, C.c_int64, C.c_size_t
            lib.tq_status_string.argtypes = [C.c_int]
            lib.tq_status_string.restype = C.c_char_p
            lib.tq_make_codebook.argtypes = [C.c_int, P, P]
            lib.tq_page_layout.argtypes = [P, P]
            lib.tq_encode.argtypes = [P, i32, P, i64, P, P, i64, P, P, P, P, P]
            lib.tq_encode_kv.argtypes = [P, P, P, i64, P, P, i64, P, P, P, P, P, P, P]
            lib.tq_append_window_workspace_size.argtypes = [P, i32, C.POINTER(sz)]
            lib.tq_append_window.argtypes = [P, i32, P, P, P, P, i32, P, P, P, P, i32, P, i64, P, P, P, P, P, P, sz, P, P]
            lib.tq_decode.argtypes = [P, i32, P, i64, P, i64, P, P, P, P, P, P]
            lib.tq_decode_attn_workspace_size.argtypes = [P, i32, i32, i32, i32, C.POINTER(sz)]
            lib.tq_decode_attn.argtypes = [P, i32, i32, P, P, i64, P, i32, P, P, P, P, i32, P, P, P, P, P, P, P, sz, P, P]
            lib.tq_decode_attn_timed.argtypes = [P, i32, i32, P, P, i64, P, i32, P, P, P, P, i32, P, P, P, P, P, P, P, sz, P, P, P, P]
            lib.tq_decode_attn_static.argtypes = [P, i32, i32, P, P, i64, P, i32, P, P, P, P, i32, P, P, P, P, P, P, P, P]
            lib.tq_kivi_page_layout.argtypes = [P, P]
            lib.tq_kivi_encode_keys.argtypes = [P, P, i64, P, P, i64, P, P]
            lib.tq_kivi_encode_values.argtypes = [P, P, i64, P, P, i64, P, P]
            lib.tq_kivi_decode.argtypes = [P, i32, P, i64, P, i64, P, P, P]
            lib.tq_kivi_decode_attn_workspace_size.argtypes = [P, i32, i32, i32, i32, C.POINTER(sz)]
            lib.tq_kivi_decode_attn.argtypes = [P, i32, i32, P, P, i64, P, i32, P, P, P, P, i32, P, P, sz, P, P]
            lib.tq_kivi_decode_attn_timed.argtypes = [P, i32, i32, P, P, i64, P, i32, P, P, P, P, i32, P, P, sz, P, P, P, P]
            for f in ("tq_make_codebook", "tq_page_layout", "tq_encode", "tq_encode_kv", "tq_append_window_workspace_size", "tq_append_window", "tq_decode", "tq_decode_attn_workspace_size", "tq_decode_attn",
                      "tq_decode_attn_timed", "tq_decode_attn_static", "tq_kivi_page_layout", "tq_kivi_encode_keys",
                      "tq_kivi_encode_values", "tq_kivi_decode", "tq_kivi_decode_attn_workspace_size", "tq_kivi_decode_attn",
                      "tq_kivi_decode_attn_timed"):
                getattr(lib, f).restype = C.c_int
            _lib = lib
    return _lib


def _fmt(f) -> tq_format:
    if isinstance(f, tq_format):
        return f
    g = (lambda k: f.get(k, 0)) if isinstance(f, dict) else (lambda k: getattr(f, k, 0))
    return tq_format(*(float(g(n)) if t is C.c_float else int(g(n)) for n, t in tq_format._fields_))


def _dev_ptr(t, dtype=None, name="tensor", allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return C.c_void_p(t.data_ptr())


def _device(*tensors) -> torch.device:
    """The one CUDA device all given tensors live on (None entries skipped).
    The library launches on the current device, so every call runs with this
    device made current."""
    devs = {t.device for t in tensors if isinstance(t, torch.Tensor)}
    if len(devs) != 1:
        raise ValueError(f"all tensors must be on one CUDA device, got {sorted(str(d) for d in devs)}")
    dev = devs.pop()
    if dev.type != "cuda":
        raise TypeError(f"tensors must be CUDA tensors, got {dev}")
    return dev


def _stream(stream):
    if stream is None:
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def _check(rc: int, where: str):
    if rc != 0:
        raise TQError(rc, where)


# ------------------------------------------------------------------- host --
def tq_status_string(status: int) -> str:
    return load_library().tq_status_string(int(status)).decode()


def tq_make_codebook(bits: int):
    """Lloyd-Max N(0,1) codebook: (centroids fp32 [2^b], midpoints fp32 [2^b-1])."""
    L = 1 << bits
    c = np.zeros(L, np.float32)
    t = np.zeros(max(L - 1, 1), np.float32)
    _check(load_library().tq_make_codebook(int(bits), c.ctypes.data, t.ctypes.data), "tq_make_codebook")
    return c, t[: L - 1]


def tq_page_layout(fmt) -> dict:
    L = tq_layout()
    F = _fmt(fmt)
    _check(load_library().tq_page_layout(C.byref(F), C.byref(L)), "tq_page_layout")
    return {n: getattr(L, n) for n, _ in tq_layout._fields_}


def device_codebook(bits: int, device="cuda") -> torch.Tensor:
    """centroids || midpoints as the fp32 device array the kernels take."""
    c, t = tq_make_codebook(bits)
    return torch.from_numpy(np.concatenate([c, t])).to(device)


def kind_codebook(fmt, kind: int, device="cuda") -> torch.Tensor:
    """The device codebook of one kind of `fmt`: device_codebook(bits), or for
    mixed-rate keys device_codebook(k_bits + 1) followed by device_codebook(k_bits)."""
    F = _fmt(fmt)
    if kind == TQ_KIND_K and F.k_mixed:
        return torch.cat([device_codebook(F.k_bits + 1, device), device_codebook(F.k_bits, device)])
    return device_codebook(F.k_bits if kind == TQ_KIND_K else F.v_bits, device)


# ----------------------------------------------------------------- device --
def tq_encode(fmt, kind: int, x, slot_mapping, page_pool, num_pages: int, signs, codebook, S=None, err_word=None, stream=None):
    F = _fmt(fmt)
    with torch.cuda.device(_device(x, slot_mapping, page_pool, signs, codebook, S, err_word)):
        rc = load_library().tq_encode(
            C.byref(F), int(kind), _dev_ptr(x, torch.float16, "x"), int(x.shape[0]), _dev_ptr(slot_mapping, torch.int32, "slot_mapping"),
            _dev_ptr(page_pool, torch.uint8, "page_pool"), int(num_pages), _dev_ptr(signs, torch.uint8, "signs"),
            _dev_ptr(codebook, torch.float32, "codebook"), _dev_ptr(S, torch.float32, "S", allow_none=True),
            _dev_ptr(err_word, torch.int32, "err_word", allow_none=True), _stream(stream),
        )
    _check(rc, "tq_encode")


def tq_encode_kv(fmt, k, v, slot_mapping, page_pool, num_pages: int, k_signs, v_signs, k_codebook, v_codebook, S=None,
                 err_word=None, stream=None):
    F = _fmt(fmt)
    if tuple(k.shape) != tuple(v.shape):
        raise ValueError("tq_encode_kv: k and v must have the same shape")
    with torch.cuda.device(_device(k, v, slot_mapping, page_pool, k_signs, v_signs, k_codebook, v_codebook, S, err_word)):
        rc = load_library().tq_encode_kv(
            C.byref(F), _dev_ptr(k, torch.float16, "k"), _dev_ptr(v, torch.float16, "v"), int(k.shape[0]),
            _dev_ptr(slot_mapping, torch.int32, "slot_mapping"), _dev_ptr(page_pool, torch.uint8, "page_pool"), int(num_pages),
            _dev_ptr(k_signs, torch.uint8, "k_signs"), _dev_ptr(v_signs, torch.uint8, "v_signs"),
            _dev_ptr(k_codebook, torch.float32, "k_codebook"), _dev_ptr(v_codebook, torch.float32, "v_codebook"),
            _dev_ptr(S, torch.float32, "S", allow_none=True), _dev_ptr(err_word, torch.int32, "err_word", allow_none=True),
            _stream(stream),
        )
    _check(rc, "tq_encode_kv")


def tq_append_window_workspace_size(fmt, batch: int) -> int:
    F = _fmt(fmt)
    n = C.c_size_t(0)
    _check(load_library().tq_append_window_workspace_size(C.byref(F), int(batch), C.byref(n)), "tq_append_window_workspace_size")
    return int(n.value)


def tq_append_window(fmt, k_new, v_new, k_win, v_win, win_lens, win_head, comp_lens, block_tables, page_pool, num_pages: int,
                     k_signs, v_signs, k_codebook, v_codebook, S=None, workspace=None, err_word=None, stream=None):
    """One decode step's append: new token into the fp16 ring window, the token
    leaving it into the pages (counters updated on the device)."""
    F = _fmt(fmt)
    B = int(k_new.shape[0])
    W = 0 if k_win is None else int(k_win.shape[2])
    if workspace is None:
        workspace = torch.empty(tq_append_window_workspace_size(F, B), dtype=torch.uint8, device=k_new.device)
    with torch.cuda.device(_device(k_new, v_new, k_win, v_win, win_lens, win_head, comp_lens, block_tables, page_pool, k_signs,
                                   v_signs, k_codebook, v_codebook, S, workspace, err_word)):
        rc = load_library().tq_append_window(
            C.byref(F), B, _dev_ptr(k_new, torch.float16, "k_new"), _dev_ptr(v_new, torch.float16, "v_new"),
            _dev_ptr(k_win, torch.float16, "k_win", allow_none=True), _dev_ptr(v_win, torch.float16, "v_win", allow_none=True), W,
            _dev_ptr(win_lens, torch.int32, "win_lens", allow_none=True), _dev_ptr(win_head, torch.int32, "win_head", allow_none=True),
            _dev_ptr(comp_lens, torch.int32, "comp_lens"), _dev_ptr(block_tables, torch.int32, "block_tables"), int(block_tables.shape[1]),
            _dev_ptr(page_pool, torch.uint8, "page_pool"), int(num_pages), _dev_ptr(k_signs, torch.uint8, "k_signs"),
            _dev_ptr(v_signs, torch.uint8, "v_signs"), _dev_ptr(k_codebook, torch.float32, "k_codebook"),
            _dev_ptr(v_codebook, torch.float32, "v_codebook"), _dev_ptr(S, torch.float32, "S", allow_none=True),
            _dev_ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()),
            _dev_ptr(err_word, torch.int32, "err_word", allow_none=True), _stream(stream),
        )
    _check(rc, "tq_append_window")


def tq_decode(fmt, kind: int, page_pool, num_pages: int, slot_mapping, signs, codebook, S=None, out=None, err_word=None, stream=None):
    F = _fmt(fmt)
    n = int(slot_mapping.shape[0])
    if out is None:
        out = torch.empty((n, F.num_kv_heads, F.head_dim), dtype=torch.float32, device=slot_mapping.device)
    with torch.cuda.device(_device(page_pool, slot_mapping, signs, codebook, S, out, err_word)):
        rc = load_library().tq_decode(
            C.byref(F), int(kind), _dev_ptr(page_pool, torch.uint8, "page_pool"), int(num_pages), _dev_ptr(slot_mapping, torch.int32, "slot_mapping"),
            n, _dev_ptr(signs, torch.uint8, "signs"), _dev_ptr(codebook, torch.float32, "codebook"),
            _dev_ptr(S, torch.float32, "S", allow_none=True), _dev_ptr(out, torch.float32, "out"),
            _dev_ptr(err_word, torch.int32, "err_word", allow_none=True), _stream(stream),
        )
    _check(rc, "tq_decode")
    return out


def tq_decode_attn_workspace_size(fmt, batch: int, num_q_heads: int, max_pages: int, window: int) -> int:
    F = _fmt(fmt)
    n = C.c_size_t(0)
    _check(load_library().tq_decode_attn_workspace_size(C.byref(F), int(batch), int(num_q_heads), int(max_pages), int(window), C.byref(n)),
           "tq_decode_attn_workspace_size")
    return int(n.value)


def tq_decode_attn(fmt, q, page_pool, num_pages: int, block_tables, comp_lens, k_win, v_win, win_lens, k_signs, v_signs,
                   k_codebook, v_codebook, S, out, workspace, err_word=None, stream=None):
    return _decode_attn(fmt, q, page_pool, num_pages, block_tables, comp_lens, k_win, v_win, win_lens, k_signs, v_signs,
                        k_codebook, v_codebook, S, out, workspace, err_word, stream, None)


def tq_decode_attn_timed(fmt, q, page_pool, num_pages: int, block_tables, comp_lens, k_win, v_win, win_lens, k_signs, v_signs,
                         k_codebook, v_codebook, S, out, workspace, main_begin, main_end, err_word=None, stream=None):
    """tq_decode_attn that also records torch.cuda.Event objects around the split-KV main kernel."""
    return _decode_attn(fmt, q, page_pool, num_pages, block_tables, comp_lens, k_win, v_win, win_lens, k_signs, v_signs,
                        k_codebook, v_codebook, S, out, workspace, err_word, stream, (main_begin, main_end))


def tq_decode_attn_static(fmt, q, page_pool, num_pages: int, block_tables, comp_lens, k_win, v_win, win_lens, k_signs, v_signs,
                          k_codebook, v_codebook, S, out, err_word=None, stream=None):
    """tq_decode_attn on the library's fixed scratch buffer: no workspace, no allocation."""
    F = _fmt(fmt)
    B, Hq, _ = q.shape
    window = 0 if k_win is None else int(k_win.shape[2])
    dev = _device(q, page_pool, block_tables, comp_lens, k_win, v_win, win_lens, k_signs, v_signs, k_codebook, v_codebook, S, out,
                  err_word)
    with torch.cuda.device(dev):  # the static scratch used is the current device's
        rc = load_library().tq_decode_attn_static(
            C.byref(F), int(B), int(Hq), _dev_ptr(q, torch.float16, "q"), _dev_ptr(page_pool, torch.uint8, "page_pool"), int(num_pages),
            _dev_ptr(block_tables, torch.int32, "block_tables"), int(block_tables.shape[1]), _dev_ptr(comp_lens, torch.int32, "comp_lens"),
            _dev_ptr(k_win, torch.float16, "k_win", allow_none=True), _dev_ptr(v_win, torch.float16, "v_win", allow_none=True),
            _dev_ptr(win_lens, torch.int32, "win_lens", allow_none=True), window, _dev_ptr(k_signs, torch.uint8, "k_signs"),
            _dev_ptr(v_signs, torch.uint8, "v_signs"), _dev_ptr(k_codebook, torch.float32, "k_codebook"),
            _dev_ptr(v_codebook, torch.float32, "v_codebook"), _dev_ptr(S, torch.float32, "S", allow_none=True),
            _dev_ptr(out, torch.float32, "out"), _dev_ptr(err_word, torch.int32, "err_word", allow_none=True), _stream(stream),
        )
    _check(rc, "tq_decode_attn_static")
    return out


def _event(ev):
    if ev is None:
        return None
    return C.c_void_p(ev.cuda_event if hasattr(ev, "cuda_event") else int(ev))


def _decode_attn(fmt, q, page_pool, num_pages, block_tables, comp_lens, k_win, v_win, win_lens, k_signs, v_signs,
                 k_codebook, v_codebook, S, out, workspace, err_word, stream, events):
    F = _fmt(fmt)
    B, Hq, _ = q.shape
    window = 0 if k_win is None else int(k_win.shape[2])
    lib = load_library()
    fn = lib.tq_decode_attn if events is None else lib.tq_decode_attn_timed
    extra = () if events is None else (_event(events[0]), _event(events[1]))
    with torch.cuda.device(_device(q, page_pool, block_tables, comp_lens, k_win, v_win, win_lens, k_signs, v_signs, k_codebook,
                                   v_codebook, S, out, workspace, err_word)):
        rc = fn(
            C.byref(F), int(B), int(Hq), _dev_ptr(q, torch.float16, "q"), _dev_ptr(page_pool, torch.uint8, "page_pool"), int(num_pages),
            _dev_ptr(block_tables, torch.int32, "block_tables"), int(block_tables.shape[1]), _dev_ptr(comp_lens, torch.int32, "comp_lens"),
            _dev_ptr(k_win, torch.float16, "k_win", allow_none=True), _dev_ptr(v_win, torch.float16, "v_win", allow_none=True),
            _dev_ptr(win_lens, torch.int32, "win_lens", allow_none=True), window, _dev_ptr(k_signs, torch.uint8, "k_signs"),
            _dev_ptr(v_signs, torch.uint8, "v_signs"), _dev_ptr(k_codebook, torch.float32, "k_codebook"),
            _dev_ptr(v_codebook, torch.float32, "v_codebook"), _dev_ptr(S, torch.float32, "S", allow_none=True),
            _dev_ptr(out, torch.float32, "out"), _dev_ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()),
            _dev_ptr(err_word, torch.int32, "err_word", allow_none=True), *extra, _stream(stream),
        )
    _check(rc, "tq_decode_attn" if events is None else "tq_decode_attn_timed")
    return out



# ------------------------------------------------------------------ KIVI --
def _kfmt(f) -> tq_kivi_format:
    if isinstance(f, tq_kivi_format):
        return f
    g = (lambda k: f.get(k, 0)) if isinstance(f, dict) else (lambda k: getattr(f, k, 0))
    return tq_kivi_format(*(int(g(n)) for n, _ in tq_kivi_format._fields_))


def tq_kivi_page_layout(fmt) -> dict:
    L = tq_kivi_layout()
    F = _kfmt(fmt)
    _check(load_library().tq_kivi_page_layout(C.byref(F), C.byref(L)), "tq_kivi_page_layout")
    return {n: getattr(L, n) for n, _ in tq_kivi_layout._fields_}


def tq_kivi_encode_keys(fmt, x, page_ids, page_pool, num_pages: int, err_word=None, stream=None):
    """Keys x [N][H][d] fp16 in token order into pages page_ids[n // P]."""
    F = _kfmt(fmt)
    with torch.cuda.device(_device(x, page_ids, page_pool, err_word)):
        rc = load_library().tq_kivi_encode_keys(
            C.byref(F), _dev_ptr(x, torch.float16, "x"), int(x.shape[0]), _dev_ptr(page_ids, torch.int32, "page_ids"),
            _dev_ptr(page_pool, torch.uint8, "page_pool"), int(num_pages), _dev_ptr(err_word, torch.int32, "err_word", allow_none=True),
            _stream(stream),
        )
    _check(rc, "tq_kivi_encode_keys")


def tq_kivi_encode_values(fmt, x, slot_mapping, page_pool, num_pages: int, err_word=None, stream=None):
    F = _kfmt(fmt)
    with torch.cuda.device(_device(x, slot_mapping, page_pool, err_word)):
        rc = load_library().tq_kivi_encode_values(
            C.byref(F), _dev_ptr(x, torch.float16, "x"), int(x.shape[0]), _dev_ptr(slot_mapping, torch.int32, "slot_mapping"),
            _dev_ptr(page_pool, torch.uint8, "page_pool"), int(num_pages), _dev_ptr(err_word, torch.int32, "err_word", allow_none=True),
            _stream(stream),
        )
    _check(rc, "tq_kivi_encode_values")


def tq_kivi_decode(fmt, kind: int, page_pool, num_pages: int, slot_mapping, out=None, err_word=None, stream=None):
    F = _kfmt(fmt)
    n = int(slot_mapping.shape[0])
    if out is None:
        out = torch.empty((n, F.num_kv_heads, F.head_dim), dtype=torch.float32, device=slot_mapping.device)
    with torch.cuda.device(_device(page_pool, slot_mapping, out, err_word)):
        rc = load_library().tq_kivi_decode(
            C.byref(F), int(kind), _dev_ptr(page_pool, torch.uint8, "page_pool"), int(num_pages),
            _dev_ptr(slot_mapping, torch.int32, "slot_mapping"), n, _dev_ptr(out, torch.float32, "out"),
            _dev_ptr(err_word, torch.int32, "err_word", allow_none=True), _stream(stream),
        )
    _check(rc, "tq_kivi_decode")
    return out


def tq_kivi_decode_attn_workspace_size(fmt, batch: int, num_q_heads: int, max_pages: int, window: int) -> int:
    F = _kfmt(fmt)
    n = C.c_size_t(0)
    _check(load_library().tq_kivi_decode_attn_workspace_size(C.byref(F), int(batch), int(num_q_heads), int(max_pages), int(window),
                                                             C.byref(n)), "tq_kivi_decode_attn_workspace_size")
    return int(n.value)


def tq_kivi_decode_attn(fmt, q, page_pool, num_pages: int, block_tables, comp_lens, k_win, v_win, win_lens, out, workspace,
                        err_word=None, stream=None, events=None):
    """Decode attention over a KIVI cache plus the fp16 window; `events`
    (begin, end) selects the timed entry point."""
    F = _kfmt(fmt)
    B, Hq, _ = q.shape
    window = 0 if k_win is None else int(k_win.shape[2])
    lib = load_library()
    fn = lib.tq_kivi_decode_attn if events is None else lib.tq_kivi_decode_attn_timed
    extra = () if events is None else (_event(events[0]), _event(events[1]))
    with torch.cuda.device(_device(q, page_pool, block_tables, comp_lens, k_win, v_win, win_lens, out, workspace, err_word)):
        rc = fn(
            C.byref(F), int(B), int(Hq), _dev_ptr(q, torch.float16, "q"), _dev_ptr(page_pool, torch.uint8, "page_pool"), int(num_pages),
            _dev_ptr(block_tables, torch.int32, "block_tables"), int(block_tables.shape[1]), _dev_ptr(comp_lens, torch.int32, "comp_lens"),
            _dev_ptr(k_win, torch.float16, "k_win", allow_none=True), _dev_ptr(v_win, torch.float16, "v_win", allow_none=True),
            _dev_ptr(win_lens, torch.int32, "win_lens", allow_none=True), window, _dev_ptr(out, torch.float32, "out"),
            _dev_ptr(workspace, torch.uint8, "workspace"), int(workspace.numel()),
            _dev_ptr(err_word, torch.int32, "err_word", allow_none=True), *extra, _stream(stream),
        )
    _check(rc, "tq_kivi_decode_attn" if events is None else "tq_kivi_decode_attn_timed")
    return out
