"""CPU oracle for the block-glue path (LN, residual add + LN, window index
map, window gather, norm-gather, bias + tanh-GELU and its backward, the
shifted-window attention bias-mask add).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg import this package; the library in
``window_gather_swin_gb300`` never does, and shares no code with it.

The arithmetic lives in ``wgs_oracle.c`` (plain C, double precision, one
element at a time).  This module only marshals numpy arrays through ctypes.
fp16 tensors are passed as ``numpy.float16`` arrays and handled as their
binary16 bit patterns.  bfloat16 tensors (``fmt="bf16"``) travel as
``numpy.uint16`` arrays of their bit patterns, numpy having no bfloat16 type.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        sig = {
            "orc_f16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
            "orc_rn16": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_rn16_array": (None, [P, P, i64]),
            "orc_f16_to_f64_array": (None, [P, P, i64]),
            "orc_rnbf16_array": (None, [P, P, i64]),
            "orc_bf16_to_f64_array": (None, [P, P, i64]),
            "orc_ln_fmt": (None, [P, P, i64, i32, f32, ctypes.c_int]),
            "orc_ln_f64_fmt": (None, [P, P, i64, i32, f32, ctypes.c_int]),
            "orc_residual_add_ln_fmt": (None, [P, P, P, P, i64, i32, f32, ctypes.c_int]),
            "orc_norm_gather_fmt": (i64, [P, P, P, i64, i64, i32, f32, ctypes.c_int]),
            "orc_bias_gelu_16": (None, [P, P, P, P, i64, i32, ctypes.c_int]),
            "orc_window_reverse_add_ln_fmt": (i64, [P, P, P, P, P, i64, i64, i32, f32, ctypes.c_int]),
            "orc_residual_add_norm_gather_fmt": (i64, [P, P, P, P, P, i64, i64, i32, f32,
                                                       ctypes.c_int]),
            "orc_ln_row_f64": (None, [P, P, i32, f32]),
            "orc_ln": (None, [P, P, i64, i32, f32]),
            "orc_ln_f64": (None, [P, P, i64, i32, f32]),
            "orc_residual_add_ln": (None, [P, P, P, P, i64, i32, f32]),
            "orc_window_index_count": (i64, [P, P, P]),
            "orc_build_window_index": (ctypes.c_int, [P, P, P, P, i32, P]),
            "orc_window_gather": (i64, [P, P, P, i64, i64, i32]),
            "orc_norm_gather": (i64, [P, P, P, i64, i64, i32, f32]),
            "orc_window_reverse_add_ln": (i64, [P, P, P, P, P, i64, i64, i32, f32]),
            "orc_invert_window_index": (None, [P, i64, P, i64]),
            "orc_residual_add_norm_gather": (i64, [P, P, P, P, P, i64, i64, i32, f32]),
            "orc_bias_gelu_f32": (None, [P, P, P, P, i64, i32]),
            "orc_bias_gelu_bwd": (None, [P, P, P, P, P, P, P, i64, i32, ctypes.c_int]),
            "orc_bias_gelu_f16": (None, [P, P, P, P, i64, i32]),
            "orc_build_shift_regions": (ctypes.c_int, [P, P, P, P, i32, i32, P]),
            "orc_window_bias_mask_add_fmt": (None, [P, P, P, P, P, i64, i32, i32, ctypes.c_double,
                                                    ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _i3(v):
    return None if v is None else np.ascontiguousarray(np.asarray(v, dtype=np.int32).reshape(3))


# ---------------------------------------------------------------- fp16 ----

def rn16(values) -> np.ndarray:
    """Round doubles to binary16 (nearest, ties to even); returns float16."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().orc_rn16_array(_ptr(v), _ptr(out), v.size)
    return out.view(np.float16)


def f16_to_f64(values) -> np.ndarray:
    """Exact double value of each binary16 element."""
    b = np.ascontiguousarray(values, dtype=np.float16).view(np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().orc_f16_to_f64_array(_ptr(b), _ptr(out), b.size)
    return out


def rnbf16(values) -> np.ndarray:
    """Round doubles to bfloat16 (nearest, ties to even); returns uint16 bits."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().orc_rnbf16_array(_ptr(v), _ptr(out), v.size)
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """Exact double value of each bfloat16 bit pattern."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().orc_bf16_to_f64_array(_ptr(b), _ptr(out), b.size)
    return out


_FMT = {"f16": (0, np.float16), "bf16": (1, np.uint16)}


def _fmt(fmt):
    if fmt not in _FMT:
        raise ValueError("fmt must be 'f16' or 'bf16'")
    return _FMT[fmt]


# ------------------------------------------------------------------ LN ----

def ln_row_f64(x, eps: float = 1e-5) -> np.ndarray:
    """Unrounded LN of one row of doubles."""
    x = _c(x, np.float64).ravel()
    y = np.empty_like(x)
    _load().orc_ln_row_f64(_ptr(x), _ptr(y), x.size, eps)
    return y


def ln(x, eps: float = 1e-5, fmt: str = "f16") -> np.ndarray:
    """No-affine LayerNorm of 16-bit rows [rows, width] -> same format."""
    code, dt = _fmt(fmt)
    x = _c(x, dt)
    rows, width = x.shape
    y = np.empty_like(x)
    _load().orc_ln_fmt(_ptr(x), _ptr(y), rows, width, eps, code)
    return y


def ln_f64(x, eps: float = 1e-5, fmt: str = "f16") -> np.ndarray:
    """Unrounded (double) LN outputs of 16-bit rows."""
    code, dt = _fmt(fmt)
    x = _c(x, dt)
    rows, width = x.shape
    y = np.empty(x.shape, dtype=np.float64)
    _load().orc_ln_f64_fmt(_ptr(x), _ptr(y), rows, width, eps, code)
    return y


def residual_add_ln(residual, branch, eps: float = 1e-5, fmt: str = "f16"):
    """Returns (residual_out, y), both in the input format."""
    code, dt = _fmt(fmt)
    a = _c(residual, dt)
    b = _c(branch, dt)
    assert a.shape == b.shape and a.ndim == 2
    r = np.empty_like(a)
    y = np.empty_like(a)
    _load().orc_residual_add_ln_fmt(_ptr(a), _ptr(b), _ptr(r), _ptr(y), a.shape[0], a.shape[1],
                                    eps, code)
    return r, y


# ----------------------------------------------------------- index map ----

def window_index_count(grid, win, padded=None) -> int:
    n = _load().orc_window_index_count(_ptr(_i3(grid)), _ptr(_i3(win)), _ptr(_i3(padded)))
    if n < 0:
        raise ValueError("invalid grid/window/padded extents")
    return int(n)


def build_window_index(grid, win, shift, padded=None, flags: int = 0) -> np.ndarray:
    """INT32 destination->source map; -1 marks a pad row."""
    n = window_index_count(grid, win, padded)
    out = np.empty(n, dtype=np.int32)
    rc = _load().orc_build_window_index(_ptr(_i3(grid)), _ptr(_i3(win)), _ptr(_i3(shift)),
                                        _ptr(_i3(padded)), flags, _ptr(out))
    if rc != 0:
        raise ValueError(f"orc_build_window_index failed ({rc})")
    return out


# -------------------------------------------------------------- gather ----

def window_gather(src, idx):
    """Returns (dst, number of indices outside [-1, n_src))."""
    s = _c(src, np.float16)
    i = _c(idx, np.int32).ravel()
    dst = np.empty((i.size, s.shape[1]), dtype=np.float16)
    bad = _load().orc_window_gather(_ptr(s), _ptr(i), _ptr(dst), s.shape[0], i.size, s.shape[1])
    return dst, int(bad)


def norm_gather(src, idx, eps: float = 1e-5, fmt: str = "f16"):
    """Returns (dst, number of indices outside [-1, n_src))."""
    code, dt = _fmt(fmt)
    s = _c(src, dt)
    i = _c(idx, np.int32).ravel()
    dst = np.empty((i.size, s.shape[1]), dtype=dt)
    bad = _load().orc_norm_gather_fmt(_ptr(s), _ptr(i), _ptr(dst), s.shape[0], i.size, s.shape[1],
                                      eps, code)
    return dst, int(bad)


# ------------------------------------------------ block-boundary fusions ----

def window_reverse_add_ln(residual, attn, idx, eps: float = 1e-5, fmt: str = "f16"):
    """Returns (residual_out, y, anomalies): r[t] = round(residual[t] + attn[d])
    for the windowed row d with idx[d] == t, y = LN(r)."""
    code, dt = _fmt(fmt)
    r = _c(residual, dt)
    w = _c(attn, dt)
    i = _c(idx, np.int32).ravel()
    assert r.ndim == 2 and w.ndim == 2 and r.shape[1] == w.shape[1] and w.shape[0] == i.size
    r_out = np.empty_like(r)
    y = np.empty_like(r)
    bad = _load().orc_window_reverse_add_ln_fmt(_ptr(r), _ptr(w), _ptr(i), _ptr(r_out), _ptr(y),
                                                r.shape[0], i.size, r.shape[1], eps, code)
    return r_out, y, int(bad)


def invert_window_index(idx, n_tokens: int) -> np.ndarray:
    """inv[t] = the windowed row that names token t (-1 if none)."""
    i = _c(idx, np.int32).ravel()
    inv = np.empty(n_tokens, dtype=np.int32)
    _load().orc_invert_window_index(_ptr(i), i.size, _ptr(inv), n_tokens)
    return inv


def residual_add_norm_gather(residual, branch, idx, eps: float = 1e-5, fmt: str = "f16"):
    """Returns (residual_out, dst, bad): r = round(residual + branch),
    dst[d] = LN(r)[idx[d]] (zero row for -1)."""
    code, dt = _fmt(fmt)
    a = _c(residual, dt)
    b = _c(branch, dt)
    i = _c(idx, np.int32).ravel()
    assert a.shape == b.shape and a.ndim == 2
    r = np.empty_like(a)
    dst = np.empty((i.size, a.shape[1]), dtype=dt)
    bad = _load().orc_residual_add_norm_gather_fmt(_ptr(a), _ptr(b), _ptr(i), _ptr(r), _ptr(dst),
                                                   a.shape[0], i.size, a.shape[1], eps, code)
    return r, dst, int(bad)


# ---------------------------------------------------------------- GELU ----

def bias_gelu_tanh(x, bias, want_f64: bool = True, fmt: str = None):
    """Returns (y, y64): y in the format of x (float32, float16, or bfloat16
    bits with fmt="bf16"), y64 the unrounded double result (None unless
    want_f64)."""
    x = np.asarray(x)
    lib = _load()
    rows, width = x.shape
    y64 = np.empty(x.shape, dtype=np.float64) if want_f64 else None
    if fmt is None and x.dtype == np.float32:
        xs, bs = _c(x, np.float32), _c(bias, np.float32)
        assert bs.shape == (width,)
        y = np.empty_like(xs)
        lib.orc_bias_gelu_f32(_ptr(xs), _ptr(bs), _ptr(y), _ptr(y64), rows, width)
        return y, y64
    if fmt is None and x.dtype == np.float16:
        fmt = "f16"
    if fmt is None:
        raise TypeError("bias_gelu_tanh oracle takes float32, float16 or fmt='bf16' bits")
    code, dt = _fmt(fmt)
    xs, bs = _c(x, dt), _c(bias, dt)
    assert bs.shape == (width,)
    y = np.empty_like(xs)
    lib.orc_bias_gelu_16(_ptr(xs), _ptr(bs), _ptr(y), _ptr(y64), rows, width, code)
    return y, y64


def bias_gelu_tanh_bwd(grad_y, x, bias, fmt: str = None):
    """Backward of y = gelu_tanh(x + bias).  Returns (grad_x, grad_bias,
    grad_x64, grad_bias64): the rounded results in the input format and the
    unrounded double values.  float32 arrays by default; fmt="f16" takes
    float16 arrays, fmt="bf16" uint16 bit patterns."""
    x = np.asarray(x)
    if fmt is None:
        fmt = {np.dtype(np.float32): "f32", np.dtype(np.float16): "f16"}.get(x.dtype)
    code, dt = {"f32": (-1, np.float32), "f16": (0, np.float16), "bf16": (1, np.uint16)}[fmt]
    gy, xs, bs = _c(grad_y, dt), _c(x, dt), _c(bias, dt).ravel()
    rows, width = xs.shape
    assert gy.shape == xs.shape and bs.shape == (width,)
    gx = np.empty_like(xs)
    gb = np.empty(width, dtype=dt)
    gx64 = np.empty(xs.shape, dtype=np.float64)
    gb64 = np.empty(width, dtype=np.float64)
    _load().orc_bias_gelu_bwd(_ptr(gy), _ptr(xs), _ptr(bs), _ptr(gx), _ptr(gb), _ptr(gx64),
                              _ptr(gb64), rows, width, code)
    return gx, gb, gx64, gb64


# ------------------------------------------------------------ bias-mask ----

def build_shift_regions(grid, win, shift, padded=None, flags: int = 0, axes_mask: int = 7):
    """INT32 region label of every windowed row (window-major order): bit k
    set when the row's cell lies past the roll's seam along masked axis k."""
    n = window_index_count(grid, win, padded)
    out = np.empty(n, dtype=np.int32)
    rc = _load().orc_build_shift_regions(_ptr(_i3(grid)), _ptr(_i3(win)), _ptr(_i3(shift)),
                                         _ptr(_i3(padded)), flags, axes_mask, _ptr(out))
    if rc != 0:
        raise ValueError(f"orc_build_shift_regions failed ({rc})")
    return out


def window_bias_mask_add(scores, bias, win_type=None, region=None, mask_value: float = -100.0,
                         fmt: str = "f16"):
    """out = round(round(scores + bias[type]) + m), m = 0 / mask_value by
    region labels (no mask add without labels).  scores [n_win, heads, n, n],
    bias [n_types, heads, n, n]; float16 arrays, or uint16 bits with
    fmt="bf16"."""
    code, dt = _fmt(fmt)
    s = _c(scores, dt)
    b = _c(bias, dt)
    n_win, heads, n, n2 = s.shape
    assert n == n2 and b.ndim == 4 and b.shape[1:] == (heads, n, n)
    t = None if win_type is None else _c(win_type, np.int32).ravel()
    r = None if region is None else _c(region, np.int32).ravel()
    assert t is None or (t.size == n_win and ((t >= 0) & (t < b.shape[0])).all())
    assert r is None or r.size == n_win * n
    out = np.empty_like(s)
    _load().orc_window_bias_mask_add_fmt(_ptr(s), _ptr(b), _ptr(t), _ptr(r), _ptr(out), n_win,
                                         heads, n, float(mask_value), code)
    return out
