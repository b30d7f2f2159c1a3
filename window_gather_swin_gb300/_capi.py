"""ctypes view of ``libwgs.so`` (the C ABI declared in include/wgs.h).

Loading never falls back to anything: if the library is missing or lacks a
symbol, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

STATUS_NAMES = {
    0: "WGS_OK", 1: "WGS_ERR_NULL", 2: "WGS_ERR_SHAPE", 3: "WGS_ERR_WIDTH",
    4: "WGS_ERR_ALIGN", 5: "WGS_ERR_DTYPE", 6: "WGS_ERR_ARCH", 7: "WGS_ERR_LAUNCH",
    8: "WGS_ERR_INDEX", 9: "WGS_ERR_ALIAS", 10: "WGS_ERR_CUDA", 11: "WGS_ERR_TOO_LARGE",
}
WGS_F32, WGS_F16, WGS_BF16 = 0, 1, 2
ABI_VERSION = 2  # WGS_ABI_VERSION of include/wgs.h that these signatures describe

_P = ctypes.c_void_p
_i64, _i32, _f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
_st = ctypes.c_int

# name -> (restype, argtypes); one line per entry point of wgs.h
SIGNATURES = {
    "wgs_status_string": (ctypes.c_char_p, [_st]),
    "wgs_abi_version": (_i32, []),
    "ln_fwd": (_st, [_P, _P, _i64, _i32, _f32, _P]),
    "residual_add_ln_fwd": (_st, [_P, _P, _P, _P, _i64, _i32, _f32, _P]),
    "window_gather": (_st, [_P, _P, _P, _i64, _i64, _i32, _P]),
    "norm_gather": (_st, [_P, _P, _P, _i64, _i64, _i32, _f32, _P]),
    "bias_gelu_tanh": (_st, [_P, _P, _P, _i64, _i32, _i32, _P]),
    "window_reverse_add_ln_fwd": (_st, [_P, _P, _P, _P, _P, _i64, _i64, _i32, _f32, _P]),
    "residual_add_norm_gather": (_st, [_P, _P, _P, _P, _P, _i64, _i64, _i32, _f32, _P]),
    "wgs_build_window_inverse": (_st, [_P, _P, _P, _P, _i32, _P, _i64]),
    "ln_fwd_bf16": (_st, [_P, _P, _i64, _i32, _f32, _P]),
    "residual_add_ln_fwd_bf16": (_st, [_P, _P, _P, _P, _i64, _i32, _f32, _P]),
    "norm_gather_bf16": (_st, [_P, _P, _P, _i64, _i64, _i32, _f32, _P]),
    "window_reverse_add_ln_fwd_bf16": (_st, [_P, _P, _P, _P, _P, _i64, _i64, _i32, _f32, _P]),
    "residual_add_norm_gather_bf16": (_st, [_P, _P, _P, _P, _P, _i64, _i64, _i32, _f32, _P]),
    "wgs_bias_gelu_bwd_workspace_bytes": (ctypes.c_size_t, [_i64, _i32]),
    "bias_gelu_tanh_bwd": (_st, [_P, _P, _P, _P, _P, _P, ctypes.c_size_t, _i64, _i32, _i32, _P]),
    "bias_gelu_tanh_bwd_noalloc": (_st, [_P, _P, _P, _P, _P, _i64, _i32, _i32, _P]),
    "wgs_window_index_count": (_i64, [_P, _P, _P]),
    "wgs_build_window_index": (_st, [_P, _P, _P, _P, _i32, _P, _i64]),
    "window_bias_mask_add": (_st, [_P, _P, _P, _P, _P, _i64, _i32, _i32, _i32, _f32, _i32, _P]),
    "wgs_build_shift_regions": (_st, [_P, _P, _P, _P, _i32, _i32, _P, _i64]),
    "wgs_check_error": (_st, [_P]),
}

_lock = threading.Lock()
_lib = None


class WgsError(RuntimeError):
    """A non-OK status from the C ABI."""

    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({message})")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libwgs.so (building it first if nvcc is present and it is stale)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIB
        if not os.path.exists(path):
            try:
                _build.build()
            except Exception as exc:  # no toolkit, compile error, ...
                raise RuntimeError(
                    f"libwgs.so is not built ({path}) and building it failed: {exc}") from exc
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)  # AttributeError: the library lacks an entry point
            fn.restype = res
            fn.argtypes = args
        if lib.wgs_abi_version() != ABI_VERSION:
            raise RuntimeError(f"{path} has ABI version {lib.wgs_abi_version()}, this binding "
                               f"expects {ABI_VERSION}: rebuild it")
        _lib = lib
        return lib


def check(fn: str, status: int) -> None:
    if status != 0:
        msg = load().wgs_status_string(status).decode()
        raise WgsError(fn, status, msg)
