"""GB300-native block-glue kernels for shifted-window transformers.

No-affine LayerNorm, fused residual add + LayerNorm, the INT32-indexed
shifted-window gather, the fused norm-then-gather, the bias + tanh-GELU
epilogue and its backward, and the attention bias + shift-mask add, as
hand-written sm_103a CUDA kernels behind a C ABI
(include/wgs.h, libwgs.so).  The functions below are thin marshalling
wrappers with the same names as the C entry points.
"""
from .api import (LN_WIDTHS, PAD_THEN_SHIFT, SHIFT_THEN_PAD, bias_gelu_tanh, bias_gelu_tanh_bwd,
                  build_shift_regions, build_window_index, build_window_inverse, check_error,
                  gelu_bwd_workspace_bytes, ln_fwd, norm_gather,
                  residual_add_ln_fwd, residual_add_norm_gather, window_gather,
                  window_bias_mask_add, window_index_count, window_reverse_add_ln_fwd)
from ._capi import WgsError

__all__ = [
    "ln_fwd", "residual_add_ln_fwd", "window_gather", "norm_gather", "bias_gelu_tanh",
    "window_reverse_add_ln_fwd", "residual_add_norm_gather", "bias_gelu_tanh_bwd",
    "gelu_bwd_workspace_bytes", "window_bias_mask_add", "build_shift_regions",
    "window_index_count",
    "build_window_index", "build_window_inverse", "check_error", "WgsError", "LN_WIDTHS",
    "SHIFT_THEN_PAD", "PAD_THEN_SHIFT",
]
