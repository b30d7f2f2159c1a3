"""Python entry points, one per C-ABI function, with the same names.

Each function checks what the C ABI cannot see (device, dtype, contiguity,
shapes of torch tensors), allocates outputs the caller did not pass, and
hands raw pointers plus the current CUDA stream of the tensors' device to
libwgs.so.  No arithmetic of the op happens here, and there is no CPU path:
CPU tensors are rejected.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _capi

_DTYPE = {torch.float32: _capi.WGS_F32, torch.float16: _capi.WGS_F16,
          torch.bfloat16: _capi.WGS_BF16}
LN_WIDTHS = (192, 384)
ROW_DTYPES = (torch.float16, torch.bfloat16)


def _entry(name: str, dtype):
    """The C entry point for a 16-bit row op: fp16 `name`, bfloat16 `name_bf16`."""
    return getattr(_capi.load(), name if dtype == torch.float16 else name + "_bf16")


def _row16(t: torch.Tensor, name: str) -> None:
    _cuda(t, name)
    _require(t.dtype in ROW_DTYPES, f"{name} must be float16 or bfloat16 (got {t.dtype})")


def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise RuntimeError(msg)


def _cuda(t: torch.Tensor, name: str, dtype=None) -> None:
    _require(isinstance(t, torch.Tensor), f"{name} must be a torch.Tensor")
    _require(t.is_cuda, f"{name} must be a CUDA tensor (got {t.device})")
    if dtype is not None:
        _require(t.dtype == dtype, f"{name} must be {dtype} (got {t.dtype})")
    _require(t.is_contiguous(), f"{name} must be contiguous")


def _same_device(*ts: torch.Tensor) -> None:
    dev = ts[0].get_device()
    for t in ts[1:]:
        _require(t.get_device() == dev, f"all tensors must be on {ts[0].device} (got {t.device})")


def _stream_ptr(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


try:  # the current stream's raw handle, without building a Stream object
    _raw_stream = torch._C._cuda_getCurrentRawStream
except AttributeError:  # pragma: no cover
    def _raw_stream(index):
        return torch.cuda.current_stream(index).cuda_stream


def _call(name: str, fn, device: torch.device, *args) -> None:
    """fn(*args, stream) with `device`'s current stream, raising on a non-OK
    status; the device is made current only when it is not already."""
    index = device.index
    if torch.cuda.current_device() == index:
        _capi.check(name, fn(*args, _raw_stream(index)))
    else:
        with torch.cuda.device(index):
            _capi.check(name, fn(*args, _raw_stream(index)))


def _ptr(t: Optional[torch.Tensor]) -> int:
    """Device address of t, or 0 (NULL) for None or an empty tensor."""
    return t.data_ptr() if t is not None and t.numel() > 0 else 0


def _out(out: Optional[torch.Tensor], like_shape, dtype, device, name: str) -> torch.Tensor:
    if out is None:
        return torch.empty(like_shape, dtype=dtype, device=device)
    _cuda(out, name, dtype)
    _require(tuple(out.shape) == tuple(like_shape),
             f"{name} must have shape {tuple(like_shape)} (got {tuple(out.shape)})")
    return out


def _rows_width(x: torch.Tensor, name: str):
    _require(x.dim() >= 2, f"{name} must be [..., width]")
    width = x.shape[-1]
    return x.numel() // width if width else 0, width


# ------------------------------------------------------------------ LN ----

def ln_fwd(x: torch.Tensor, eps: float = 1e-5, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """No-affine LayerNorm over the last dim (192 or 384) of an fp16 or
    bfloat16 tensor."""
    _row16(x, "x")
    rows, width = _rows_width(x, "x")
    _require(width in LN_WIDTHS, f"width must be one of {LN_WIDTHS} (got {width})")
    y = _out(out, x.shape, x.dtype, x.device, "out")
    _same_device(x, y)
    _call("ln_fwd", _entry("ln_fwd", x.dtype), x.device, _ptr(x), _ptr(y), rows, width,
          float(eps))
    return y


def residual_add_ln_fwd(residual: torch.Tensor, branch: torch.Tensor, eps: float = 1e-5,
                        residual_out: Optional[torch.Tensor] = None,
                        out: Optional[torch.Tensor] = None):
    """Returns (residual_out, y): residual_out = round(residual + branch) in
    the tensors' 16-bit format (fp16 or bfloat16),
    y = LN(residual_out)."""
    _row16(residual, "residual")
    _cuda(branch, "branch", residual.dtype)
    _require(residual.shape == branch.shape, "residual and branch must have the same shape")
    rows, width = _rows_width(residual, "residual")
    _require(width in LN_WIDTHS, f"width must be one of {LN_WIDTHS} (got {width})")
    r = _out(residual_out, residual.shape, residual.dtype, residual.device, "residual_out")
    y = _out(out, residual.shape, residual.dtype, residual.device, "out")
    _same_device(residual, branch, r, y)
    _call("residual_add_ln_fwd", _entry("residual_add_ln_fwd", residual.dtype), residual.device,
          _ptr(residual), _ptr(branch), _ptr(r), _ptr(y), rows, width, float(eps))
    return r, y


# -------------------------------------------------------------- gather ----

def _gather_args(src, idx, out, name):
    _row16(src, "src")
    _cuda(idx, "idx", torch.int32)
    _require(src.dim() == 2, "src must be [n_src, width]")
    _require(idx.dim() == 1, "idx must be 1-D")
    n_src, width = src.shape
    dst = _out(out, (idx.numel(), width), src.dtype, src.device, "out")
    _same_device(src, idx, dst)
    return n_src, width, dst


def window_gather(src: torch.Tensor, idx: torch.Tensor,
                  out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """dst[d] = src[idx[d]] (idx >= 0) or a zero row (idx == -1).  Rows are
    copied bit for bit, so fp16 and bfloat16 use the same kernel."""
    n_src, width, dst = _gather_args(src, idx, out, "window_gather")
    _call("window_gather", _capi.load().window_gather, src.device,
          _ptr(src), _ptr(idx), _ptr(dst), n_src, idx.numel(), width)
    return dst


def norm_gather(src: torch.Tensor, idx: torch.Tensor, eps: float = 1e-5,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """dst[d] = LN(src[idx[d]]) (idx >= 0) or a zero row (idx == -1)."""
    n_src, width, dst = _gather_args(src, idx, out, "norm_gather")
    _require(width in LN_WIDTHS, f"width must be one of {LN_WIDTHS} (got {width})")
    _call("norm_gather", _entry("norm_gather", src.dtype), src.device,
          _ptr(src), _ptr(idx), _ptr(dst), n_src, idx.numel(), width, float(eps))
    return dst


# ------------------------------------------------ block-boundary fusions ----

def window_reverse_add_ln_fwd(residual: torch.Tensor, windows: torch.Tensor,
                              inv_idx: torch.Tensor, eps: float = 1e-5,
                              residual_out: Optional[torch.Tensor] = None,
                              out: Optional[torch.Tensor] = None):
    """Returns (residual_out, y): residual_out[t] = round(residual[t] +
    windows[inv_idx[t]]), y = LN(residual_out)."""
    _row16(residual, "residual")
    _cuda(windows, "windows", residual.dtype)
    _cuda(inv_idx, "inv_idx", torch.int32)
    _require(residual.dim() == 2 and windows.dim() == 2, "residual and windows must be 2-D")
    rows, width = residual.shape
    _require(windows.shape[1] == width, "windows must have the residual's width")
    _require(width in LN_WIDTHS, f"width must be one of {LN_WIDTHS} (got {width})")
    _require(inv_idx.dim() == 1 and inv_idx.numel() == rows, "inv_idx must have one entry per row")
    r = _out(residual_out, residual.shape, residual.dtype, residual.device, "residual_out")
    y = _out(out, residual.shape, residual.dtype, residual.device, "out")
    _same_device(residual, windows, inv_idx, r, y)
    _call("window_reverse_add_ln_fwd", _entry("window_reverse_add_ln_fwd", residual.dtype),
          residual.device, _ptr(residual), _ptr(windows), _ptr(inv_idx), _ptr(r), _ptr(y), rows,
          windows.shape[0], width, float(eps))
    return r, y


def residual_add_norm_gather(residual: torch.Tensor, branch: torch.Tensor, idx: torch.Tensor,
                             eps: float = 1e-5, residual_out: Optional[torch.Tensor] = None,
                             out: Optional[torch.Tensor] = None):
    """Returns (residual_out, dst): residual_out = round(residual + branch),
    dst[d] = LN(residual_out)[idx[d]] (zero row for -1)."""
    _row16(residual, "residual")
    _cuda(branch, "branch", residual.dtype)
    _cuda(idx, "idx", torch.int32)
    _require(residual.shape == branch.shape and residual.dim() == 2,
             "residual and branch must be 2-D and of the same shape")
    n_src, width = residual.shape
    _require(width in LN_WIDTHS, f"width must be one of {LN_WIDTHS} (got {width})")
    _require(idx.dim() == 1, "idx must be 1-D")
    r = _out(residual_out, residual.shape, residual.dtype, residual.device, "residual_out")
    dst = _out(out, (idx.numel(), width), residual.dtype, residual.device, "out")
    _same_device(residual, branch, idx, r, dst)
    _call("residual_add_norm_gather", _entry("residual_add_norm_gather", residual.dtype),
          residual.device, _ptr(residual), _ptr(branch), _ptr(idx), _ptr(r), _ptr(dst), n_src,
          idx.numel(), width, float(eps))
    return r, dst


# ---------------------------------------------------------------- GELU ----

def bias_gelu_tanh(x: torch.Tensor, bias: torch.Tensor,
                   out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """gelu_tanh(x + bias) over the last dim, fp32, fp16 or bfloat16."""
    _cuda(x, "x")
    _require(x.dtype in _DTYPE, f"x must be float32, float16 or bfloat16 (got {x.dtype})")
    _cuda(bias, "bias", x.dtype)
    _require(x.dim() >= 1, "x must have at least one dimension")
    width = x.shape[-1]
    _require(bias.dim() == 1 and bias.numel() == width,
             f"bias must be 1-D with {width} elements (got shape {tuple(bias.shape)})")
    rows = x.numel() // width if width else 0
    y = _out(out, x.shape, x.dtype, x.device, "out")
    _same_device(x, bias, y)
    _call("bias_gelu_tanh", _capi.load().bias_gelu_tanh, x.device,
          _ptr(x), _ptr(bias), _ptr(y), rows, width, _DTYPE[x.dtype])
    return y


def gelu_bwd_workspace_bytes(rows: int, width: int) -> int:
    """Bytes of workspace bias_gelu_tanh_bwd needs for a [rows, width] tensor."""
    return int(_capi.load().wgs_bias_gelu_bwd_workspace_bytes(int(rows), int(width)))


def bias_gelu_tanh_bwd(grad_y: torch.Tensor, x: torch.Tensor, bias: torch.Tensor,
                       grad_x: Optional[torch.Tensor] = None,
                       grad_bias: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None):
    """Backward of gelu_tanh(x + bias).  Returns (grad_x, grad_bias).  The
    deterministic column sum needs a workspace of
    wgs_bias_gelu_bwd_workspace_bytes(rows, width) bytes; one is allocated
    here unless the caller passes a uint8 CUDA tensor that large."""
    _cuda(x, "x")
    _require(x.dtype in _DTYPE, f"x must be float32, float16 or bfloat16 (got {x.dtype})")
    _cuda(grad_y, "grad_y", x.dtype)
    _cuda(bias, "bias", x.dtype)
    _require(grad_y.shape == x.shape and x.dim() >= 1, "grad_y and x must have the same shape")
    width = x.shape[-1]
    _require(bias.dim() == 1 and bias.numel() == width,
             f"bias must be 1-D with {width} elements (got shape {tuple(bias.shape)})")
    rows = x.numel() // width if width else 0
    gx = _out(grad_x, x.shape, x.dtype, x.device, "grad_x")
    gb = _out(grad_bias, bias.shape, x.dtype, x.device, "grad_bias")
    lib = _capi.load()
    need = int(lib.wgs_bias_gelu_bwd_workspace_bytes(rows, width))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _cuda(workspace, "workspace", torch.uint8)
    _same_device(grad_y, x, bias, gx, gb, workspace)
    _call("bias_gelu_tanh_bwd", lib.bias_gelu_tanh_bwd, x.device,
          _ptr(grad_y), _ptr(x), _ptr(bias), _ptr(gx), _ptr(gb), _ptr(workspace),
          workspace.numel(), rows, width, _DTYPE[x.dtype])
    return gx, gb


def window_bias_mask_add(scores: torch.Tensor, bias: torch.Tensor,
                         win_type: Optional[torch.Tensor] = None,
                         region: Optional[torch.Tensor] = None, mask_value: float = -100.0,
                         out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Attention logits plus position bias and shift mask: scores
    [n_win, heads, n, n] (float16 or bfloat16), bias [n_types, heads, n, n],
    win_type int32 [n_win] (None: type 0), region int32 [n_win * n] labels
    (None: no mask).  out may be scores."""
    _row16(scores, "scores")
    _cuda(bias, "bias", scores.dtype)
    _require(scores.dim() == 4 and scores.shape[2] == scores.shape[3],
             f"scores must be [n_win, heads, n, n] (got {tuple(scores.shape)})")
    n_win, heads, n, _ = scores.shape
    _require(bias.dim() == 4 and tuple(bias.shape[1:]) == (heads, n, n),
             f"bias must be [n_types, {heads}, {n}, {n}] (got {tuple(bias.shape)})")
    n_types = bias.shape[0]
    ts = [scores, bias]
    if win_type is not None:
        _cuda(win_type, "win_type", torch.int32)
        _require(win_type.numel() == n_win, f"win_type must have {n_win} entries")
        ts.append(win_type)
    if region is not None:
        _cuda(region, "region", torch.int32)
        _require(region.numel() == n_win * n, f"region must have {n_win * n} entries")
        ts.append(region)
    y = _out(out, scores.shape, scores.dtype, scores.device, "out")
    _same_device(*ts, y)
    _call("window_bias_mask_add", _capi.load().window_bias_mask_add, scores.device,
          _ptr(scores), _ptr(bias), _ptr(win_type), _ptr(region), _ptr(y), n_win, heads, n,
          n_types, float(mask_value), _DTYPE[scores.dtype])
    return y


# ----------------------------------------------------------- index map ----

SHIFT_THEN_PAD, PAD_THEN_SHIFT = 0, 1


def _i3(v, name):
    vals = [int(a) for a in v]
    _require(len(vals) == 3, f"{name} must have 3 entries")
    return (ctypes.c_int32 * 3)(*vals)


def window_index_count(grid: Sequence[int], window: Sequence[int],
                       padded: Optional[Sequence[int]] = None) -> int:
    n = _capi.load().wgs_window_index_count(_i3(grid, "grid"), _i3(window, "window"),
                                            _i3(padded, "padded") if padded is not None else None)
    _require(n >= 0, "invalid grid / window / padded extents")
    return int(n)


def build_window_index(grid: Sequence[int], window: Sequence[int], shift: Sequence[int],
                       padded: Optional[Sequence[int]] = None, flags: int = SHIFT_THEN_PAD,
                       device=None) -> torch.Tensor:
    """The INT32 destination -> source map (host-built); on `device` if given."""
    n = window_index_count(grid, window, padded)
    out = torch.empty(n, dtype=torch.int32)
    _capi.check("wgs_build_window_index", _capi.load().wgs_build_window_index(
        _i3(grid, "grid"), _i3(window, "window"), _i3(shift, "shift"),
        _i3(padded, "padded") if padded is not None else None, int(flags),
        ctypes.c_void_p(out.data_ptr()), n))
    return out if device is None else out.to(device)


def build_window_inverse(grid: Sequence[int], window: Sequence[int], shift: Sequence[int],
                         padded: Optional[Sequence[int]] = None, flags: int = SHIFT_THEN_PAD,
                         device=None) -> torch.Tensor:
    """inv[t] = the windowed row that holds token t (host-built); on `device` if given."""
    n = 1
    for g in grid:
        n *= int(g)
    out = torch.empty(n, dtype=torch.int32)
    _capi.check("wgs_build_window_inverse", _capi.load().wgs_build_window_inverse(
        _i3(grid, "grid"), _i3(window, "window"), _i3(shift, "shift"),
        _i3(padded, "padded") if padded is not None else None, int(flags),
        ctypes.c_void_p(out.data_ptr()), n))
    return out if device is None else out.to(device)


def build_shift_regions(grid: Sequence[int], window: Sequence[int], shift: Sequence[int],
                        padded: Optional[Sequence[int]] = None, flags: int = SHIFT_THEN_PAD,
                        axes_mask: int = 7, device=None) -> torch.Tensor:
    """INT32 shift-mask region label per windowed row (host-built), in the
    index map's order; on `device` if given."""
    n = window_index_count(grid, window, padded)
    out = torch.empty(n, dtype=torch.int32)
    _capi.check("wgs_build_shift_regions", _capi.load().wgs_build_shift_regions(
        _i3(grid, "grid"), _i3(window, "window"), _i3(shift, "shift"),
        _i3(padded, "padded") if padded is not None else None, int(flags), int(axes_mask),
        ctypes.c_void_p(out.data_ptr()), n))
    return out if device is None else out.to(device)


def check_error(device=None) -> None:
    """Raise if any gather on `device` met an index outside [-1, n_src), or
    any bias-mask add a window type outside [0, n_types), since the last
    check.  Synchronises that device's current stream."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        _capi.check("wgs_check_error", _capi.load().wgs_check_error(_stream_ptr(dev)))
