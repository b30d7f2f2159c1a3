"""The backward of bias + GELU without a caller workspace.

bias_gelu_tanh_bwd_noalloc serves callers that cannot give this library
device memory -- an op inside a host runtime that owns every allocation and
passes no allocator or workspace, or a hot path that must not call
cudaMalloc because it can synchronise the device.  Its partial sums live in
a fixed array inside the library instead of a workspace.  This file checks,
through the C ABI, that it returns exactly what the workspace entry point
returns, on two calls in a row with different inputs and on a run of calls
from the largest size the array takes down to smaller ones (the array
keeps the previous call's contents, which must not leak into the next
result), and that sizes beyond the array are refused.  It sits in its own
file, named to be collected last.
"""
import ctypes

import pytest
import torch

import window_gather_swin_gb300 as wgs
from window_gather_swin_gb300 import _capi, synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
TOO_LARGE = 11


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, gy, x, b, gx, gb):
    rows, width = x.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return lib.bias_gelu_tanh_bwd_noalloc(_p(gy), _p(x), _p(b), _p(gx), _p(gb), rows, width,
                                          CODES[x.dtype], stream)


@pytest.mark.parametrize("dtype,rows,width", [(torch.float32, 131040, 768),
                                              (torch.float16, 32760, 1536),
                                              (torch.bfloat16, 1000, 8)])
def test_noalloc_backward_matches_the_workspace_entry_point_twice(dtype, rows, width):
    lib = _capi.load()
    with torch.cuda.device(DEV):
        for call, seed in enumerate((40, 41)):      # two calls in a row, different inputs
            x, b = synth.gelu_input(rows, width, dtype, seed=seed)
            gy, _ = synth.gelu_input(rows, width, dtype, seed=seed + 7)
            x, b, gy = x.to(DEV), b.to(DEV), gy.to(DEV)
            want_gx, want_gb = wgs.bias_gelu_tanh_bwd(gy, x, b)
            gx = torch.full_like(x, float("nan"))
            gb = torch.full_like(b, float("nan"))
            assert _noalloc(lib, gy, x, b, gx, gb) == 0
            torch.cuda.synchronize(DEV)
            # same kernels and the same fixed summation order: identical bits,
            # which is inside every tolerance the other tests apply
            assert torch.equal(gx.view(torch.uint8), want_gx.view(torch.uint8)), (call, "grad_x")
            assert torch.equal(gb.view(torch.uint8), want_gb.view(torch.uint8)), (call, "grad_bias")


def test_noalloc_backward_larger_then_smaller_shapes_read_no_stale_partials():
    """The first call fills as much of the array as any call can (608 slabs
    x 2048 columns); each later call has fewer slabs, a narrower row or the
    scalar path, and new inputs.  A partial sum left by an earlier
    call and read again would change grad_bias, so every result must equal
    the workspace entry point's bit for bit."""
    lib = _capi.load()
    cases = [(torch.float16, 131328, 2048, 50), (torch.float16, 5000, 1024, 51),
             (torch.float32, 777, 520, 52), (torch.bfloat16, 333, 13, 53)]
    with torch.cuda.device(DEV):
        for dtype, rows, width, seed in cases:
            x, b = synth.gelu_input(rows, width, dtype, seed=seed)
            gy, _ = synth.gelu_input(rows, width, dtype, seed=seed + 7)
            x, b, gy = x.to(DEV), b.to(DEV), gy.to(DEV)
            want_gx, want_gb = wgs.bias_gelu_tanh_bwd(gy, x, b)
            gx = torch.full_like(x, float("nan"))
            gb = torch.full_like(b, float("nan"))
            assert _noalloc(lib, gy, x, b, gx, gb) == 0
            torch.cuda.synchronize(DEV)
            what = (str(dtype), rows, width)
            assert torch.equal(gx.view(torch.uint8), want_gx.view(torch.uint8)), (what, "grad_x")
            assert torch.equal(gb.view(torch.uint8), want_gb.view(torch.uint8)), (what, "grad_bias")


def test_noalloc_backward_refuses_sizes_beyond_its_array():
    lib = _capi.load()
    rows, width = 100_000, 4096       # 463 slabs x 4096 columns > the array's 1,310,720 floats
    x = torch.zeros(rows, width, device=DEV)
    b = torch.zeros(width, device=DEV)
    gx = torch.full_like(x, 7.0)
    with torch.cuda.device(DEV):
        assert _noalloc(lib, x, x, b, gx, b.clone()) == TOO_LARGE
    torch.cuda.synchronize(DEV)
    assert (gx == 7.0).all()                       # nothing was launched
    assert b"scratch" in lib.wgs_status_string(TOO_LARGE)
