"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every entry point include/wgs.h declares, the host index-map
builder equals the oracle's bit for bit, and argument errors come back as
status codes before anything touches a device.

Every call here with fake device pointers carries at least one error that
the library rejects during argument checking, so no kernel is ever
launched on them (on a machine with or without a GPU).
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from window_gather_swin_gb300 import _capi, synth
from window_gather_swin_gb300 import api as wgs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wgs.h")

OK, NULL, SHAPE, WIDTH, ALIGN, DTYPE, ARCH, LAUNCH, INDEX, ALIAS = range(10)
A = 0x10000000  # fake 16-byte aligned "device" addresses; never dereferenced
B = 0x20000000
C = 0x30000000
D = 0x40000000


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    return _capi.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"ln_fwd", "residual_add_ln_fwd", "window_gather", "norm_gather",
            "bias_gelu_tanh", "wgs_build_window_index", "wgs_window_index_count",
            "wgs_check_error", "wgs_status_string", "wgs_abi_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_capi.SIGNATURES), "binding table out of step with wgs.h"


def test_abi_version_and_status_strings(lib):
    assert lib.wgs_abi_version() == 2
    for s in range(11):
        assert lib.wgs_status_string(s)
    assert b"unknown" in lib.wgs_status_string(99)


# ------------------------------------------------------- index map (a3) ----

CASES = [
    (synth.STAGE_192.grid, None, 0), (synth.STAGE_192.grid, None, 1),
    (synth.STAGE_384.grid, synth.STAGE_384.padded, 0),
    (synth.STAGE_384.grid, (4, 96, 96), 0), (synth.STAGE_384.grid, synth.STAGE_384.padded, 1),
    (synth.TINY.grid, None, 0), (synth.TINY_PADDED.grid, None, 0),
    (synth.TINY_PADDED.grid, None, 1), ((2, 6, 18), (2, 6, 18), 0),
]


@pytest.mark.parametrize("grid,padded,flags", CASES)
def test_library_index_map_equals_oracle(grid, padded, flags):
    got = wgs.build_window_index(grid, synth.WINDOW, synth.SHIFT, padded, flags).numpy()
    want = oracle.build_window_index(grid, synth.WINDOW, synth.SHIFT, padded, flags)
    assert got.dtype == np.int32
    assert np.array_equal(got, want)
    assert wgs.window_index_count(grid, synth.WINDOW, padded) == want.size


@pytest.mark.parametrize("shift", [(0, 0, 0), (-1, -3, -6), (9, 100, -250), (1, 3, 6)])
@pytest.mark.parametrize("flags", [0, 1])
def test_library_index_map_odd_shifts(shift, flags):
    grid, win = (3, 7, 10), (2, 3, 4)
    got = wgs.build_window_index(grid, win, shift, None, flags).numpy()
    want = oracle.build_window_index(grid, win, shift, None, flags)
    assert np.array_equal(got, want)


def test_index_builder_errors(lib):
    g = (ctypes.c_int32 * 3)(2, 12, 24)
    w = (ctypes.c_int32 * 3)(2, 6, 12)
    s = (ctypes.c_int32 * 3)(1, 3, 6)
    small = (ctypes.c_int32 * 3)(2, 11, 24)
    bad_w = (ctypes.c_int32 * 3)(0, 6, 12)
    out = (ctypes.c_int32 * 576)()
    assert lib.wgs_window_index_count(g, w, None) == 576
    assert lib.wgs_window_index_count(g, w, small) == -1
    assert lib.wgs_window_index_count(g, bad_w, None) == -1
    assert lib.wgs_build_window_index(g, w, s, None, 0, out, 575) == SHAPE
    assert lib.wgs_build_window_index(g, w, s, None, 2, out, 576) == SHAPE
    assert lib.wgs_build_window_index(None, w, s, None, 0, out, 576) == NULL
    assert lib.wgs_build_window_index(g, w, s, None, 0, None, 576) == NULL
    assert lib.wgs_build_window_index(g, w, s, small, 0, out, 576) == SHAPE
    assert lib.wgs_build_window_index(g, w, s, None, 0, out, 576) == OK


def test_index_builders_reject_extents_whose_cell_count_overflows(lib):
    """Padded extents near INT32_MAX multiply past INT64_MAX: the count is
    -1 and every builder refuses with WGS_ERR_SHAPE before writing, even
    with an out_len a wrapped product would have passed."""
    big = 2 ** 31 - 1
    g = (ctypes.c_int32 * 3)(2, 12, 24)
    w = (ctypes.c_int32 * 3)(2, 6, 12)
    s = (ctypes.c_int32 * 3)(1, 3, 6)
    huge = (ctypes.c_int32 * 3)(big, big, big)
    wide_grid = (ctypes.c_int32 * 3)(big, big, 4)     # grid cells overflow too
    one = (ctypes.c_int32 * 3)(1, 1, 1)
    out = (ctypes.c_int32 * 8)(*([7] * 8))
    assert lib.wgs_window_index_count(g, w, huge) == -1
    assert lib.wgs_window_index_count(wide_grid, one, None) == -1
    # rounding a grid extent up to whole windows may not pass INT32_MAX
    assert lib.wgs_window_index_count((ctypes.c_int32 * 3)(1, 1, big), (ctypes.c_int32 * 3)(1, 1, 2),
                                      None) == -1
    for fn in (lib.wgs_build_window_index, lib.wgs_build_window_inverse):
        assert fn(g, w, s, huge, 0, out, 2 ** 62) == SHAPE
        assert fn(wide_grid, one, s, None, 0, out, 2 ** 62) == SHAPE
    assert lib.wgs_build_shift_regions(g, w, s, huge, 0, 7, out, 2 ** 62) == SHAPE
    assert list(out) == [7] * 8  # nothing written
    # the largest padded volume that fits still counts exactly
    fits = (ctypes.c_int32 * 3)(2, 2 ** 30, 2 ** 30)
    assert lib.wgs_window_index_count(g, w, fits) == 2 ** 61


# ------------------------------------------------ argument checking ----

def test_ln_argument_errors(lib):
    assert lib.ln_fwd(A, B, 10, 100, 1e-5, None) == WIDTH
    assert lib.ln_fwd(A, B, 10, 191, 1e-5, None) == WIDTH
    assert lib.ln_fwd(A, B, -1, 192, 1e-5, None) == SHAPE
    assert lib.ln_fwd(A, B, 2 ** 62, 192, 1e-5, None) == SHAPE
    assert lib.ln_fwd(None, None, 0, 192, 1e-5, None) == OK      # empty: nothing launched
    assert lib.ln_fwd(None, B, 10, 192, 1e-5, None) == NULL
    assert lib.ln_fwd(A + 8, B, 10, 192, 1e-5, None) == ALIGN
    assert lib.ln_fwd(A, A + 16, 10, 192, 1e-5, None) == ALIAS    # partial overlap


def test_residual_add_ln_argument_errors(lib):
    f = lib.residual_add_ln_fwd
    assert f(A, B, C, D, 10, 96, 1e-5, None) == WIDTH
    assert f(A, B, C, D, -3, 384, 1e-5, None) == SHAPE
    assert f(None, None, None, None, 0, 384, 1e-5, None) == OK
    assert f(A, None, C, D, 10, 384, 1e-5, None) == NULL
    assert f(A, B, C + 2, D, 10, 384, 1e-5, None) == ALIGN
    assert f(A, B, C, C, 10, 384, 1e-5, None) == ALIAS           # residual_out == y
    assert f(A, B, C, C + 768, 10, 384, 1e-5, None) == ALIAS     # they overlap
    assert f(A, B, A + 768, D, 10, 384, 1e-5, None) == ALIAS     # shifted in-place


def test_gather_argument_errors(lib):
    for fn, extra in ((lib.window_gather, ()), (lib.norm_gather, (1e-5,))):
        assert fn(A, B, C, 10, 5, 100, *extra, None) == WIDTH
        assert fn(A, B, C, -1, 5, 192, *extra, None) == SHAPE
        assert fn(A, B, C, 10, -5, 192, *extra, None) == SHAPE
        assert fn(None, None, None, 10, 0, 192, *extra, None) == OK
        assert fn(A, None, C, 10, 5, 192, *extra, None) == NULL
        assert fn(None, B, C, 10, 5, 192, *extra, None) == NULL   # n_src > 0 needs src
        assert fn(A, B + 2, C, 10, 5, 192, *extra, None) == ALIGN
        assert fn(A, B, C + 4, 10, 5, 192, *extra, None) == ALIGN
        assert fn(A, B, A + 384, 10, 5, 192, *extra, None) == ALIAS  # dst inside src
        assert fn(A, C + 16, C, 10, 5, 192, *extra, None) == ALIAS   # idx inside dst
    assert lib.norm_gather(A, B, C, 10, 5, 64, 1e-5, None) == WIDTH   # LN widths only
    assert lib.window_gather(A, B, C, 10, 5, 12, None) == WIDTH       # not a 16-byte row


def test_gelu_argument_errors(lib):
    f = lib.bias_gelu_tanh
    assert f(A, B, C, 10, 768, 7, None) == DTYPE
    assert f(A, B, C, -1, 768, 0, None) == SHAPE
    assert f(A, B, C, 10, -2, 0, None) == SHAPE
    assert f(None, None, None, 0, 768, 0, None) == OK
    assert f(None, None, None, 10, 0, 1, None) == OK
    assert f(A, None, C, 10, 768, 0, None) == NULL
    assert f(A + 2, B, C, 10, 768, 0, None) == ALIGN                # f32 needs 4 bytes
    assert f(A + 1, B, C, 10, 768, 1, None) == ALIGN                # f16 needs 2 bytes
    assert f(A, B, A + 4, 10, 768, 0, None) == ALIAS
    assert f(A, C + 8, C, 10, 768, 0, None) == ALIAS                # bias inside y


# ------------------------------------------- Python-side contract checks ----

def test_python_rejects_cpu_and_bad_tensors():
    import torch
    x = torch.zeros(4, 192, dtype=torch.float16)
    with pytest.raises(RuntimeError, match="CUDA"):
        wgs.ln_fwd(x)
    with pytest.raises(RuntimeError, match="CUDA"):
        wgs.bias_gelu_tanh(torch.zeros(2, 3), torch.zeros(3))
    with pytest.raises(RuntimeError, match="CUDA"):
        wgs.window_gather(x, torch.zeros(3, dtype=torch.int32))
    with pytest.raises(RuntimeError):
        wgs.build_window_index((2, 12, 24), (2, 6, 12), (1, 3, 6), padded=(2, 11, 24))


# --------------------------------------------------- inverse index map ----

@pytest.mark.parametrize("grid,padded,flags", CASES)
def test_library_inverse_map_equals_inverted_oracle_map(grid, padded, flags):
    got = wgs.build_window_inverse(grid, synth.WINDOW, synth.SHIFT, padded, flags).numpy()
    fwd = oracle.build_window_index(grid, synth.WINDOW, synth.SHIFT, padded, flags)
    want = oracle.invert_window_index(fwd, int(np.prod(grid)))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("shift", [(0, 0, 0), (-1, -3, -6), (9, 100, -250)])
@pytest.mark.parametrize("flags", [0, 1])
def test_library_inverse_map_odd_shifts(shift, flags):
    grid, win = (3, 7, 10), (2, 3, 4)
    got = wgs.build_window_inverse(grid, win, shift, None, flags).numpy()
    fwd = oracle.build_window_index(grid, win, shift, None, flags)
    assert np.array_equal(got, oracle.invert_window_index(fwd, 210))


def test_inverse_builder_errors(lib):
    g = (ctypes.c_int32 * 3)(2, 12, 24)
    w = (ctypes.c_int32 * 3)(2, 6, 12)
    s = (ctypes.c_int32 * 3)(1, 3, 6)
    out = (ctypes.c_int32 * 576)()
    assert lib.wgs_build_window_inverse(g, w, s, None, 0, out, 575) == SHAPE
    assert lib.wgs_build_window_inverse(g, w, s, None, 3, out, 576) == SHAPE
    assert lib.wgs_build_window_inverse(g, w, None, None, 0, out, 576) == NULL
    assert lib.wgs_build_window_inverse(g, w, s, None, 0, out, 576) == OK


def test_block_boundary_argument_errors(lib):
    rev = lib.window_reverse_add_ln_fwd
    assert rev(A, B, C, D, A + 2 ** 20, 10, 12, 256, 1e-5, None) == WIDTH
    assert rev(A, B, C, D, A + 2 ** 20, -1, 12, 192, 1e-5, None) == SHAPE
    assert rev(None, None, None, None, None, 0, 12, 192, 1e-5, None) == OK
    assert rev(A, B, None, D, A + 2 ** 20, 10, 12, 192, 1e-5, None) == NULL
    assert rev(A, B, C + 2, D, A + 2 ** 20, 10, 12, 192, 1e-5, None) == ALIGN
    assert rev(A, B, C, D, D, 10, 12, 192, 1e-5, None) == ALIAS          # r == y
    assert rev(A, D + 384, C, D, A + 2 ** 20, 10, 12, 192, 1e-5, None) == ALIAS  # windows in r
    ang = lib.residual_add_norm_gather
    assert ang(A, B, C, D, A + 2 ** 20, 10, 12, 100, 1e-5, None) == WIDTH
    assert ang(A, B, C, D, A + 2 ** 20, 10, -1, 192, 1e-5, None) == SHAPE
    assert ang(None, None, C, None, D, 10, 0, 192, 1e-5, None) == OK
    assert ang(A, None, C, D, A + 2 ** 20, 10, 12, 192, 1e-5, None) == NULL
    assert ang(A, B, C + 1, D, A + 2 ** 20, 10, 12, 192, 1e-5, None) == ALIGN
    assert ang(A, B, C, D, D + 128, 10, 12, 192, 1e-5, None) == ALIAS    # dst inside r
    assert ang(A, B, C, A + 768, A + 2 ** 20, 10, 12, 192, 1e-5, None) == ALIAS  # shifted r


def test_gelu_backward_argument_errors(lib):
    f = lib.bias_gelu_tanh_bwd
    need = lib.wgs_bias_gelu_bwd_workspace_bytes(1000, 768)
    assert need == 5 * 768 * 4                       # 1000 rows -> ceil(1000 / 216) = 5 slabs
    assert lib.wgs_bias_gelu_bwd_workspace_bytes(131040, 768) == 607 * 768 * 4   # ceil(131040 / 216)
    assert lib.wgs_bias_gelu_bwd_workspace_bytes(200000, 768) == 608 * 768 * 4   # the slab cap
    assert lib.wgs_bias_gelu_bwd_workspace_bytes(0, 768) == 768 * 4   # one slab: grad_bias = 0
    assert lib.wgs_bias_gelu_bwd_workspace_bytes(1000, 0) == 0
    W = 0x50000000
    assert f(A, B, C, D, A + 2 ** 24, W, need, 1000, 768, 5, None) == DTYPE
    assert f(A, B, C, D, A + 2 ** 24, W, need, -1, 768, 0, None) == SHAPE
    assert f(None, None, None, None, None, None, 0, 1000, 0, 0, None) == OK   # width 0
    assert f(A, B, None, D, A + 2 ** 24, W, need, 1000, 768, 0, None) == NULL
    assert f(A, B, C, D, A + 2 ** 24, None, need, 1000, 768, 0, None) == NULL
    assert f(A, B, C, D, A + 2 ** 24, W, need - 4, 1000, 768, 0, None) == SHAPE
    assert f(A, B, C, D, A + 2 ** 24, W + 4, need, 1000, 768, 0, None) == ALIGN
    assert f(A + 2, B, C, D, A + 2 ** 24, W, need, 1000, 768, 0, None) == ALIGN
    assert f(A, B, C, B + 64, A + 2 ** 24, W, need, 1000, 768, 0, None) == ALIAS   # grad_x in x
    assert f(A, B, C, D, C + 4, W, need, 1000, 768, 0, None) == ALIAS             # grad_bias in bias
    assert f(A, B, C, D, A + 2 ** 24, D + 64, need, 1000, 768, 0, None) == ALIAS  # workspace in grad_x


# ------------------------------------------------------------ bias-mask ----

REGION_CASES = [((8, 91, 180), (8, 96, 180), 0, 7), ((4, 91, 90), (4, 96, 96), 0, 7),
                ((4, 91, 90), (4, 96, 96), 0, 3), ((3, 11, 20), None, 1, 7),
                ((3, 11, 20), None, 0, 5), ((2, 12, 24), None, 0, 7)]


@pytest.mark.parametrize("grid,padded,flags,axes", REGION_CASES)
def test_library_shift_regions_equal_oracle(grid, padded, flags, axes):
    ours = wgs.build_shift_regions(grid, synth.WINDOW, synth.SHIFT, padded, flags, axes).numpy()
    want = oracle.build_shift_regions(grid, synth.WINDOW, synth.SHIFT, padded, flags, axes)
    assert np.array_equal(ours, want)


@pytest.mark.parametrize("shift", [(0, 0, 0), (-1, 5, 0), (3, -7, 25), (1, 1, 1)])
@pytest.mark.parametrize("flags", [0, 1])
def test_library_shift_regions_odd_shifts(shift, flags):
    grid, win = (5, 13, 27), (2, 6, 12)
    ours = wgs.build_shift_regions(grid, win, shift, None, flags, 7).numpy()
    assert np.array_equal(ours, oracle.build_shift_regions(grid, win, shift, None, flags, 7))


def test_shift_region_builder_errors(lib):
    g, w, s = (ctypes.c_int32 * 3)(2, 12, 24), (ctypes.c_int32 * 3)(2, 6, 12), (ctypes.c_int32 * 3)(1, 3, 6)
    out = (ctypes.c_int32 * 576)()
    f = lib.wgs_build_shift_regions
    assert f(g, w, s, None, 0, 7, out, 576) == OK
    assert f(g, w, s, None, 0, 7, out, 575) == SHAPE
    assert f(g, w, s, None, 2, 7, out, 576) == SHAPE
    assert f(g, w, s, None, 0, 8, out, 576) == SHAPE
    assert f(g, w, s, None, 0, -1, out, 576) == SHAPE
    assert f(None, w, s, None, 0, 7, out, 576) == NULL
    assert f(g, w, s, None, 0, 7, None, 576) == NULL
    bad = (ctypes.c_int32 * 3)(2, 12, 20)
    assert f(g, w, s, bad, 0, 7, out, 576) == SHAPE              # padded < grid


def test_bias_mask_argument_errors(lib):
    f = lib.window_bias_mask_add
    R = 0x50000000
    # (scores, bias, win_type, region, out, n_win, heads, n, n_types, mask, dtype, stream)
    assert f(A, B, None, R, C, 4, 6, 144, 1, -100.0, 0, None) == DTYPE          # fp32
    assert f(A, B, None, R, C, 4, 6, 144, 1, -100.0, 3, None) == DTYPE
    assert f(A, B, None, R, C, -1, 6, 144, 1, -100.0, 1, None) == SHAPE
    assert f(A, B, None, R, C, 4, 6, 144, -1, -100.0, 1, None) == SHAPE
    assert f(None, None, None, None, None, 0, 6, 144, 1, -100.0, 1, None) == OK  # empty
    assert f(None, None, None, None, None, 4, 0, 144, 0, -100.0, 1, None) == OK
    assert f(A, B, None, R, C, 4, 6, 144, 0, -100.0, 1, None) == SHAPE          # no bias slab
    assert f(A, B, None, R, C, 2 ** 31 // 144 + 1, 1, 144, 1, -100.0, 1, None) == SHAPE  # 2^31 rows
    assert f(None, B, None, R, C, 4, 6, 144, 1, -100.0, 1, None) == NULL
    assert f(A, None, None, R, C, 4, 6, 144, 1, -100.0, 2, None) == NULL
    assert f(A, B, None, R, None, 4, 6, 144, 1, -100.0, 1, None) == NULL
    assert f(A + 1, B, None, R, C, 4, 6, 144, 1, -100.0, 1, None) == ALIGN
    assert f(A, B, None, R + 2, C, 4, 6, 144, 1, -100.0, 1, None) == ALIGN
    assert f(A, B, R + 2, None, C, 4, 6, 144, 1, -100.0, 1, None) == ALIGN
    assert f(A, B, None, R, A + 64, 4, 6, 144, 1, -100.0, 1, None) == ALIAS      # shifted out
    assert f(A, B, None, R, B, 4, 6, 144, 1, -100.0, 1, None) == ALIAS           # out = bias
    assert f(A, B, None, C + 16, C, 4, 6, 144, 1, -100.0, 1, None) == ALIAS      # region in out


# -------------------------------------------- randomised host builders ----

def test_host_builders_equal_oracle_on_random_grids():
    """Library index map, inverse map and region labels against the oracle
    on random grids, windows (including cut last windows), shifts of any
    sign and size, explicit padded extents, both orders and mask axes."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=300, deadline=None, derandomize=True)
    @hyp.given(st.data())
    def run(data):
        grid = tuple(data.draw(st.integers(1, 9)) for _ in range(3))
        win = tuple(data.draw(st.integers(1, 5)) for _ in range(3))
        shift = tuple(data.draw(st.integers(-20, 20)) for _ in range(3))
        padded = None
        if data.draw(st.booleans()):
            padded = tuple(g + data.draw(st.integers(0, 6)) for g in grid)
        flags = data.draw(st.integers(0, 1))
        axes = data.draw(st.integers(0, 7))
        idx = wgs.build_window_index(grid, win, shift, padded, flags).numpy()
        assert np.array_equal(idx, oracle.build_window_index(grid, win, shift, padded, flags))
        lab = wgs.build_shift_regions(grid, win, shift, padded, flags, axes).numpy()
        assert np.array_equal(lab, oracle.build_shift_regions(grid, win, shift, padded, flags, axes))
        n_tokens = grid[0] * grid[1] * grid[2]
        covered = np.bincount(idx[idx >= 0], minlength=n_tokens)
        if (covered == 1).all():   # the map names every token once
            inv = wgs.build_window_inverse(grid, win, shift, padded, flags).numpy()
            assert np.array_equal(inv, oracle.invert_window_index(idx, n_tokens))

    run()
