"""Model-level regression gate: one shifted-window transformer block whose
glue runs on the library (norm1 + window gather, the attention bias-mask
add, window reverse + residual add + norm2, bias + GELU) with the dense parts
(QKV, softmax, projections, MLP) in torch fp16.  It is compared with the
same block written in plain torch float32: LayerNorm, torch.roll, zero
padding and reshapes for the windows, the mask from the same reading built
from coordinates.  Random weights; the grids are the tiny configurations.
"""
import math

import numpy as np
import pytest
import torch

import window_gather_swin_gb300 as wgs
from window_gather_swin_gb300 import synth

DEV = "cuda:0"
EPS = 1e-5


def _weights(c, heads, seed):
    g = torch.Generator().manual_seed(seed)
    n = synth.WINDOW[0] * synth.WINDOW[1] * synth.WINDOW[2]
    w = {
        "qkv": torch.randn(c, 3 * c, generator=g) / math.sqrt(c),
        "qkv_b": torch.randn(3 * c, generator=g) * 0.02,
        "proj": torch.randn(c, c, generator=g) / math.sqrt(c),
        "proj_b": torch.randn(c, generator=g) * 0.02,
        "fc1": torch.randn(c, 4 * c, generator=g) / math.sqrt(c),
        "fc1_b": torch.randn(4 * c, generator=g) * 0.02,
        "fc2": torch.randn(4 * c, c, generator=g) / math.sqrt(4 * c),
        "fc2_b": torch.randn(c, generator=g) * 0.02,
        "pos": torch.randn(1, heads, n, n, generator=g) * 0.02,
    }
    return {k: v.to(DEV) for k, v in w.items()}


def _windows_torch(t, grid, padded, shift=synth.SHIFT):
    """[Z*H*W, C] -> [n_win, n, C]: roll by -shift, zero-pad at the high end,
    window-major partition, row-major inside a window."""
    (Z, H, W), (wz, wh, ww) = grid, synth.WINDOW
    c = t.shape[-1]
    x = t.view(Z, H, W, c).roll(shifts=tuple(-s for s in shift), dims=(0, 1, 2))
    x = torch.nn.functional.pad(x, (0, 0, 0, padded[2] - W, 0, padded[1] - H, 0, padded[0] - Z))
    x = x.view(padded[0] // wz, wz, padded[1] // wh, wh, padded[2] // ww, ww, c)
    return x.permute(0, 2, 4, 1, 3, 5, 6).reshape(-1, wz * wh * ww, c)


def _unwindows_torch(w, grid, padded, shift=synth.SHIFT):
    (Z, H, W), (wz, wh, ww) = grid, synth.WINDOW
    c = w.shape[-1]
    x = w.view(padded[0] // wz, padded[1] // wh, padded[2] // ww, wz, wh, ww, c)
    x = x.permute(0, 3, 1, 4, 2, 5, 6).reshape(*padded, c)[:Z, :H, :W]
    return x.roll(shifts=tuple(shift), dims=(0, 1, 2)).reshape(Z * H * W, c)


def _labels_torch(grid, padded, shift=synth.SHIFT):
    """Region label of every padded cell from its coordinates (the reading of
    the shift mask: bit k when the cell lies past the roll's seam along k),
    laid out like the windows."""
    coords = torch.meshgrid(*(torch.arange(p) for p in padded), indexing="ij")
    lab = torch.zeros(padded, dtype=torch.int64)
    for k in range(3):
        s = shift[k] % grid[k]
        if s:
            lab += ((coords[k] + s) >= grid[k]).long() << k
    return _windows_torch_cells(lab, padded)


def _windows_torch_cells(lab, padded):
    wz, wh, ww = synth.WINDOW
    x = lab.view(padded[0] // wz, wz, padded[1] // wh, wh, padded[2] // ww, ww)
    return x.permute(0, 2, 4, 1, 3, 5).reshape(-1, wz * wh * ww)


def _attention(xw, w, heads, mask_add):
    """xw [n_win, n, C] -> [n_win, n, C]; mask_add(scores) adds bias and mask."""
    nw, n, c = xw.shape
    qkv = (xw @ w["qkv"] + w["qkv_b"]).view(nw, n, 3, heads, c // heads).permute(2, 0, 3, 1, 4)
    q, k, v = qkv[0], qkv[1], qkv[2]
    s = (q @ k.transpose(-1, -2)) * (c // heads) ** -0.5
    s = mask_add(s)
    p = torch.softmax(s.float(), dim=-1).to(v.dtype)
    o = (p @ v).transpose(1, 2).reshape(nw, n, c)
    return o @ w["proj"] + w["proj_b"]


def _block_reference(x, w, grid, padded, heads):
    """Plain torch float32, no library call."""
    c = x.shape[1]
    w = {k: v.float() for k, v in w.items()}
    h = torch.nn.functional.layer_norm(x, (c,), eps=EPS)
    hw = _windows_torch(h, grid, padded)
    lab = _labels_torch(grid, padded).to(x.device)
    mask = torch.where(lab[:, :, None] == lab[:, None, :], 0.0, -100.0)[:, None]

    a = _attention(hw, w, heads, lambda s: s + w["pos"] + mask)
    r = x + _unwindows_torch(a, grid, padded)
    m = torch.nn.functional.layer_norm(r, (c,), eps=EPS) @ w["fc1"]
    m = torch.nn.functional.gelu(m + w["fc1_b"], approximate="tanh") @ w["fc2"] + w["fc2_b"]
    return r + m


def _block_library(x, w, grid, padded, heads, dtype):
    """x's 16-bit format throughout, glue on the library."""
    c = x.shape[1]
    w = {k: v.to(dtype) for k, v in w.items()}
    idx = wgs.build_window_index(grid, synth.WINDOW, synth.SHIFT, padded, device=DEV)
    inv = wgs.build_window_inverse(grid, synth.WINDOW, synth.SHIFT, padded, device=DEV)
    reg = wgs.build_shift_regions(grid, synth.WINDOW, synth.SHIFT, padded, device=DEV)
    n = synth.WINDOW[0] * synth.WINDOW[1] * synth.WINDOW[2]
    hw = wgs.norm_gather(x, idx, EPS).view(-1, n, c)                     # norm1 + window gather

    def mask_add(s):
        return wgs.window_bias_mask_add(s.contiguous(), w["pos"], None, reg, -100.0)

    a = _attention(hw, w, heads, mask_add).reshape(-1, c)
    r, y = wgs.window_reverse_add_ln_fwd(x, a, inv, EPS)                 # reverse + add + norm2
    m = wgs.bias_gelu_tanh((y @ w["fc1"]).contiguous(), w["fc1_b"])     # bias + GELU
    out = r + (m @ w["fc2"] + w["fc2_b"])
    wgs.check_error(DEV)
    return out


# (grid, padded, width) of the gate's blocks: the tiny grids, and the two
# stages at full size (the 384 stage on its fully padded grid, as attention
# needs equal windows)
BLOCKS = {
    "tiny": (synth.TINY.grid, synth.TINY.padded, 192),
    "tiny_padded": (synth.TINY_PADDED.grid, synth.TINY_PADDED.padded, 192),
    "c192": (synth.ATTN_192.grid, synth.ATTN_192.padded, 192),
    "c384": (synth.ATTN_384.grid, synth.ATTN_384.padded, 384),
}
# max / mean bounds per format, about 4x what GB300 measured (fp16: max
# 4.4e-3, mean 5e-4 on the tiny grids, outputs of magnitude ~1)
BOUNDS = {torch.float16: (0.02, 2e-3), torch.bfloat16: (0.16, 1.6e-2)}


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("name", sorted(BLOCKS))
def test_one_block_against_a_float32_torch_block(name, dtype):
    grid, padded, width = BLOCKS[name]
    heads = width // 32
    tokens = grid[0] * grid[1] * grid[2]
    x, _ = synth.residual_branch(tokens, width, seed=12)
    w = _weights(width, heads, seed=13)
    ref = _block_reference(x.to(DEV).float(), w, grid, padded, heads)
    got = _block_library(x.to(DEV).to(dtype), w, grid, padded, heads, dtype).float()
    err = (got - ref).abs()
    scale = ref.abs().mean().item()
    print(name, dtype, "max", err.max().item(), "mean", err.mean().item(), "scale", scale)
    bmax, bmean = BOUNDS[dtype]
    assert err.max().item() < bmax, (err.max().item(), scale)
    assert err.mean().item() < bmean, (err.mean().item(), scale)


def test_the_torch_window_helpers_match_the_library_maps():
    """The reference's own partition agrees with the library's host maps, so
    the block comparison checks the kernels, not a shared convention (CPU)."""
    for stage in (synth.TINY, synth.TINY_PADDED):
        t = torch.arange(stage.tokens, dtype=torch.float64)[:, None] + 1.0
        win = _windows_torch(t, stage.grid, stage.padded).reshape(-1)
        idx = wgs.build_window_index(stage.grid, synth.WINDOW, synth.SHIFT, stage.padded)
        want = torch.where(idx >= 0, idx.double() + 1.0, torch.zeros(()))
        assert torch.equal(win, want)
        back = _unwindows_torch(win.view(-1, 144, 1), stage.grid, stage.padded).reshape(-1)
        assert torch.equal(back, t.reshape(-1))
        lab = _labels_torch(stage.grid, stage.padded).reshape(-1).numpy()
        ours = wgs.build_shift_regions(stage.grid, synth.WINDOW, synth.SHIFT, stage.padded)
        assert np.array_equal(lab, ours.numpy())


def _two_blocks_reference(x, w1, w2, grid, padded, heads):
    """Float32 torch: an unshifted block, then a shifted one (Swin's pair)."""
    c = x.shape[1]

    def block(x, w, shift):
        w = {k: v.float() for k, v in w.items()}
        h = _windows_torch(torch.nn.functional.layer_norm(x, (c,), eps=EPS), grid, padded, shift)
        lab = _labels_torch(grid, padded, shift).to(x.device)
        mask = torch.where(lab[:, :, None] == lab[:, None, :], 0.0, -100.0)[:, None]
        a = _attention(h, w, heads, lambda s: s + w["pos"] + mask)
        r = x + _unwindows_torch(a, grid, padded, shift)
        m = torch.nn.functional.layer_norm(r, (c,), eps=EPS) @ w["fc1"]
        return r + torch.nn.functional.gelu(m + w["fc1_b"], approximate="tanh") @ w["fc2"] + w["fc2_b"]

    return block(block(x, w1, (0, 0, 0)), w2, synth.SHIFT)


def _two_blocks_library(x, w1, w2, grid, padded, heads, dtype):
    """The same pair in x's format.  The block boundary is one
    residual_add_norm_gather: block 1's residual stream + its MLP output,
    written out, normalised by block 2's norm1 and gathered into block 2's
    shifted windows."""
    c = x.shape[1]
    n = synth.WINDOW[0] * synth.WINDOW[1] * synth.WINDOW[2]
    maps = {}
    for tag, shift in (("a", (0, 0, 0)), ("b", synth.SHIFT)):
        maps[tag] = (wgs.build_window_index(grid, synth.WINDOW, shift, padded, device=DEV),
                     wgs.build_window_inverse(grid, synth.WINDOW, shift, padded, device=DEV),
                     wgs.build_shift_regions(grid, synth.WINDOW, shift, padded, device=DEV))

    def attention_and_mlp(resid, windows, w, tag, masked):
        w = {k: v.to(dtype) for k, v in w.items()}
        _, inv, reg = maps[tag]

        def mask_add(s):
            return wgs.window_bias_mask_add(s.contiguous(), w["pos"], None,
                                            reg if masked else None, -100.0)

        a = _attention(windows.view(-1, n, c), w, heads, mask_add).reshape(-1, c)
        r, y = wgs.window_reverse_add_ln_fwd(resid, a, inv, EPS)
        m = wgs.bias_gelu_tanh((y @ w["fc1"]).contiguous(), w["fc1_b"])
        return r, (m @ w["fc2"] + w["fc2_b"]).contiguous()

    r1, mlp1 = attention_and_mlp(x, wgs.norm_gather(x, maps["a"][0], EPS), w1, "a", False)
    r2_in, windows2 = wgs.residual_add_norm_gather(r1, mlp1, maps["b"][0], EPS)
    r2, mlp2 = attention_and_mlp(r2_in, windows2, w2, "b", True)
    wgs.check_error(DEV)
    return r2 + mlp2


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["fp16", "bf16"])
@pytest.mark.parametrize("name", ["tiny_padded", "c192", "c384"])
def test_two_blocks_with_the_fused_block_boundary(name, dtype):
    """Every op of the path in one sequence: norm1 + gather, bias-mask,
    reverse + add + norm2, bias + GELU, then the fused residual add + norm1
    + gather into the next, shifted block."""
    grid, padded, width = BLOCKS[name]
    heads = width // 32
    tokens = grid[0] * grid[1] * grid[2]
    x, _ = synth.residual_branch(tokens, width, seed=14)
    w1, w2 = _weights(width, heads, seed=15), _weights(width, heads, seed=16)
    ref = _two_blocks_reference(x.to(DEV).float(), w1, w2, grid, padded, heads)
    got = _two_blocks_library(x.to(DEV).to(dtype), w1, w2, grid, padded, heads, dtype).float()
    err = (got - ref).abs()
    print(name, dtype, "two blocks: max", err.max().item(), "mean", err.mean().item(),
          "scale", ref.abs().mean().item())
    bmax, bmean = BOUNDS[dtype]
    assert err.max().item() < 2 * bmax and err.mean().item() < 2 * bmean
