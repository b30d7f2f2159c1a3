"""Seeded synthetic inputs with the shapes and value distributions of the
Pangu-Weather block-glue workloads.

This module draws random numbers and nothing else: it holds none of the
arithmetic of the kernels it feeds, so the CUDA path and the CPU oracle can
both take its tensors.  Every tensor is drawn on the CPU from an explicitly
seeded ``torch.Generator`` in float32 and then rounded (nearest-even) to the
kernel's dtype.

Workloads (token grids Z x H x W, channel width C), from the page "BW1000
gfx936 Pangu-Weather inference profiling", s3 and s5:
  * C = 192 on an 8 x 91 x 180 grid  -> 131040 tokens;
  * C = 384 on a 4 x 91 x 90 grid    ->  32760 tokens;
window (2, 6, 12) and cyclic shift (1, 3, 6) for both.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

WINDOW = (2, 6, 12)
SHIFT = (1, 3, 6)


@dataclass(frozen=True)
class Stage:
    """One hidden width of the model with its token grid and padded grid."""
    name: str
    grid: tuple
    width: int
    padded: tuple

    @property
    def tokens(self) -> int:
        return self.grid[0] * self.grid[1] * self.grid[2]

    @property
    def windowed_rows(self) -> int:
        return self.padded[0] * self.padded[1] * self.padded[2]


# The 384 stage pads H to a window multiple but keeps W = 90, which is not a
# multiple of 12; its last window along W is six columns wide.
STAGE_192 = Stage("c192", (8, 91, 180), 192, (8, 96, 180))
STAGE_384 = Stage("c384", (4, 91, 90), 384, (4, 96, 90))
TINY = Stage("tiny", (2, 12, 24), 192, (2, 12, 24))
TINY_PADDED = Stage("tiny_padded", (3, 11, 20), 192, (4, 12, 24))
STAGES = {s.name: s for s in (STAGE_192, STAGE_384, TINY, TINY_PADDED)}

# Attention over uniform windows (window-major rows, as the index map lays
# them out): the 192 stage's padded grid, and the 384 stage padded to whole
# windows (4 x 96 x 96) since a batched attention needs equal windows.
# Heads = width / 32.
@dataclass(frozen=True)
class AttnStage:
    name: str
    grid: tuple
    padded: tuple
    heads: int

    @property
    def n(self) -> int:
        return WINDOW[0] * WINDOW[1] * WINDOW[2]

    @property
    def n_win(self) -> int:
        return (self.padded[0] * self.padded[1] * self.padded[2]) // self.n

    @property
    def z_h_windows(self) -> int:
        """Windows per longitude band: one position-bias type each."""
        return (self.padded[0] // WINDOW[0]) * (self.padded[1] // WINDOW[1])


ATTN_192 = AttnStage("c192", (8, 91, 180), (8, 96, 180), 6)
ATTN_384 = AttnStage("c384", (4, 91, 90), (4, 96, 96), 12)

# MLP hidden width is 4x the stage width.
GELU_F32_SHAPE = (131040, 768)
GELU_F16_SHAPE = (32760, 1536)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def ln_input(rows: int, width: int, seed: int = 1, dtype=torch.float16) -> torch.Tensor:
    """[rows, width] (fp16 by default): N(0,1) plus a per-row offset drawn from U(-4, 4)."""
    g = _gen(seed)
    x = torch.randn(rows, width, generator=g, dtype=torch.float32)
    off = torch.rand(rows, 1, generator=g, dtype=torch.float32) * 8.0 - 4.0
    return (x + off).to(dtype)


def residual_branch(rows: int, width: int, seed: int = 2, branch_std: float = 0.1,
                    dtype=torch.float16):
    """(residual, branch), [rows, width]: N(0,1) and N(0, branch_std)."""
    g = _gen(seed)
    a = torch.randn(rows, width, generator=g, dtype=torch.float32)
    b = torch.randn(rows, width, generator=g, dtype=torch.float32) * branch_std
    return a.to(dtype), b.to(dtype)


def gather_source(rows: int, width: int, seed: int = 3, dtype=torch.float16) -> torch.Tensor:
    """[rows, width] ~ N(0,1)."""
    g = _gen(seed)
    return torch.randn(rows, width, generator=g, dtype=torch.float32).to(dtype)


def gelu_input(rows: int, width: int, dtype=torch.float32, seed: int = 4):
    """(x, bias): x [rows, width] ~ N(0,1), bias [width] ~ N(0, 0.02)."""
    g = _gen(seed)
    x = torch.randn(rows, width, generator=g, dtype=torch.float32)
    b = torch.randn(width, generator=g, dtype=torch.float32) * 0.02
    return x.to(dtype), b.to(dtype)


def attention_logits(n_win: int, heads: int, n: int, n_types: int = 1, seed: int = 6,
                     dtype=torch.float16):
    """(scores [n_win, heads, n, n] ~ N(0, 2^2), bias [n_types, heads, n, n]
    ~ N(0, 0.02^2)): pre-softmax logits of n-token windows and an expanded
    position bias per window type."""
    g = _gen(seed)
    s = torch.randn(n_win, heads, n, n, generator=g, dtype=torch.float32) * 2.0
    b = torch.randn(n_types, heads, n, n, generator=g, dtype=torch.float32) * 0.02
    return s.to(dtype), b.to(dtype)


def random_index(n_idx: int, n_src: int, pad_fraction: float = 0.1, seed: int = 5) -> torch.Tensor:
    """int32 [n_idx]: uniform source indices in [0, n_src), about
    ``pad_fraction`` of them replaced by -1.  Repeats are allowed: this is a
    generic gather index, not a window map."""
    g = _gen(seed)
    idx = torch.randint(0, max(n_src, 1), (n_idx,), generator=g, dtype=torch.int64)
    pad = torch.rand(n_idx, generator=g) < pad_fraction
    idx[pad] = -1
    if n_src == 0:
        idx[:] = -1
    return idx.to(torch.int32)


def tiny_block(seed: int = 0, stage: Stage = TINY):
    """The tiny end-to-end case: residual/branch on the stage's grid and a
    [tokens, 768] fp32 GELU input with its bias."""
    a, b = residual_branch(stage.tokens, stage.width, seed=seed)
    x, bias = gelu_input(stage.tokens, 4 * stage.width, torch.float32, seed=seed + 100)
    return a, b, x, bias
