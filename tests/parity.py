"""Comparison rules between the CUDA path and the oracle.

* Bitwise outputs (residual_out, gathered rows, pad rows): identical bits.
* fp16 outputs computed in FP32 (LayerNorm, fp16 GELU): every element obeys
      |gpu - y| <= ulp16(gpu) / 2 + TIE_REL * |y| + tie_abs,
  where y is the oracle's unrounded double value: the kernel's FP32 result
  is within TIE_REL relative plus tie_abs absolute of y, and rounding it to
  fp16 adds at most half a spacing.  For LayerNorm the absolute term
  LN_TIE_ABS covers the FP32 error of d = x - mean, which dominates near
  y = 0 where fp16 spacings are tiny: with the shifted-data two-pass (sums
  of x - x[0]), recursive summation over at most ~27 levels bounds the
  error of the mean by ~27 u * 1.5 sigma (u = 2^-24), i.e. about 2.4e-6
  after scaling by 1/sigma; LN_TIE_ABS = 4e-6 leaves margin.
* LayerNorm additionally meets the 2e-3 max-abs bar, except for elements
  one fp16 spacing away from the oracle's fp16 value whose unrounded value
  lies within TIE_REL * |y| + tie_abs of the midpoint (legitimate rounding
  flips at |y| >= 4, where one spacing is 3.9e-3).
* fp32 GELU: |gpu - y| <= 1e-5 |y| + FLT_MIN (the floor only matters for
  results that underflow single precision).
"""
import numpy as np

LN_ABS_TOL = 2e-3
TIE_REL = 1e-5
LN_TIE_ABS = 4e-6
GELU_TIE_ABS = 1e-12
GELU_F32_REL = 1e-5
FLT_MIN = float(np.finfo(np.float32).tiny)


def f16_ordinal(h: np.ndarray) -> np.ndarray:
    """Monotone integer image of fp16 bit patterns (+0 and -0 both map to 0)."""
    b = np.ascontiguousarray(h, dtype=np.float16).view(np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(f16_ordinal(a) - f16_ordinal(b))


def assert_bitwise(gpu: np.ndarray, want: np.ndarray, what: str) -> None:
    g = np.ascontiguousarray(gpu).view(np.uint8)
    w = np.ascontiguousarray(want).view(np.uint8)
    assert g.shape == w.shape, f"{what}: shape {gpu.shape} vs {want.shape}"
    if not np.array_equal(g, w):
        bad = np.argwhere(np.ascontiguousarray(gpu).view(np.uint16 if gpu.dtype == np.float16 else np.uint8)
                          != np.ascontiguousarray(want).view(np.uint16 if want.dtype == np.float16 else np.uint8))
        raise AssertionError(f"{what}: {len(bad)} elements differ, first at {bad[:5].tolist()}")


def _near_tie(g: np.ndarray, o16: np.ndarray, y64: np.ndarray, tie_abs: float) -> np.ndarray:
    mid = (g.astype(np.float64) + o16.astype(np.float64)) / 2.0
    return np.abs(y64 - mid) <= TIE_REL * np.abs(y64) + tie_abs


def fp16_spacing(v: np.ndarray) -> np.ndarray:
    """Distance from |v| to the next larger fp16 value (2^-24 below 2^-14)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return np.exp2(e - 10.0)


def check_fp16_near(gpu: np.ndarray, o16: np.ndarray, y64: np.ndarray, what: str,
                    abs_tol=None, tie_abs: float = GELU_TIE_ABS) -> dict:
    """fp16 outputs against the oracle's rounded (o16) and unrounded (y64) values."""
    assert gpu.shape == o16.shape == y64.shape, what
    gf = gpu.astype(np.float64)
    of = o16.astype(np.float64)
    fin = np.isfinite(of)
    assert np.array_equal(np.isnan(gf), np.isnan(of)), f"{what}: NaN positions differ"
    inf = np.isinf(of)
    assert np.array_equal(gf[inf], of[inf]), f"{what}: infinities differ"
    g, o, y = gpu[fin], o16[fin], y64[fin]
    gd = g.astype(np.float64)
    dist = ulp_distance(g, o)
    diff = np.abs(gd - o.astype(np.float64))
    err = np.abs(gd - y)
    bound = 0.5 * fp16_spacing(gd) + TIE_REL * np.abs(y) + tie_abs
    viol = err > bound
    stats = {"n": int(g.size), "mismatches": int((dist > 0).sum()),
             "max_ulp": int(dist.max(initial=0)), "max_abs": float(diff.max(initial=0.0)),
             "max_err_over_bound": float((err / bound).max(initial=0.0))}
    if viol.any():
        k = np.argmax(err - bound)
        raise AssertionError(f"{what}: {int(viol.sum())} elements outside the FP32 error bound, "
                             f"worst gpu={gd[k]!r} oracle={y[k]!r}; {stats}")
    if abs_tol is not None:
        above = diff > abs_tol
        if above.any():
            ok = (dist[above] == 1) & _near_tie(g[above], o[above], y[above], tie_abs)
            assert ok.all(), (f"{what}: {int((~ok).sum())} elements exceed {abs_tol} without "
                              f"being a one-spacing rounding flip at a midpoint; {stats}")
            stats["above_abs_tol_tie_flips"] = int(above.sum())
    return stats


def check_ln(gpu: np.ndarray, o16: np.ndarray, y64: np.ndarray, what: str) -> dict:
    return check_fp16_near(gpu, o16, y64, what, abs_tol=LN_ABS_TOL, tie_abs=LN_TIE_ABS)


def check_gelu_f32(gpu: np.ndarray, y64: np.ndarray, what: str) -> dict:
    g = gpu.astype(np.float64)
    nan_g, nan_o = np.isnan(g), np.isnan(y64)
    assert np.array_equal(nan_g, nan_o), f"{what}: NaN positions differ"
    ok = ~nan_g
    err = np.abs(g[ok] - y64[ok])
    lim = GELU_F32_REL * np.abs(y64[ok]) + FLT_MIN
    rel = err / np.maximum(np.abs(y64[ok]), FLT_MIN)
    stats = {"n": int(ok.sum()), "max_rel": float(rel.max(initial=0.0)),
             "violations": int((err > lim).sum())}
    assert stats["violations"] == 0, f"{what}: {stats}"
    return stats


# ------------------------------------------------------------ bfloat16 ----

def bf16_values(bits: np.ndarray) -> np.ndarray:
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).astype(np.int16)).view(
        torch.bfloat16).double().numpy()


def bf16_spacing(v: np.ndarray) -> np.ndarray:
    """Distance from |v| to the next larger bfloat16 value (2^-133 below 2^-126)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7.0)


def check_bf16_near(gpu_bits: np.ndarray, o_bits: np.ndarray, y64: np.ndarray, what: str,
                    tie_abs: float = GELU_TIE_ABS) -> dict:
    """bfloat16 outputs (bit patterns) against the oracle: the same FP32
    error bound as for fp16, with bfloat16's spacing."""
    g, o = bf16_values(gpu_bits), bf16_values(o_bits)
    assert g.shape == o.shape == y64.shape, what
    assert np.array_equal(np.isnan(g), np.isnan(o)), f"{what}: NaN positions differ"
    fin = np.isfinite(o)
    assert np.array_equal(g[~fin & ~np.isnan(o)], o[~fin & ~np.isnan(o)]), f"{what}: infinities"
    g, o, y = g[fin], o[fin], y64[fin]
    dist = ulp_distance(np.asarray(gpu_bits)[fin].view(np.float16), np.asarray(o_bits)[fin].view(np.float16))
    err = np.abs(g - y)
    bound = 0.5 * bf16_spacing(g) + TIE_REL * np.abs(y) + tie_abs
    viol = err > bound
    stats = {"n": int(g.size), "mismatches": int((dist > 0).sum()), "max_ulp": int(dist.max(initial=0)),
             "max_abs": float(np.abs(g - o).max(initial=0.0)),
             "max_err_over_bound": float((err / bound).max(initial=0.0))}
    if viol.any():
        k = np.argmax(err - bound)
        raise AssertionError(f"{what}: {int(viol.sum())} elements outside the FP32 error bound, "
                             f"worst gpu={g[k]!r} oracle={y[k]!r}; {stats}")
    return stats
