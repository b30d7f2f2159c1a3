"""Comparison rules between the CUDA path and the oracle.

* Bitwise outputs (residual_out, gathered rows, pad rows): identical bits.
* LayerNorm outputs (fp16): max |gpu - oracle| <= 2e-3 (about one fp16 ulp
  near 1).  Above that, and independently of it, every element that differs
  from the oracle's fp16 value must be its immediate fp16 neighbour AND the
  oracle's unrounded value must sit within TIE_REL * |y| + tie_abs of the
  midpoint between the two: the kernel computes in FP32, so it can only land
  on the other side of a rounding boundary when the exact value is that
  close to it.  For LN, tie_abs = LN_TIE_ABS covers the absolute error of
  x - mean in FP32 (the mean of 192 or 384 values of magnitude up to ~8 is
  good to about 3e-7); the rule is stricter than the 2e-3 bound wherever
  |y| < 0.5.
* fp32 GELU: |gpu - y64| <= 1e-5 |y64| + FLT_MIN (the floor only matters for
  results that underflow single precision).
* fp16 GELU: within one fp16 ulp of fp16(y64), and every differing element
  is a near-tie in the same sense as LN.
"""
import numpy as np

LN_ABS_TOL = 2e-3
TIE_REL = 1e-5
LN_TIE_ABS = 2e-6
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


def check_fp16_near(gpu: np.ndarray, o16: np.ndarray, y64: np.ndarray, what: str,
                    abs_tol=None, tie_abs: float = GELU_TIE_ABS) -> dict:
    """fp16 outputs against the oracle's rounded and unrounded values."""
    assert gpu.shape == o16.shape == y64.shape, what
    nan_g, nan_o = np.isnan(gpu.astype(np.float32)), np.isnan(o16.astype(np.float32))
    assert np.array_equal(nan_g, nan_o), f"{what}: NaN positions differ"
    ok = ~nan_g
    g, o, y = gpu[ok], o16[ok], y64[ok]
    dist = ulp_distance(g, o)
    diff = np.abs(g.astype(np.float64) - o.astype(np.float64))
    mism = dist > 0
    stats = {"n": int(g.size), "mismatches": int(mism.sum()), "max_ulp": int(dist.max(initial=0)),
             "max_abs": float(diff.max(initial=0.0))}
    assert stats["max_ulp"] <= 1, f"{what}: {stats}"
    if mism.any():
        tie = _near_tie(g[mism], o[mism], y[mism], tie_abs)
        assert tie.all(), (f"{what}: {int((~tie).sum())} one-ulp differences are not near a "
                           f"rounding midpoint; {stats}")
    if abs_tol is not None and stats["max_abs"] > abs_tol:
        # only near-tie one-ulp flips (checked above) may exceed the bound
        stats["above_abs_tol"] = int((diff > abs_tol).sum())
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
