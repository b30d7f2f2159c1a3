"""Pins of the CPU oracle against facts fixed outside itself: IEEE binary16
rounding as numpy implements it, closed forms and invariants of LayerNorm,
torch's float64 layer_norm and tanh-GELU, hand-derived index-map entries and
a sort-based brute-force index-map builder.

Each pin is chosen so that a plausible slip in the oracle (a dropped eps, an
unbiased variance, a wrong shift sign, a transposed window order, a bias
indexed by row, an LN taken before the fp16 rounding point) fails here.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from golden_io import gelu_tiny_input, window_index_cases
from window_gather_swin_gb300 import synth

EPS = float(np.float32(1e-5))


# ------------------------------------------------------------- binary16 ----

def _all_f16():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)


def test_f16_decode_matches_numpy_on_every_pattern():
    h = _all_f16()
    ours = oracle.f16_to_f64(h)
    ref = h.astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_rn16_round_trips_every_pattern():
    h = _all_f16()
    back = oracle.rn16(oracle.f16_to_f64(h))
    nan = np.isnan(h.astype(np.float64))
    assert np.array_equal(back.view(np.uint16)[~nan], h.view(np.uint16)[~nan])
    assert np.isnan(back[nan].astype(np.float64)).all()


def test_rn16_matches_numpy_on_random_doubles():
    rng = np.random.default_rng(11)
    mag = np.exp2(rng.uniform(-30.0, 17.0, 400_000))
    v = mag * rng.choice([-1.0, 1.0], mag.size)
    with np.errstate(over="ignore"):   # values past 65520 round to +-inf, as intended
        ref = v.astype(np.float16)
    assert np.array_equal(oracle.rn16(v).view(np.uint16), ref.view(np.uint16))


def test_rn16_ties_go_to_even_and_near_ties_to_nearest():
    h = _all_f16()
    vals = h.astype(np.float64)
    pos = vals[(vals >= 0) & np.isfinite(vals)]
    pos = np.unique(pos)
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2.0  # exact in double
    got = oracle.rn16(mid).view(np.uint16)
    lo_bits = lo.astype(np.float16).view(np.uint16)
    hi_bits = hi.astype(np.float16).view(np.uint16)
    want = np.where(lo_bits % 2 == 0, lo_bits, hi_bits)
    assert np.array_equal(got, want)
    # a hair either side of the midpoint goes to the nearer neighbour
    below = np.nextafter(mid, -np.inf)
    above = np.nextafter(mid, np.inf)
    assert np.array_equal(oracle.rn16(below).view(np.uint16), lo_bits)
    assert np.array_equal(oracle.rn16(above).view(np.uint16), hi_bits)


def test_rn16_range_edges():
    bits = lambda v: int(oracle.rn16(np.array([v])).view(np.uint16)[0])
    assert bits(65519.99) == 0x7BFF          # rounds down to 65504
    assert bits(65520.0) == 0x7C00           # tie goes to 2^16 = inf
    assert bits(-65520.0) == 0xFC00
    assert bits(2.0 ** -25) == 0x0000        # tie between 0 and 2^-24 -> 0
    assert bits(3 * 2.0 ** -25) == 0x0002    # tie between 1 and 2 quanta -> 2
    assert bits(2.0 ** -24) == 0x0001
    assert bits(-0.0) == 0x8000
    assert bits(np.inf) == 0x7C00


# ----------------------------------------------------------- LayerNorm ----

@pytest.mark.parametrize("width", [192, 384])
def test_ln_constant_rows_map_to_zero(width):
    consts = np.array([0.0, 1.0, -3.5, 1000.0, -65504.0, 2.0 ** -20], dtype=np.float16)
    x = np.repeat(consts[:, None], width, axis=1)
    y = oracle.ln(x, EPS).astype(np.float64)
    assert (y == 0.0).all()


@pytest.mark.parametrize("width", [192, 384, 7])
def test_ln_moments_closed_form(width):
    rng = np.random.default_rng(width)
    for _ in range(20):
        x = rng.normal(rng.uniform(-4, 4), rng.uniform(0.01, 3.0), width)
        y = oracle.ln_row_f64(x, EPS)
        var = np.var(x)  # population variance
        assert abs(y.mean()) < 1e-13
        assert np.mean(y * y) == pytest.approx(var / (var + EPS), rel=1e-12)


def test_ln_alternating_row_is_plus_minus_one():
    x = np.tile(np.array([1.0, -1.0], dtype=np.float16), 96)[None, :]
    y = oracle.ln(x, EPS).astype(np.float64)
    # unrounded value is +-1/sqrt(1 + eps), which is within half an ulp of 1
    assert np.array_equal(y[0], np.tile([1.0, -1.0], 96))
    y64 = oracle.ln_f64(x, EPS)
    assert y64[0, 0] == pytest.approx(1.0 / np.sqrt(1.0 + EPS), rel=1e-15)


def test_ln_shift_invariance_on_integer_rows():
    rng = np.random.default_rng(3)
    x = rng.integers(-50, 50, (16, 192)).astype(np.float16)
    for k in (-100, 7, 512):
        assert np.array_equal(oracle.ln(x, EPS).view(np.uint16),
                              oracle.ln((x.astype(np.float64) + k).astype(np.float16), EPS).view(np.uint16))


@pytest.mark.parametrize("width", [192, 384])
def test_ln_matches_torch_float64_layer_norm(width):
    x = synth.ln_input(512, width, seed=21).numpy()
    ours = oracle.ln_f64(x, EPS)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x.astype(np.float64)), (width,),
                                         eps=EPS).numpy()
    assert np.max(np.abs(ours - ref)) < 1e-12
    assert np.array_equal(oracle.ln(x, EPS).view(np.uint16), ref.astype(np.float16).view(np.uint16))


# ------------------------------------------------- residual add + LN ----

def test_residual_sum_is_fp16_of_fp32_sum():
    """numpy adds float16 arrays by widening to float32, adding and rounding
    back: the page's fp16(fp32 a + fp32 b), computed by someone else."""
    a = np.repeat(_all_f16(), 96)
    rng = np.random.default_rng(5)
    b = rng.permutation(np.repeat(_all_f16(), 96))
    finite = np.isfinite(a.astype(np.float64)) & np.isfinite(b.astype(np.float64))
    a, b = a[finite], b[finite]
    n = (a.size // 192) * 192
    a, b = a[:n].reshape(-1, 192), b[:n].reshape(-1, 192)
    r, _ = oracle.residual_add_ln(a, b, EPS)
    with np.errstate(over="ignore", invalid="ignore"):
        want = (a + b)
    assert np.array_equal(r.view(np.uint16), want.view(np.uint16))


def test_residual_sum_exhaustive_over_b_for_chosen_a():
    """Every finite binary16 b against 80 chosen a (signed zeros, the
    smallest and largest subnormals and normals, a value at and one between
    every power of two from 2^-14 to 2^15, the largest finite, odd
    mantissas): 5.2 M pairs, all exact against numpy's widen-add-round."""
    every = _all_f16()
    picks = [0.0, -0.0, 6e-8, -6e-8, 6.1e-5, -6.1e-5, 65504.0, -65504.0]
    for e in range(-14, 16):
        picks += [2.0 ** e, -(2.0 ** e) * 1.5]
    picks += [0.1, -0.3, 1.0009765625, 3.14, 1000.5, -2049.0, 0.33325, -7.998]
    picks += [1.0 - 2 ** -11, 2049.0, 4097.0, -8191.0]
    a_vals = np.array(picks, dtype=np.float16)
    assert a_vals.size == 80
    fin_b = every[np.isfinite(every.astype(np.float64))]
    n = (fin_b.size // 192) * 192
    b = fin_b[:n].reshape(-1, 192)
    for av in a_vals:
        a = np.full_like(b, av)
        r, _ = oracle.residual_add_ln(a, b, EPS)
        with np.errstate(over="ignore", invalid="ignore"):
            want = a + b
        assert np.array_equal(r.view(np.uint16), want.view(np.uint16)), float(av)


def test_residual_ln_is_taken_after_the_fp16_rounding():
    a, b = synth.residual_branch(576, 192, seed=0)
    a, b = a.numpy(), b.numpy()
    r, y = oracle.residual_add_ln(a, b, EPS)
    assert np.array_equal(y.view(np.uint16), oracle.ln(r, EPS).view(np.uint16))
    # LN of the unrounded sum differs somewhere, so the check above has teeth
    exact = a.astype(np.float64) + b.astype(np.float64)
    unrounded = torch.nn.functional.layer_norm(torch.from_numpy(exact), (192,), eps=EPS).numpy()
    assert not np.array_equal(unrounded.astype(np.float16).view(np.uint16), y.view(np.uint16))


# ---------------------------------------------------------- index map ----

def brute_force_index(grid, win, shift, padded, flags):
    """Sort-based construction, independent of the oracle's scatter: list
    every padded cell with its (window, in-window) key, sort, read sources."""
    Z, H, W = grid
    P = padded
    cells = []
    for z, h, w in itertools.product(range(P[0]), range(P[1]), range(P[2])):
        key = (z // win[0], h // win[1], w // win[2], z % win[0], h % win[1], w % win[2])
        if flags == 0:
            if z < Z and h < H and w < W:
                s = (((z + shift[0]) % Z) * H + (h + shift[1]) % H) * W + (w + shift[2]) % W
            else:
                s = -1
        else:
            zs, hs, ws = (z + shift[0]) % P[0], (h + shift[1]) % P[1], (w + shift[2]) % P[2]
            s = (zs * H + hs) * W + ws if (zs < Z and hs < H and ws < W) else -1
        cells.append((key, s))
    cells.sort()
    return np.array([s for _, s in cells], dtype=np.int32)


def test_index_map_worked_entries():
    for name, c in window_index_cases().items():
        m = oracle.build_window_index(c["grid"], c["win"], c["shift"], c["padded"], c["flags"])
        assert m.size == c["n_idx"], name
        assert int((m == -1).sum()) == c["n_pads"], name
        for dst, src in c["entries"]:
            assert m[dst] == src, (name, dst, m[dst], src)


BRUTE_CASES = [
    ((2, 12, 24), (2, 6, 12), (1, 3, 6), None, 0),
    ((3, 11, 20), (2, 6, 12), (1, 3, 6), None, 0),
    ((3, 11, 20), (2, 6, 12), (1, 3, 6), None, 1),
    ((2, 6, 18), (2, 6, 12), (1, 3, 6), (2, 6, 18), 0),
    ((3, 5, 7), (2, 2, 3), (-1, 2, -3), None, 0),
    ((3, 5, 7), (2, 2, 3), (4, -7, 10), (5, 5, 8), 1),
    ((1, 1, 1), (1, 1, 1), (0, 0, 0), None, 0),
    ((4, 13, 9), (2, 6, 12), (0, 0, 0), (4, 18, 9), 0),
]


@pytest.mark.parametrize("grid,win,shift,padded,flags", BRUTE_CASES)
def test_index_map_matches_brute_force(grid, win, shift, padded, flags):
    P = padded or tuple(-(-g // w) * w for g, w in zip(grid, win))
    want = brute_force_index(grid, win, shift, P, flags)
    got = oracle.build_window_index(grid, win, shift, padded, flags)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("stage,padded", [
    (synth.STAGE_192, None), (synth.STAGE_384, synth.STAGE_384.padded),
    (synth.STAGE_384, (4, 96, 96)), (synth.TINY_PADDED, None)])
@pytest.mark.parametrize("flags", [0, 1])
def test_index_map_is_permutation_plus_pads(stage, padded, flags):
    m = oracle.build_window_index(stage.grid, synth.WINDOW, synth.SHIFT, padded, flags)
    P = padded or tuple(-(-g // w) * w for g, w in zip(stage.grid, synth.WINDOW))
    assert m.size == P[0] * P[1] * P[2] == oracle.window_index_count(stage.grid, synth.WINDOW, padded)
    real = m[m >= 0]
    assert ((m >= -1) & (m < stage.tokens)).all()
    assert real.size == stage.tokens
    assert np.array_equal(np.sort(real), np.arange(stage.tokens, dtype=np.int32))
    assert int((m == -1).sum()) == m.size - stage.tokens


def test_index_map_rejects_bad_extents():
    with pytest.raises(ValueError):
        oracle.build_window_index((2, 12, 24), (2, 6, 12), (1, 3, 6), (2, 11, 24))
    with pytest.raises(ValueError):
        oracle.build_window_index((2, 12, 24), (0, 6, 12), (1, 3, 6))


# ------------------------------------------------------------- gather ----

def _iota_rows(n, width):
    """Row r carries r in its first two elements' bit patterns; the rest are
    random bits, so any row mix-up or partial copy shows."""
    rng = np.random.default_rng(n)
    bits = rng.integers(0, 65536, (n, width), dtype=np.uint32).astype(np.uint16)
    r = np.arange(n, dtype=np.uint32)
    bits[:, 0] = (r & 0xFFFF).astype(np.uint16)
    bits[:, 1] = (r >> 16).astype(np.uint16)
    return bits.view(np.float16)


def test_gather_one_hot_probe():
    src = _iota_rows(1000, 192)
    idx = synth.random_index(3000, 1000, 0.2, seed=9).numpy()
    idx[5] = 1000      # out of range: zero row, counted
    idx[6] = -7        # below -1: zero row, counted
    dst, bad = oracle.window_gather(src, idx)
    assert bad == 2
    b = dst.view(np.uint16)
    for d in range(idx.size):
        if 0 <= idx[d] < 1000:
            assert int(b[d, 0]) | (int(b[d, 1]) << 16) == idx[d]
            assert np.array_equal(b[d], src.view(np.uint16)[idx[d]])
        else:
            assert not b[d].any()


def test_gather_window_map_places_tokens():
    st = synth.TINY_PADDED
    src = _iota_rows(st.tokens, 16)
    m = oracle.build_window_index(st.grid, synth.WINDOW, synth.SHIFT)
    dst, bad = oracle.window_gather(src, m)
    assert bad == 0
    b = dst.view(np.uint16)
    decoded = b[:, 0].astype(np.int64) | (b[:, 1].astype(np.int64) << 16)
    assert np.array_equal(decoded[m >= 0], m[m >= 0])
    assert not b[m < 0].any()


def test_norm_gather_is_ln_then_gather():
    st = synth.TINY_PADDED
    src = synth.gather_source(st.tokens, 192, seed=3).numpy()
    m = oracle.build_window_index(st.grid, synth.WINDOW, synth.SHIFT)
    fused, bad = oracle.norm_gather(src, m, EPS)
    assert bad == 0
    two_step, _ = oracle.window_gather(oracle.ln(src, EPS), m)
    assert np.array_equal(fused.view(np.uint16), two_step.view(np.uint16))


def test_gather_empty():
    dst, bad = oracle.window_gather(np.zeros((4, 8), np.float16), np.zeros(0, np.int32))
    assert dst.shape == (0, 8) and bad == 0


# --------------------------------------------------------------- GELU ----

def _torch_gelu64(t):
    return torch.nn.functional.gelu(torch.from_numpy(np.asarray(t, np.float64)),
                                    approximate="tanh").numpy()


def _close_to_torch(y64, t, ref):
    """torch evaluates 1 + tanh(u) literally in float64, which leaves an
    absolute error of a few 1e-16 * |t| where tanh(u) is near -1."""
    t = np.asarray(t, np.float64)
    return np.all(np.abs(y64 - ref) <= 1e-13 * np.abs(ref) + 4e-16 * np.abs(t))


def test_gelu_f32_matches_torch_float64():
    x, b = synth.gelu_input(64, 768, torch.float32, seed=4)
    x, b = x.numpy(), b.numpy()
    y, y64 = oracle.bias_gelu_tanh(x, b)
    t = x + b[None, :]  # numpy float32 add: one binary32 rounding
    ref = _torch_gelu64(t)
    assert _close_to_torch(y64, t, ref)
    assert np.array_equal(y, ref.astype(np.float32))


def test_gelu_tiny_page_input():
    rows, bias = gelu_tiny_input()
    x = np.array(rows, dtype=np.float32)
    b = np.array(bias, dtype=np.float32)
    _, y64 = oracle.bias_gelu_tanh(x, b)
    ref = _torch_gelu64(x + b[None, :])
    assert _close_to_torch(y64, x + b[None, :], ref)
    # the bias is indexed by column: a row-indexed bias would differ here
    wrong = _torch_gelu64(x + b[: x.shape[0], None])
    assert not np.allclose(y64, wrong)


def test_gelu_closed_forms():
    t = np.array([[0.0, 0.5, 1.0, 2.5, 6.0, 20.0]], dtype=np.float32)
    zero = np.zeros(t.shape[1], np.float32)
    _, gp = oracle.bias_gelu_tanh(t, zero)
    _, gm = oracle.bias_gelu_tanh(-t, zero)
    assert gp[0, 0] == 0.0
    # tanh is odd, so gelu(t) - gelu(-t) = t exactly in real arithmetic
    assert np.allclose(gp - gm, t.astype(np.float64), rtol=1e-15, atol=1e-15)
    assert gp[0, -1] == pytest.approx(20.0, rel=1e-15)
    # the tanh form, not the erf form: they differ by ~1.5e-4 at t = 1
    erf_gelu_1 = 0.5 * (1.0 + torch.erf(torch.tensor(1.0, dtype=torch.float64) / np.sqrt(2.0))).item()
    assert abs(gp[0, 2] - erf_gelu_1) > 1e-4


def _decimal_gelu(t: float) -> float:
    """The page's formula, literally, in 250-digit decimal arithmetic: there
    1 + tanh(u) loses nothing for the arguments used here."""
    import decimal
    with decimal.localcontext() as ctx:
        ctx.prec = 250
        D = decimal.Decimal
        pi = D("3.14159265358979323846264338327950288419716939937510582097494459230781640628620899")
        T = D(t)
        u = (D(2) / pi).sqrt() * (T + D("0.044715") * T * T * T)
        e2 = (2 * u).exp()
        tanh = (e2 - 1) / (e2 + 1)
        return float(D("0.5") * T * (1 + tanh))


def test_gelu_matches_high_precision_formula_far_left():
    ts = np.concatenate([np.linspace(-12.0, 12.0, 97), [-9.5, -7.25, -5.0, -3.3]]).astype(np.float32)
    x = ts[None, :]
    _, y64 = oracle.bias_gelu_tanh(x, np.zeros(ts.size, np.float32))
    want = np.array([_decimal_gelu(float(t)) for t in ts])
    rel = np.abs(y64[0] - want) / np.maximum(np.abs(want), 1e-300)
    assert rel.max() < 1e-13


def test_gelu_f16_rounding_point():
    x, b = synth.gelu_input(48, 1536, torch.float16, seed=4)
    x, b = x.numpy(), b.numpy()
    y, y64 = oracle.bias_gelu_tanh(x, b)
    t16 = x + b[None, :]  # numpy float16 add: fp16(fp32 x + fp32 b)
    ref = _torch_gelu64(t16.astype(np.float64))
    assert _close_to_torch(y64, t16, ref)
    assert np.array_equal(y.view(np.uint16), ref.astype(np.float16).view(np.uint16))


# ------------------------------------------------ the comparison rules ----

def _ln_fp32_shifted(x16, eps=EPS, unbiased=False, drop_eps=False):
    """An FP32 LayerNorm by the shifted-data two-pass method, in numpy."""
    x = x16.astype(np.float32)
    k = x[:, :1]
    xs = x - k
    m = xs.mean(axis=1, keepdims=True, dtype=np.float32)
    d = xs - m
    n = x.shape[1] - (1 if unbiased else 0)
    var = (d * d).sum(axis=1, keepdims=True, dtype=np.float32) / np.float32(n)
    rstd = np.float32(1) / np.sqrt(var + (np.float32(0) if drop_eps else np.float32(eps)))
    return (d * rstd).astype(np.float16)


def test_parity_rules_accept_fp32_rounding_and_reject_real_errors():
    """The fp16 comparison accepts what an FP32 evaluation produces and
    rejects a missing eps, an unbiased variance or a one-ulp bias."""
    from parity import check_fp16_near, check_ln
    x = synth.ln_input(256, 192, seed=12).numpy()
    y64, o16 = oracle.ln_f64(x, EPS), oracle.ln(x, EPS)
    check_ln(_ln_fp32_shifted(x), o16, y64, "fp32 evaluation")
    with pytest.raises(AssertionError):
        check_ln(_ln_fp32_shifted(x, unbiased=True), o16, y64, "unbiased variance")
    bumped = (o16.view(np.uint16) + (o16.view(np.uint16) % 7 == 0)).view(np.float16)
    with pytest.raises(AssertionError):
        check_fp16_near(bumped, o16, y64, "one ulp off")
    # rows with an offset and a variance close to eps expose an eps mistake
    xs = (np.float32(2.0) + synth.gather_source(256, 192, seed=2).numpy().astype(np.float32)
          * np.float32(0.003)).astype(np.float16)
    ys64, ys16 = oracle.ln_f64(xs, EPS), oracle.ln(xs, EPS)
    check_ln(_ln_fp32_shifted(xs), ys16, ys64, "small variance")
    with pytest.raises(AssertionError):
        check_ln(_ln_fp32_shifted(xs, drop_eps=True), ys16, ys64, "eps dropped")


# --------------------------------------------- block-boundary fusions ----

REV_CASES = [(synth.TINY, None, 0), (synth.TINY_PADDED, None, 0), (synth.TINY_PADDED, None, 1),
             (synth.STAGE_384, synth.STAGE_384.padded, 0)]


@pytest.mark.parametrize("stage,padded,flags", REV_CASES)
def test_window_reverse_undoes_the_window_gather(stage, padded, flags):
    m = oracle.build_window_index(stage.grid, synth.WINDOW, synth.SHIFT, padded, flags)
    x = synth.gather_source(stage.tokens, 64, seed=5).numpy()
    windows, _ = oracle.window_gather(x, m)
    r, _, bad = oracle.window_reverse_add_ln(np.zeros_like(x), windows, m)
    assert bad == 0
    assert np.array_equal(r.view(np.uint16), x.view(np.uint16))


@pytest.mark.parametrize("stage,padded,flags", REV_CASES[:3])
def test_window_reverse_add_ln_matches_numpy_composition(stage, padded, flags):
    m = oracle.build_window_index(stage.grid, synth.WINDOW, synth.SHIFT, padded, flags)
    res, _ = synth.residual_branch(stage.tokens, 192, seed=6)
    res = res.numpy()
    attn = synth.gather_source(m.size, 192, seed=7).numpy() * np.float16(0.1)
    r, y, bad = oracle.window_reverse_add_ln(res, attn, m, EPS)
    assert bad == 0
    # independent: numpy's own inverse by fancy assignment and its float16 add
    inv = np.full(stage.tokens, -1, dtype=np.int64)
    inv[m[m >= 0]] = np.nonzero(m >= 0)[0]
    want = res + attn[inv]
    assert np.array_equal(r.view(np.uint16), want.view(np.uint16))
    assert np.array_equal(y.view(np.uint16), oracle.ln(want, EPS).view(np.uint16))


def test_window_reverse_counts_uncovered_tokens():
    m = oracle.build_window_index(synth.TINY.grid, synth.WINDOW, synth.SHIFT)
    m2 = m.copy()
    lost = m2[5]
    m2[5] = -1
    res = synth.gather_source(synth.TINY.tokens, 64, seed=1).numpy()
    attn = synth.gather_source(m.size, 64, seed=2).numpy()
    r, _, bad = oracle.window_reverse_add_ln(res, attn, m2)
    assert bad == 1
    assert np.array_equal(r[lost].view(np.uint16), res[lost].view(np.uint16))


def test_invert_window_index():
    st = synth.TINY_PADDED
    m = oracle.build_window_index(st.grid, synth.WINDOW, synth.SHIFT)
    inv = oracle.invert_window_index(m, st.tokens)
    assert (inv >= 0).all()
    assert np.array_equal(m[inv], np.arange(st.tokens))
    assert np.array_equal(np.sort(inv), np.nonzero(m >= 0)[0])


def test_residual_add_norm_gather_matches_numpy_composition():
    st = synth.TINY_PADDED
    m = oracle.build_window_index(st.grid, synth.WINDOW, synth.SHIFT)
    a, b = synth.residual_branch(st.tokens, 192, seed=8)
    a, b = a.numpy(), b.numpy()
    r, dst, bad = oracle.residual_add_norm_gather(a, b, m, EPS)
    assert bad == 0
    want_r = a + b  # numpy float16 add: fp16(fp32 a + fp32 b)
    assert np.array_equal(r.view(np.uint16), want_r.view(np.uint16))
    ln = oracle.ln(want_r, EPS)
    want = np.where((m >= 0)[:, None], ln[np.maximum(m, 0)], np.float16(0))
    assert np.array_equal(dst.view(np.uint16), want.view(np.uint16))


# ------------------------------------------------------------ bfloat16 ----

def _all_bf16_bits():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _torch_bf16_of_bits(bits):
    return torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16)


def _bits_of_torch_bf16(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_decode_matches_torch_on_every_pattern():
    bits = _all_bf16_bits()
    ours = oracle.bf16_to_f64(bits)
    ref = _torch_bf16_of_bits(bits).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_rnbf16_round_trips_and_matches_torch():
    bits = _all_bf16_bits()
    vals = oracle.bf16_to_f64(bits)
    ok = ~np.isnan(vals)
    assert np.array_equal(oracle.rnbf16(vals[ok]), bits[ok])
    rng = np.random.default_rng(17)
    f = (np.exp2(rng.uniform(-140, 127, 300_000)) * rng.choice([-1, 1], 300_000)).astype(np.float32)
    want = _bits_of_torch_bf16(torch.from_numpy(f).to(torch.bfloat16))
    assert np.array_equal(oracle.rnbf16(f.astype(np.float64)), want)


def test_rnbf16_ties_go_to_even_and_range_edges():
    pos = oracle.bf16_to_f64(np.arange(0x7F80, dtype=np.uint16))  # +0 .. largest finite
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2.0
    lo_b, hi_b = oracle.rnbf16(lo), oracle.rnbf16(hi)
    assert np.array_equal(oracle.rnbf16(mid), np.where(lo_b % 2 == 0, lo_b, hi_b))
    bits = lambda v: int(oracle.rnbf16(np.array([v]))[0])
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127
    assert bits(big) == 0x7F7F
    assert bits((2.0 - 2.0 ** -8) * 2.0 ** 127) == 0x7F80   # tie above the largest finite
    assert bits(2.0 ** -133) == 0x0001
    assert bits(2.0 ** -134) == 0x0000                      # tie between 0 and 2^-133


def test_bf16_residual_add_ln():
    g = torch.Generator().manual_seed(3)
    a = torch.randn(96, 192, generator=g).to(torch.bfloat16)
    b = (torch.randn(96, 192, generator=g) * 0.1).to(torch.bfloat16)
    r, y = oracle.residual_add_ln(_bits_of_torch_bf16(a), _bits_of_torch_bf16(b), EPS, fmt="bf16")
    assert np.array_equal(r, _bits_of_torch_bf16(a + b))     # torch: fp32 add, round to bf16
    r64 = _torch_bf16_of_bits(r).double()
    ref = torch.nn.functional.layer_norm(r64, (192,), eps=EPS).numpy()
    assert np.max(np.abs(oracle.ln_f64(r, EPS, fmt="bf16") - ref)) < 1e-12
    assert np.array_equal(y, oracle.rnbf16(ref))


def test_bf16_gelu():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(32, 768, generator=g).to(torch.bfloat16)
    b = (torch.randn(768, generator=g) * 0.02).to(torch.bfloat16)
    y, y64 = oracle.bias_gelu_tanh(_bits_of_torch_bf16(x), _bits_of_torch_bf16(b), fmt="bf16")
    t = (x + b[None, :]).double()
    ref = torch.nn.functional.gelu(t, approximate="tanh").numpy()
    assert _close_to_torch(y64, t.numpy(), ref)
    assert np.array_equal(y, oracle.rnbf16(ref))


# ------------------------------------------------------- GELU backward ----

def test_gelu_backward_matches_torch_autograd_float64():
    g = torch.Generator().manual_seed(9)
    x = torch.randn(64, 96, generator=g, dtype=torch.float32)
    b = torch.randn(96, generator=g, dtype=torch.float32) * 0.02
    gy = torch.randn(64, 96, generator=g, dtype=torch.float32)
    gx, gb, gx64, gb64 = oracle.bias_gelu_tanh_bwd(gy.numpy(), x.numpy(), b.numpy())
    t = (x + b).double().requires_grad_(True)           # fp32 add, then exact
    torch.nn.functional.gelu(t, approximate="tanh").backward(gy.double())
    ref = t.grad.numpy()
    assert np.all(np.abs(gx64 - ref) <= 1e-13 * np.abs(ref) + 1e-15 * np.abs(gy.numpy()))
    assert np.array_equal(gx, ref.astype(np.float32))
    assert np.allclose(gb64, gx.astype(np.float64).sum(axis=0), rtol=1e-14, atol=0)


def _decimal_gelu_derivative(t: float) -> float:
    """Central difference of the page's formula in 250-digit decimal
    arithmetic with h = 1e-30 (truncation error ~1e-60)."""
    import decimal
    with decimal.localcontext() as ctx:
        ctx.prec = 250
        D = decimal.Decimal
        pi = D("3.14159265358979323846264338327950288419716939937510582097494459230781640628620899")
        k = (D(2) / pi).sqrt()

        def f(v):
            u = k * (v + D("0.044715") * v * v * v)
            e2 = (2 * u).exp()
            return D("0.5") * v * (1 + (e2 - 1) / (e2 + 1))

        h = D("1e-30")
        T = D(t)
        return float((f(T + h) - f(T - h)) / (2 * h))


def test_gelu_derivative_matches_high_precision_differences():
    ts = np.array([-11.0, -9.5, -7.0, -4.5, -2.0, -0.5, 0.0, 0.3, 1.7, 6.0], dtype=np.float32)
    one = np.ones((1, ts.size), np.float32)
    _, _, d64, _ = oracle.bias_gelu_tanh_bwd(one, ts[None, :], np.zeros(ts.size, np.float32))
    want = np.array([_decimal_gelu_derivative(float(t)) for t in ts])
    assert np.all(np.abs(d64[0] - want) <= 1e-13 * np.abs(want) + 1e-300), (d64[0], want)


def test_gelu_backward_16_bit_rounding_points():
    g = torch.Generator().manual_seed(10)
    for dt, fmt in ((torch.float16, "f16"), (torch.bfloat16, "bf16")):
        x = torch.randn(48, 64, generator=g).to(dt)
        b = (torch.randn(64, generator=g) * 0.02).to(dt)
        gy = torch.randn(48, 64, generator=g).to(dt)
        conv = (lambda a: a.numpy()) if fmt == "f16" else (lambda a: a.view(torch.int16).numpy().view(np.uint16))
        gx, gb, gx64, gb64 = oracle.bias_gelu_tanh_bwd(conv(gy), conv(x), conv(b), fmt=fmt)
        t = (x + b).double().requires_grad_(True)       # 16-bit add rounds t, then exact
        torch.nn.functional.gelu(t, approximate="tanh").backward(gy.double())
        ref = t.grad
        assert np.allclose(gx64, ref.numpy(), rtol=1e-13, atol=1e-15)
        want_gx = conv(ref.to(dt))
        assert np.array_equal(gx, want_gx)
        exact_sum = ref.to(dt).double().sum(0)         # sum of the rounded gradients
        assert np.allclose(gb64, exact_sum.numpy(), rtol=1e-14, atol=1e-15)
        assert np.array_equal(gb, conv(exact_sum.to(dt)))


# ------------------------------------------------------------ bias-mask ----

from golden_io import shift_region_cases  # noqa: E402


def _window_rows(P, win):
    """Cells of every window in the destination order: [(window_id, [(z,h,w), ...])]."""
    nwin = [-(-P[k] // win[k]) for k in range(3)]
    out = []
    for bz, bh, bw in itertools.product(*(range(m) for m in nwin)):
        lo = (bz * win[0], bh * win[1], bw * win[2])
        hi = [min(lo[k] + win[k], P[k]) for k in range(3)]
        out.append(list(itertools.product(*(range(lo[k], hi[k]) for k in range(3)))))
    return out


@pytest.mark.parametrize("name", sorted(shift_region_cases()))
def test_shift_regions_match_worked_fixture(name):
    c = shift_region_cases()[name]
    lab = oracle.build_shift_regions(c["grid"], c["win"], c["shift"], c["padded"], c["flags"],
                                     c["axes"])
    rows = _window_rows(c["padded"], c["win"])
    assert lab.size == sum(len(r) for r in rows)
    start = np.cumsum([0] + [len(r) for r in rows])
    assert sorted(c["windows"]) == list(range(len(rows)))
    for wid, want in c["windows"].items():
        assert list(lab[start[wid]:start[wid + 1]]) == want, (name, wid)


def _swin_slice_ids(P, win, shift):
    """Region ids of the classic shifted-window mask: on the padded grid,
    each axis is cut into [0, P-w), [P-w, P-s), [P-s, P) (one slice when
    s = 0) and every cell gets the index of its slice triple."""
    ids = np.zeros(P, dtype=np.int64)
    cnt = 0
    cuts = []
    for k in range(3):
        s = shift[k] % P[k]
        cuts.append([slice(0, P[k] - win[k]), slice(P[k] - win[k], P[k] - s), slice(P[k] - s, P[k])]
                    if s else [slice(0, P[k])])
    for a in cuts[0]:
        for b in cuts[1]:
            for c in cuts[2]:
                ids[a, b, c] = cnt
                cnt += 1
    return ids


@pytest.mark.parametrize("grid,win,shift", [((4, 12, 24), (2, 6, 12), (1, 3, 6)),
                                            ((3, 11, 20), (2, 6, 12), (1, 3, 6)),
                                            ((2, 6, 8), (2, 3, 4), (1, 1, 2)),
                                            ((4, 6, 6), (2, 3, 3), (1, 2, 1))])
def test_shift_regions_partition_windows_like_the_classic_slice_mask(grid, win, shift):
    # pad-then-shift on full windows is the classic construction's setting
    P = [-(-grid[k] // win[k]) * win[k] for k in range(3)]
    lab = oracle.build_shift_regions(grid, win, shift, None, 1, 7)
    ids = _swin_slice_ids(P, win, shift)
    d = 0
    for cells in _window_rows(P, win):
        ours = lab[d:d + len(cells)]
        theirs = np.array([ids[c] for c in cells])
        assert np.array_equal(ours[:, None] == ours[None, :], theirs[:, None] == theirs[None, :])
        d += len(cells)
    assert d == lab.size


@pytest.mark.parametrize("flags", [0, 1])
@pytest.mark.parametrize("axes", [7, 3, 4])
def test_shift_regions_separate_exactly_the_rows_the_roll_cut_apart(flags, axes):
    # Two tokens of a window share a region iff, along every masked axis,
    # their source coordinates are as far apart as their cells (the roll
    # put no seam between them).  Checked on real tokens through the index
    # map, with no use of the label formula.
    grid, win, shift = (3, 11, 20), (2, 6, 12), (1, 3, 6)
    P = [-(-grid[k] // win[k]) * win[k] for k in range(3)]
    idx = oracle.build_window_index(grid, win, shift, None, flags)
    lab = oracle.build_shift_regions(grid, win, shift, None, flags, axes)
    d = 0
    for cells in _window_rows(P, win):
        rows = [(c, idx[d + i], lab[d + i]) for i, c in enumerate(cells) if idx[d + i] >= 0]
        for (c1, t1, l1), (c2, t2, l2) in itertools.combinations(rows, 2):
            s1 = np.unravel_index(t1, grid)
            s2 = np.unravel_index(t2, grid)
            together = all(s2[k] - s1[k] == c2[k] - c1[k] for k in range(3) if (axes >> k) & 1)
            assert (l1 == l2) == together, (c1, c2)
        d += len(cells)


def test_shift_regions_without_shift_are_one_region():
    lab = oracle.build_shift_regions((4, 11, 20), (2, 6, 12), (0, 0, 0), None, 0, 7)
    assert lab.size == 4 * 12 * 24 and not lab.any()


def _torch_bias_mask(s, b, win_type, region, mask_value, tdtype):
    """The eager sequence attn + bias; attn + mask in the tensor format."""
    t = s + b[torch.as_tensor(win_type, dtype=torch.long)]
    if region is None:
        return t
    r = torch.as_tensor(region).view(s.shape[0], 1, s.shape[2])
    m = torch.where(r.transpose(1, 2) == r, torch.tensor(0.0), torch.tensor(float(mask_value)))
    return t + m.to(tdtype).unsqueeze(1)


def _as_np(t, fmt):
    return t.numpy() if fmt == "f16" else t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("fmt,tdtype", [("f16", torch.float16), ("bf16", torch.bfloat16)])
@pytest.mark.parametrize("masked", [True, False])
def test_bias_mask_add_matches_the_eager_torch_sequence(fmt, tdtype, masked):
    n_win, heads, n, n_types = 6, 3, 24, 2
    s, b = synth.attention_logits(n_win, heads, n, n_types, seed=11, dtype=tdtype)
    s = s.clone()
    flat = s.view(-1)
    # special values: signed zeros, infinities, NaN, overflow, exact cancellation
    big = 60000.0 if fmt == "f16" else 3.0e38
    flat[:8] = torch.tensor([0.0, -0.0, float("inf"), -float("inf"), float("nan"), big, -big, 1.0],
                            dtype=tdtype)
    b.view(-1)[:8] = torch.tensor([-0.0, -0.0, 1.0, -1.0, 0.0, big, -big, -1.0], dtype=tdtype)
    win_type = np.arange(n_win, dtype=np.int32) % n_types
    region = (np.arange(n_win * n, dtype=np.int32) // 5) % 3 if masked else None
    ours = oracle.window_bias_mask_add(_as_np(s, fmt), _as_np(b, fmt), win_type, region, -100.0,
                                       fmt=fmt)
    ref = _as_np(_torch_bias_mask(s, b, win_type, region, -100.0, tdtype), fmt)
    dec = oracle.f16_to_f64 if fmt == "f16" else oracle.bf16_to_f64
    o, r = dec(ours), dec(ref)
    assert np.array_equal(np.isnan(o), np.isnan(r))
    ok = ~np.isnan(o)
    assert np.array_equal(o[ok], r[ok])
    assert np.array_equal(np.signbit(o[ok]), np.signbit(r[ok]))   # -0 + 0 = +0 when masked


def test_bias_mask_add_uses_the_window_type_and_both_rounding_points():
    # a bias picked by row instead of window type, or one rounding instead
    # of two, changes these values
    s = np.array([[[[1.0, 2048.0], [0.5, -3.0]]]], dtype=np.float16)      # [1,1,2,2]
    b = np.array([[[[0.0, 0.0], [0.0, 0.0]]], [[[0.25, 1.0], [0.0009765625, 0.5]]]],
                 dtype=np.float16)                                       # [2,1,2,2]
    out = oracle.window_bias_mask_add(s, b, np.array([1], np.int32), np.array([0, 1], np.int32),
                                      -100.0)
    # (1 + 0.25) -> 1.25; masked pair (0,1): 2048 + 1 -> 2048 (tie to even), then -100 -> 1948
    # (1,0): 0.5 + 2^-10 = 0.5009765625, then -100 -> -99.5 (one rounding would give -99.5 too,
    # so (1,1) checks the second point: -3 + 0.5 = -2.5 exactly, unmasked)
    assert out.ravel().tolist() == [1.25, 1948.0, -99.5, -2.5]
    one_round = np.float16(np.float64(2048.0) + 1.0 - 100.0)
    assert one_round != np.float16(1948.0)
