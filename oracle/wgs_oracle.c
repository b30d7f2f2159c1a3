/*
 * CPU oracle for the shifted-window transformer block-glue path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library: every step below is written out from the definition it
 * cites, in double precision, one element at a time, with no blocking,
 * fusion or reordering.
 *
 * Sources (page title, section):
 *   [P1] "BW1000 gfx936 Pangu-Weather inference profiling" (l189.com news
 *        2144533): s3 fixed-width LayerNorm, s4 residual add + norm and its
 *        FP16 rounding point, s5 window gather with the INT32 index protocol
 *        and the fused norm-gather.
 *        s1, s7 the restore path after attention; s6, s7 the "bias-mask" op
 *        kept in the final combination (its arithmetic is a reading, see
 *        orc_window_bias_mask_add_fmt).
 *   [P3] "PyTorch + HIP fused bias + GELU on Hygon DCU" (forum.sourcefind.cn):
 *        s3 math semantics (tanh-approximate GELU of input + bias); the
 *        backward it leaves out is the derivative of that formula.
 *        s10, s12 other formats as hardening (bfloat16 here).
 *
 * fp16 values travel as their IEEE binary16 bit patterns (uint16_t).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* IEEE-754 binary16 <-> double                                        */
/* ------------------------------------------------------------------ */

/* Exact value of a binary16 bit pattern (IEEE 754-2008, s3.4). */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);             /* subnormal or zero */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round q >= 0 (an integer plus a fraction, exactly representable) to the
 * nearest integer, ties to the even integer. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double frac = q - fl;
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* double -> binary16 bits, round to nearest, ties to even (IEEE 754-2008
 * s4.3.1).  Overflow goes to infinity, tiny values to subnormals or zero,
 * NaN stays NaN (quiet), the sign of zero is kept. */
uint16_t orc_rn16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return (uint16_t)(sign | 0x7E00);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00);
    /* 65504 is the largest finite value; the midpoint between it and 2^16
     * is 65520, and a tie there goes to the even neighbour 2^16 = inf. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: the quantum is 2^-24 */
        double n = round_half_even(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)n); /* n == 1024 encodes 2^-14 */
    }
    int ex;
    frexp(a, &ex);                 /* a = m * 2^ex, m in [0.5, 1) */
    int E = ex - 1;                 /* a = (2m) * 2^E, 2m in [1, 2) */
    double n = round_half_even(ldexp(a, 10 - E)); /* in [1024, 2048] */
    if (n == 2048.0) { n = 1024.0; E += 1; }
    if (E + 15 >= 31) return (uint16_t)(sign | 0x7C00);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(n - 1024.0));
}

/* Element-wise forms of the two conversions above. */
void orc_rn16_array(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_rn16(v[i]);
}

void orc_f16_to_f64_array(const uint16_t *h, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f64(h[i]);
}

/* bfloat16: the top half of a binary32 (8 exponent bits, 7 fraction bits). */
double orc_bf16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int m = h & 0x7F;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -133);            /* subnormal or zero */
    } else if (e == 255) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + m), e - 134); /* (1 + m/128) * 2^(e-127) */
    }
    return sign ? -v : v;
}

/* double -> bfloat16 bits, round to nearest, ties to even, as orc_rn16 but
 * with 7 fraction bits and binary32's exponent range. */
uint16_t orc_rnbf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return (uint16_t)(sign | 0x7FC0);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    /* largest finite (2 - 2^-7) 2^127; the midpoint to 2^128 ties to inf */
    if (a >= ldexp(2.0 - ldexp(1.0, -8), 127)) return (uint16_t)(sign | 0x7F80);
    if (a < ldexp(1.0, -126)) {
        double n = round_half_even(ldexp(a, 133)); /* quantum 2^-133 */
        return (uint16_t)(sign | (uint16_t)n);
    }
    int ex;
    frexp(a, &ex);
    int E = ex - 1;
    double n = round_half_even(ldexp(a, 7 - E)); /* in [128, 256] */
    if (n == 256.0) { n = 128.0; E += 1; }
    if (E + 127 >= 255) return (uint16_t)(sign | 0x7F80);
    return (uint16_t)(sign | (uint16_t)((E + 127) << 7) | (uint16_t)(n - 128.0));
}

void orc_rnbf16_array(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_rnbf16(v[i]);
}

void orc_bf16_to_f64_array(const uint16_t *h, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f64(h[i]);
}

/* The 16-bit storage formats of the row ops: fmt 0 = binary16, 1 = bfloat16. */
static double dec16(uint16_t h, int fmt) { return fmt ? orc_bf16_to_f64(h) : orc_f16_to_f64(h); }
static uint16_t enc16(double v, int fmt) { return fmt ? orc_rnbf16(v) : orc_rn16(v); }

/* ------------------------------------------------------------------ */
/* LayerNorm without affine  [P1 s3]                                   */
/* ------------------------------------------------------------------ */

/* One row, unrounded: y = (x - mean) / sqrt(var + eps) with the biased
 * (divide by width) variance, both statistics taken in two passes.  eps
 * is the single-precision value the caller passes. */
void orc_ln_row_f64(const double *x, double *y, int32_t width, float eps)
{
    double mean = 0.0;
    for (int32_t i = 0; i < width; ++i) mean += x[i];
    mean /= (double)width;
    double var = 0.0;
    for (int32_t i = 0; i < width; ++i) {
        double d = x[i] - mean;
        var += d * d;
    }
    var /= (double)width;
    double denom = sqrt(var + (double)eps);
    for (int32_t i = 0; i < width; ++i) y[i] = (x[i] - mean) / denom;
}

/* 16-bit rows in, 16-bit rows out (format fmt): each output is the rounding
 * of the exact (double) normalised value. */
void orc_ln_fmt(const uint16_t *x, uint16_t *y, int64_t rows, int32_t width, float eps, int fmt)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)width);
    double *yd = (double *)malloc(sizeof(double) * (size_t)width);
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * (int64_t)width;
        for (int32_t i = 0; i < width; ++i) xd[i] = dec16(xr[i], fmt);
        orc_ln_row_f64(xd, yd, width, eps);
        for (int32_t i = 0; i < width; ++i) y[r * (int64_t)width + i] = enc16(yd[i], fmt);
    }
    free(xd);
    free(yd);
}

void orc_ln(const uint16_t *x, uint16_t *y, int64_t rows, int32_t width, float eps)
{
    orc_ln_fmt(x, y, rows, width, eps, 0);
}

/* Unrounded LN outputs of 16-bit rows, for tolerance decisions. */
void orc_ln_f64_fmt(const uint16_t *x, double *y, int64_t rows, int32_t width, float eps, int fmt)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)width);
    for (int64_t r = 0; r < rows; ++r) {
        for (int32_t i = 0; i < width; ++i) xd[i] = dec16(x[r * (int64_t)width + i], fmt);
        orc_ln_row_f64(xd, y + r * (int64_t)width, width, eps);
    }
    free(xd);
}

void orc_ln_f64(const uint16_t *x, double *y, int64_t rows, int32_t width, float eps)
{
    orc_ln_f64_fmt(x, y, rows, width, eps, 0);
}

/* ------------------------------------------------------------------ */
/* Residual add + LayerNorm  [P1 s4]                                   */
/* ------------------------------------------------------------------ */

/* residual_out = fp16(residual + branch); y = LN(residual_out), taken from
 * the rounded fp16 value.  The page states the sum as fp16(fp32 a + fp32 b);
 * the sum of two binary16 values is exact in double, and since binary32
 * carries 24 >= 2*11 + 2 significand bits, rounding first to binary32 and
 * then to binary16 gives the same result as rounding the exact sum once
 * (Figueroa, "When is double rounding innocuous?", 1995). */
void orc_residual_add_ln_fmt(const uint16_t *a, const uint16_t *b, uint16_t *r_out, uint16_t *y,
                             int64_t rows, int32_t width, float eps, int fmt)
{
    int64_t n = rows * (int64_t)width;
    for (int64_t i = 0; i < n; ++i) r_out[i] = enc16(dec16(a[i], fmt) + dec16(b[i], fmt), fmt);
    orc_ln_fmt(r_out, y, rows, width, eps, fmt);
}

/* bfloat16 (fmt 1) keeps the same rounding point: binary32's 24 bits are
 * at least 2 * 8 + 2, so fp32 then bfloat16 equals one rounding of the
 * exact sum. */
void orc_residual_add_ln(const uint16_t *a, const uint16_t *b, uint16_t *r_out, uint16_t *y,
                         int64_t rows, int32_t width, float eps)
{
    orc_residual_add_ln_fmt(a, b, r_out, y, rows, width, eps, 0);
}

/* ------------------------------------------------------------------ */
/* Shifted-window index map  [P1 s5]                                   */
/* ------------------------------------------------------------------ */
/*
 * The page fixes the protocol (one INT32 per destination row; a value >= 0
 * names the source token, -1 asks for a zero row) but not the construction.
 * The reading taken here:
 *   - tokens are the row-major flattening of a (Z, H, W) grid;
 *   - the padded grid has extents padded[] (each >= the grid extent), by
 *     default each extent rounded up to a multiple of the window;
 *   - windows tile the padded grid from the origin; where a padded extent is
 *     not a multiple of the window, the last window on that axis is cut short;
 *   - destination rows are ordered window by window (row-major over the
 *     window grid), then row-major over the cells inside each window;
 *   - flags == 0 (shift, then pad): a cell (z,h,w) inside the original grid
 *     reads source ((z+sz) mod Z, (h+sh) mod H, (w+sw) mod W), a cyclic roll
 *     by -shift; cells outside it are pads (-1);
 *   - flags == 1 (pad, then shift): the roll runs over the padded grid and a
 *     cell whose rolled position falls outside the original grid is a pad.
 *
 * This builder scatters: for every padded cell it computes where that cell
 * lands in the destination order.
 */

static int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }
static int64_t pos_mod(int64_t a, int64_t m) { int64_t r = a % m; return r < 0 ? r + m : r; }

static int resolve_padded(const int32_t grid[3], const int32_t win[3], const int32_t *padded,
                          int64_t P[3])
{
    for (int k = 0; k < 3; ++k) {
        if (grid[k] < 1 || win[k] < 1) return -1;
        P[k] = padded ? (int64_t)padded[k] : ceil_div64(grid[k], win[k]) * win[k];
        if (P[k] < grid[k]) return -1;
    }
    return 0;
}

int64_t orc_window_index_count(const int32_t grid[3], const int32_t win[3], const int32_t *padded)
{
    int64_t P[3];
    if (resolve_padded(grid, win, padded, P) != 0) return -1;
    return P[0] * P[1] * P[2];
}

int orc_build_window_index(const int32_t grid[3], const int32_t win[3], const int32_t shift[3],
                           const int32_t *padded, int32_t flags, int32_t *out)
{
    int64_t P[3];
    if (resolve_padded(grid, win, padded, P) != 0) return -1;
    if (flags != 0 && flags != 1) return -1;
    const int64_t Z = grid[0], H = grid[1], W = grid[2];
    int64_t nwin[3];
    for (int k = 0; k < 3; ++k) nwin[k] = ceil_div64(P[k], win[k]);

    /* size of every window, then where each window starts in the output */
    int64_t n_windows = nwin[0] * nwin[1] * nwin[2];
    int64_t *start = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_windows + 1));
    if (!start) return -2;
    start[0] = 0;
    for (int64_t bz = 0; bz < nwin[0]; ++bz)
        for (int64_t bh = 0; bh < nwin[1]; ++bh)
            for (int64_t bw = 0; bw < nwin[2]; ++bw) {
                int64_t ez = P[0] - bz * win[0]; if (ez > win[0]) ez = win[0];
                int64_t eh = P[1] - bh * win[1]; if (eh > win[1]) eh = win[1];
                int64_t ew = P[2] - bw * win[2]; if (ew > win[2]) ew = win[2];
                int64_t w_id = (bz * nwin[1] + bh) * nwin[2] + bw;
                start[w_id + 1] = start[w_id] + ez * eh * ew;
            }

    for (int64_t z = 0; z < P[0]; ++z)
        for (int64_t h = 0; h < P[1]; ++h)
            for (int64_t w = 0; w < P[2]; ++w) {
                int64_t bz = z / win[0], bh = h / win[1], bw = w / win[2];
                int64_t iz = z % win[0], ih = h % win[1], iw = w % win[2];
                int64_t eh = P[1] - bh * win[1]; if (eh > win[1]) eh = win[1];
                int64_t ew = P[2] - bw * win[2]; if (ew > win[2]) ew = win[2];
                int64_t w_id = (bz * nwin[1] + bh) * nwin[2] + bw;
                int64_t dst = start[w_id] + (iz * eh + ih) * ew + iw;

                int64_t src = -1;
                if (flags == 0) {
                    if (z < Z && h < H && w < W) {
                        int64_t zs = pos_mod(z + shift[0], Z);
                        int64_t hs = pos_mod(h + shift[1], H);
                        int64_t ws = pos_mod(w + shift[2], W);
                        src = (zs * H + hs) * W + ws;
                    }
                } else {
                    int64_t zs = pos_mod(z + shift[0], P[0]);
                    int64_t hs = pos_mod(h + shift[1], P[1]);
                    int64_t ws = pos_mod(w + shift[2], P[2]);
                    if (zs < Z && hs < H && ws < W) src = (zs * H + hs) * W + ws;
                }
                out[dst] = (int32_t)src;
            }
    free(start);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Window gather and fused norm-gather  [P1 s5]                        */
/* ------------------------------------------------------------------ */

/* dst[d] = src[idx[d]] for idx[d] >= 0 (bit copy), an all-zero row for
 * idx[d] == -1.  Any other index is outside the protocol: the oracle writes
 * a zero row for it and counts it in the return value. */
int64_t orc_window_gather(const uint16_t *src, const int32_t *idx, uint16_t *dst,
                          int64_t n_src, int64_t n_idx, int32_t width)
{
    int64_t bad = 0;
    for (int64_t d = 0; d < n_idx; ++d) {
        int64_t s = idx[d];
        int ok = (s >= 0 && s < n_src);
        if (!ok && s != -1) ++bad;
        for (int32_t i = 0; i < width; ++i)
            dst[d * (int64_t)width + i] = ok ? src[s * (int64_t)width + i] : (uint16_t)0;
    }
    return bad;
}

/* dst[d] = LN(src[idx[d]]) for idx[d] >= 0, zero row for -1: the
 * normalised tensor is defined row by row, so this is LN applied to each
 * gathered row. */
int64_t orc_norm_gather_fmt(const uint16_t *src, const int32_t *idx, uint16_t *dst,
                            int64_t n_src, int64_t n_idx, int32_t width, float eps, int fmt)
{
    int64_t bad = 0;
    for (int64_t d = 0; d < n_idx; ++d) {
        int64_t s = idx[d];
        uint16_t *out = dst + d * (int64_t)width;
        if (s >= 0 && s < n_src) {
            orc_ln_fmt(src + s * (int64_t)width, out, 1, width, eps, fmt);
        } else {
            if (s != -1) ++bad;
            for (int32_t i = 0; i < width; ++i) out[i] = 0;
        }
    }
    return bad;
}

int64_t orc_norm_gather(const uint16_t *src, const int32_t *idx, uint16_t *dst,
                        int64_t n_src, int64_t n_idx, int32_t width, float eps)
{
    return orc_norm_gather_fmt(src, idx, dst, n_src, n_idx, width, eps, 0);
}

/* ------------------------------------------------------------------ */
/* Bias + tanh-approximate GELU  [P3 s3]                               */
/* ------------------------------------------------------------------ */

/* gelu(t) = 0.5 t (1 + tanh(u)),  u = sqrt(2/pi) (t + 0.044715 t^3).
 * For u < 0 the sum 1 + tanh(u) cancels (in double it is exactly 0 once
 * u < -18.7, i.e. t < -5.6 gives a wrong result long before that), so there
 * it is evaluated through the exact identity 1 + tanh(u) = 2 e^{2u} / (1 + e^{2u}). */
static double gelu_tanh(double t)
{
    const double k = sqrt(2.0 / acos(-1.0));
    const double u = k * (t + 0.044715 * t * t * t);
    double one_plus_tanh;
    if (u >= 0.0) {
        one_plus_tanh = 1.0 + tanh(u);
    } else {
        const double e = exp(2.0 * u);
        one_plus_tanh = 2.0 * e / (1.0 + e);
    }
    return 0.5 * t * one_plus_tanh;
}

/* fp32: t = fp32(x + bias[col]) (the sum of two floats rounded once to
 * binary32; going through double first is innocuous since 53 >= 2*24 + 2),
 * y64 = gelu(t) exactly in double, y = fp32(y64). */
void orc_bias_gelu_f32(const float *x, const float *bias, float *y, double *y64,
                       int64_t rows, int32_t width)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int32_t c = 0; c < width; ++c) {
            int64_t i = r * (int64_t)width + c;
            float t = (float)((double)x[i] + (double)bias[c]);
            double g = gelu_tanh((double)t);
            if (y64) y64[i] = g;
            if (y) y[i] = (float)g;
        }
}

/* 16-bit formats: t = fp16(x + bias[col]) (or bfloat16), keeping the
 * rounding point an eager `gelu(x + bias)` in that precision would have;
 * y = round(gelu(t)). */
void orc_bias_gelu_16(const uint16_t *x, const uint16_t *bias, uint16_t *y, double *y64,
                      int64_t rows, int32_t width, int fmt)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int32_t c = 0; c < width; ++c) {
            int64_t i = r * (int64_t)width + c;
            uint16_t t = enc16(dec16(x[i], fmt) + dec16(bias[c], fmt), fmt);
            double g = gelu_tanh(dec16(t, fmt));
            if (y64) y64[i] = g;
            if (y) y[i] = enc16(g, fmt);
        }
}

void orc_bias_gelu_f16(const uint16_t *x, const uint16_t *bias, uint16_t *y, double *y64,
                       int64_t rows, int32_t width)
{
    orc_bias_gelu_16(x, bias, y, y64, rows, width, 0);
}

/* ------------------------------------------------------------------ */
/* Window reverse fused with residual add + LN                         */
/* ------------------------------------------------------------------ */
/* [P1 s7] keeps a "restore path" custom op; [P1 s1] counts two
 * index_select calls per block (32 over 16 blocks).  The plainest reading:
 * after window attention the windowed rows go back to token order (the
 * inverse of the s5 gather: crop pads, undo the window order and the cyclic
 * shift), are added to the residual stream and normalised (norm2), keeping
 * the s4 rounding point:
 *     r[t] = fp16(residual[t] + attn[d])  for the windowed row d with idx[d] = t
 *     y[t] = LN(r[t])
 * It is written here as a scatter through the forward map idx.  A token
 * that no windowed row names takes a zero branch (r = residual) and is
 * counted, as is a token named more than once (the last row wins).
 * Returns that count (0 for any map from orc_build_window_index). */
int64_t orc_window_reverse_add_ln_fmt(const uint16_t *residual, const uint16_t *attn,
                                      const int32_t *idx, uint16_t *r_out, uint16_t *y,
                                      int64_t n_tokens, int64_t n_idx, int32_t width, float eps,
                                      int fmt)
{
    int32_t *seen = (int32_t *)calloc((size_t)(n_tokens > 0 ? n_tokens : 1), sizeof(int32_t));
    for (int64_t t = 0; t < n_tokens * (int64_t)width; ++t) r_out[t] = residual[t];
    for (int64_t d = 0; d < n_idx; ++d) {
        int64_t t = idx[d];
        if (t < 0 || t >= n_tokens) continue;
        seen[t] += 1;
        for (int32_t i = 0; i < width; ++i) {
            int64_t k = t * (int64_t)width + i;
            r_out[k] = enc16(dec16(residual[k], fmt) + dec16(attn[d * (int64_t)width + i], fmt), fmt);
        }
    }
    int64_t bad = 0;
    for (int64_t t = 0; t < n_tokens; ++t) bad += seen[t] != 1;
    free(seen);
    orc_ln_fmt(r_out, y, n_tokens, width, eps, fmt);
    return bad;
}

int64_t orc_window_reverse_add_ln(const uint16_t *residual, const uint16_t *attn,
                                  const int32_t *idx, uint16_t *r_out, uint16_t *y,
                                  int64_t n_tokens, int64_t n_idx, int32_t width, float eps)
{
    return orc_window_reverse_add_ln_fmt(residual, attn, idx, r_out, y, n_tokens, n_idx, width,
                                         eps, 0);
}

/* token -> windowed row: inv[idx[d]] = d; tokens no row names get -1 */
void orc_invert_window_index(const int32_t *idx, int64_t n_idx, int32_t *inv, int64_t n_tokens)
{
    for (int64_t t = 0; t < n_tokens; ++t) inv[t] = -1;
    for (int64_t d = 0; d < n_idx; ++d)
        if (idx[d] >= 0 && idx[d] < n_tokens) inv[idx[d]] = (int32_t)d;
}

/* ------------------------------------------------------------------ */
/* Residual add + norm1 + shifted-window gather                        */
/* ------------------------------------------------------------------ */
/* The block boundary: the residual stream r = fp16(a + b) is written out
 * ([P1 s4]) and the next block's norm1 output is consumed only by its
 * window gather ([P1 s5]), so
 *     r = fp16(a + b),   dst[d] = LN(r)[idx[d]]  (zero row for -1).
 * Written as the composition of the two definitions above.  Returns the
 * number of indices outside [-1, n_src). */
int64_t orc_residual_add_norm_gather_fmt(const uint16_t *a, const uint16_t *b, const int32_t *idx,
                                         uint16_t *r_out, uint16_t *dst, int64_t n_src,
                                         int64_t n_idx, int32_t width, float eps, int fmt)
{
    uint16_t *y = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(n_src * (int64_t)width + 1));
    orc_residual_add_ln_fmt(a, b, r_out, y, n_src, width, eps, fmt);
    int64_t bad = orc_window_gather(y, idx, dst, n_src, n_idx, width);
    free(y);
    return bad;
}

int64_t orc_residual_add_norm_gather(const uint16_t *a, const uint16_t *b, const int32_t *idx,
                                     uint16_t *r_out, uint16_t *dst, int64_t n_src,
                                     int64_t n_idx, int32_t width, float eps)
{
    return orc_residual_add_norm_gather_fmt(a, b, idx, r_out, dst, n_src, n_idx, width, eps, 0);
}

/* ------------------------------------------------------------------ */
/* Backward of bias + tanh-GELU                                        */
/* ------------------------------------------------------------------ */
/* [P3 s3] lists backward among what its tutorial op leaves out; this is the
 * gradient of y = gelu(x + bias) with the rounding points of an eager
 * backward (gelu backward in the tensor dtype, then a column sum):
 *     t          = round(x + bias[c])                   (as the forward)
 *     grad_x     = round(grad_y * gelu'(t))
 *     grad_bias  = round(sum over rows of grad_x[., c])  (exact sum)
 * With s = sigma(2u) = 0.5 (1 + tanh(u)), u = sqrt(2/pi)(t + 0.044715 t^3):
 *     gelu'(t) = s + t * 2 s (1 - s) * sqrt(2/pi) (1 + 3 * 0.044715 t^2),
 * the derivative of t * s; s and 1 - s = sigma(-2u) are each evaluated on
 * the side where they do not cancel. */
static double sigmoid_exact(double z)
{
    if (z >= 0.0) return 1.0 / (1.0 + exp(-z));
    const double e = exp(z);
    return e / (1.0 + e);
}

static double gelu_tanh_grad(double t)
{
    const double k = sqrt(2.0 / acos(-1.0));
    const double u = k * (t + 0.044715 * t * t * t);
    const double s = sigmoid_exact(2.0 * u), one_minus_s = sigmoid_exact(-2.0 * u);
    return s + t * 2.0 * s * one_minus_s * k * (1.0 + 3.0 * 0.044715 * t * t);
}

/* fmt: -1 = binary32, 0 = binary16, 1 = bfloat16.  Values travel as raw
 * element bits (uint32 for binary32, uint16 otherwise).  gx64 / gb64, when
 * given, receive the unrounded products and sums. */
static double dec_any(const void *p, int64_t i, int fmt)
{
    if (fmt < 0) { float f; uint32_t b = ((const uint32_t *)p)[i]; memcpy(&f, &b, 4); return f; }
    return dec16(((const uint16_t *)p)[i], fmt);
}

static void enc_any(void *p, int64_t i, double v, int fmt)
{
    if (fmt < 0) { float f = (float)v; uint32_t b; memcpy(&b, &f, 4); ((uint32_t *)p)[i] = b; }
    else ((uint16_t *)p)[i] = enc16(v, fmt);
}

void orc_bias_gelu_bwd(const void *grad_y, const void *x, const void *bias, void *grad_x,
                       void *grad_bias, double *gx64, double *gb64, int64_t rows, int32_t width,
                       int fmt)
{
    double *sum = (double *)calloc((size_t)(width > 0 ? width : 1), sizeof(double));
    for (int64_t r = 0; r < rows; ++r)
        for (int32_t c = 0; c < width; ++c) {
            int64_t i = r * (int64_t)width + c;
            double t = dec_any(x, i, fmt) + dec_any(bias, c, fmt);
            if (fmt < 0) t = (double)(float)t;   /* binary32 add: one rounding */
            else t = dec16(enc16(t, fmt), fmt);
            double g = dec_any(grad_y, i, fmt) * gelu_tanh_grad(t);
            if (gx64) gx64[i] = g;
            enc_any(grad_x, i, g, fmt);
            sum[c] += dec_any(grad_x, i, fmt);     /* the rounded gradient, summed exactly */
        }
    for (int32_t c = 0; c < width; ++c) {
        if (gb64) gb64[c] = sum[c];
        enc_any(grad_bias, c, sum[c], fmt);
    }
    free(sum);
}

/* ------------------------------------------------------------------ */
/* Shifted-window attention bias and mask ("bias-mask")  [P1 s7]       */
/* ------------------------------------------------------------------ */
/* [P1 s7] names a "bias-mask" op among the kernels kept in the final
 * combination and s6 rejects fusing it with softmax; neither gives its
 * arithmetic.  The reading here is the shifted-window transformer's
 * general one (Swin): before softmax the attention logits of every window
 * and head get a position bias and, for shifted blocks, a mask that keeps
 * tokens from attending across a seam that the cyclic roll created.
 *
 * Region labels.  Along axis k a windowed row's cell c (its coordinate in
 * the rolled, padded grid) holds the token rolled in from coordinate
 * c + s_k of the period (the grid, or the padded grid for pad-then-shift);
 * when the roll moves that axis (s_k mod period_k != 0) the cell lies past
 * the seam if c + s_k >= period_k.  The label of a
 * row is the sum over the masked axes (bit k of axes_mask) of
 * 2^k * [past the seam along k].  Pad cells are labelled by the same rule.
 * Labels come out in the window-major destination order of
 * orc_build_window_index; like that builder this one scatters from every
 * padded cell to its destination row. */
int orc_build_shift_regions(const int32_t grid[3], const int32_t win[3], const int32_t shift[3],
                            const int32_t *padded, int32_t flags, int32_t axes_mask,
                            int32_t *out)
{
    int64_t P[3];
    if (resolve_padded(grid, win, padded, P) != 0) return -1;
    if (flags != 0 && flags != 1) return -1;
    int64_t period[3], s[3], nwin[3];
    for (int k = 0; k < 3; ++k) {
        period[k] = flags == 1 ? P[k] : (int64_t)grid[k];
        s[k] = pos_mod(shift[k], period[k]);
        nwin[k] = ceil_div64(P[k], win[k]);
    }
    /* rows before each window: the same window-major order as the index map */
    int64_t n_windows = nwin[0] * nwin[1] * nwin[2];
    int64_t *start = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_windows + 1));
    if (!start) return -2;
    start[0] = 0;
    for (int64_t w_id = 0; w_id < n_windows; ++w_id) {
        int64_t bz = w_id / (nwin[1] * nwin[2]), bh = (w_id / nwin[2]) % nwin[1], bw = w_id % nwin[2];
        int64_t e[3] = {P[0] - bz * win[0], P[1] - bh * win[1], P[2] - bw * win[2]};
        for (int k = 0; k < 3; ++k) if (e[k] > win[k]) e[k] = win[k];
        start[w_id + 1] = start[w_id] + e[0] * e[1] * e[2];
    }
    for (int64_t z = 0; z < P[0]; ++z)
        for (int64_t h = 0; h < P[1]; ++h)
            for (int64_t w = 0; w < P[2]; ++w) {
                const int64_t c[3] = {z, h, w};
                int64_t b[3], e[3], i[3];
                for (int k = 0; k < 3; ++k) {
                    b[k] = c[k] / win[k];
                    i[k] = c[k] % win[k];
                    e[k] = P[k] - b[k] * win[k];
                    if (e[k] > win[k]) e[k] = win[k];
                }
                int64_t w_id = (b[0] * nwin[1] + b[1]) * nwin[2] + b[2];
                int64_t dst = start[w_id] + (i[0] * e[1] + i[1]) * e[2] + i[2];
                int32_t label = 0;
                for (int k = 0; k < 3; ++k)
                    if (((axes_mask >> k) & 1) && s[k] != 0)
                        label += (c[k] + s[k] >= period[k]) << k;
                out[dst] = label;
            }
    free(start);
    return 0;
}

/* out[w,h,i,j] = round(round(scores[w,h,i,j] + bias[type(w),h,i,j]) + m)
 * with m = 0 when rows i and j of window w carry the same region label and
 * m = round(mask_value) otherwise; without labels (region == NULL, an
 * unshifted block) out = round(scores + bias).  Two rounding points, as an
 * eager "attn + bias; attn + mask" sequence in the tensor's format makes
 * them; the mask is added to every element, zeros included (so -0 + 0
 * gives +0).  scores/out [n_win, heads, n, n], bias [n_types, heads, n, n],
 * win_type [n_win] (NULL: type 0), region [n_win * n]; fmt 0 = binary16,
 * 1 = bfloat16. */
void orc_window_bias_mask_add_fmt(const uint16_t *scores, const uint16_t *bias,
                                  const int32_t *win_type, const int32_t *region, uint16_t *out,
                                  int64_t n_win, int32_t heads, int32_t n, double mask_value,
                                  int fmt)
{
    const double m = dec16(enc16(mask_value, fmt), fmt);
    for (int64_t w = 0; w < n_win; ++w) {
        const int64_t type = win_type ? win_type[w] : 0;
        for (int32_t h = 0; h < heads; ++h)
            for (int32_t i = 0; i < n; ++i)
                for (int32_t j = 0; j < n; ++j) {
                    const int64_t k = ((w * heads + h) * (int64_t)n + i) * n + j;
                    const int64_t kb = ((type * heads + h) * (int64_t)n + i) * n + j;
                    double t = dec16(enc16(dec16(scores[k], fmt) + dec16(bias[kb], fmt), fmt), fmt);
                    if (region) {
                        const int same = region[w * n + i] == region[w * n + j];
                        t = dec16(enc16(t + (same ? 0.0 : m), fmt), fmt);
                    }
                    out[k] = enc16(t, fmt);
                }
    }
}
