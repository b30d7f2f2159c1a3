/*
 * wgs.h -- C ABI of the GB300 (sm_103a) block-glue kernels of a
 * shifted-window (Swin / Pangu-Weather style) transformer block.
 *
 * Sources (page title, section):
 *   [P1] "BW1000 gfx936 Pangu-Weather inference profiling"
 *        (l189.com news 2144533)
 *        s1  the profile: LayerNorm, index_select (two per block), GELU
 *        s3  fixed-width LayerNorm, affine folded into the next Linear
 *        s4  fused residual add + norm, keeping the FP16 rounding point
 *        s5  window gather with a precomputed INT32 index protocol, and the
 *            fused norm-then-gather
 *        s6, s7  the ops kept in the final combination (bias-mask, restore
 *            path) and the fusions rejected
 *   [P3] "PyTorch + HIP fused bias + GELU on Hygon DCU"
 *        (forum.sourcefind.cn)
 *        s3  math semantics: tanh-approximate GELU of input + bias (backward
 *            left out there; added here)
 *        s6  interface checks: clear errors for bad inputs, empty input
 *            launches nothing, work goes on the caller's stream, launch
 *            status is checked
 *        s10, s12  other dtypes as hardening (bfloat16 here)
 *
 * Conventions shared by every device entry point
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     row-major and dense (row r starts at r * width elements).
 *   - The caller owns every buffer.  The library allocates no device
 *     memory, never synchronises the stream and never touches the default
 *     stream unless the caller passes it (stream 0).
 *   - Work is enqueued on `stream`; the call returns once it is enqueued.
 *     Kernels are launched with programmatic dependent launch: one may be
 *     scheduled while the previous kernel on the stream drains, and before
 *     waiting for it may ask L2 to fetch the lines of its first input rows
 *     (an index-driven kernel also reads its first index entries, L2 only,
 *     to steer those fetches).  No value read before the previous kernel
 *     has completed reaches a result: indices and rows are read again after
 *     the wait, so the usual stream order holds for every buffer.
 *   - Arguments are checked before anything is launched; a failed check
 *     returns a status and launches nothing.  A launch failure reported by
 *     the runtime returns WGS_ERR_LAUNCH.
 *   - A call with zero rows (or zero indices) returns WGS_OK and launches
 *     nothing; its pointers may then be NULL.
 *   - fp16 is IEEE binary16; "fp16(v)" below is round-to-nearest-even.
 *   - The kernels run only on compute capability 10.3 (sm_103a); on any
 *     other device the entry points return WGS_ERR_ARCH.
 *   - Calls are thread-safe; the shared state is the per-device index
 *     error words read by wgs_check_error() (and the scratch array of
 *     bias_gelu_tanh_bwd_noalloc).  Kernels name the error words
 *     directly, so no device address is kept between calls.
 *   - The first call of an entry point on a device (per dtype) caches what it
 *     needs from the runtime (SM count, resident CTAs per SM); make those
 *     calls outside stream capture.  Other calls, captured or not, make no
 *     such query.  Both depend on the device only, not on its context.  The
 *     16-bit GELU backward also raises its first pass's shared-memory limit,
 *     which belongs to the context: the first call on a device does it, and
 *     in a later context (after cudaDeviceReset, say) the first launch there
 *     is rejected by the runtime, the limit raised and the launch retried;
 *     make that call outside stream capture too.
 */
#ifndef WGS_H
#define WGS_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 1: the LayerNorm family, gathers and bias + GELU in fp16 / fp32.
 * 2: adds the bfloat16 forms, the GELU backward (with and without a
 *    workspace), the attention bias-mask add and the region-label builder;
 *    the backward's workspace query covers zero rows. */
#define WGS_ABI_VERSION 2

typedef enum {
    WGS_OK = 0,
    WGS_ERR_NULL = 1,    /* a required pointer is NULL                      */
    WGS_ERR_SHAPE = 2,   /* negative size, or sizes inconsistent            */
    WGS_ERR_WIDTH = 3,   /* width not supported by this entry point         */
    WGS_ERR_ALIGN = 4,   /* a pointer is not aligned as required            */
    WGS_ERR_DTYPE = 5,   /* unknown dtype code                              */
    WGS_ERR_ARCH = 6,    /* current device is not compute capability 10.3   */
    WGS_ERR_LAUNCH = 7,  /* the CUDA runtime rejected the launch            */
    WGS_ERR_INDEX = 8,   /* a gather index was outside [-1, n_src)          */
    WGS_ERR_ALIAS = 9,   /* buffers overlap in a way the operation forbids  */
    WGS_ERR_CUDA = 10,   /* another CUDA runtime call failed                */
    WGS_ERR_TOO_LARGE = 11 /* larger than the library's fixed scratch       */
} wgs_status;

typedef enum { WGS_F32 = 0, WGS_F16 = 1, WGS_BF16 = 2 } wgs_dtype;

/* Index-map construction order (wgs_build_window_index). */
#define WGS_SHIFT_THEN_PAD 0
#define WGS_PAD_THEN_SHIFT 1

/* Human-readable name of a status; never NULL. */
const char *wgs_status_string(wgs_status s);

/* WGS_ABI_VERSION of the built library. */
int32_t wgs_abi_version(void);

/* ------------------------------------------------------------------ */
/* ln_fwd -- LayerNorm without affine                          [P1 s3] */
/* ------------------------------------------------------------------ */
/* For each of `rows` rows of `width` fp16 values:
 *     mean = sum(x) / width,  var = sum((x - mean)^2) / width   (FP32)
 *     y    = fp16((x - mean) / sqrt(var + eps))
 * The affine scale and shift are not applied: the model folds them into
 * the following Linear at load time.
 *   x, y   fp16 [rows, width], 16-byte aligned.  y == x (in place) is
 *          allowed; any other overlap returns WGS_ERR_ALIAS.
 *   width  192 or 384 only (else WGS_ERR_WIDTH): the model's two hidden
 *          widths; there is no generic fallback.
 *   eps    added to the variance inside the square root (1e-5 in the model). */
wgs_status ln_fwd(const void *x, void *y, int64_t rows, int32_t width, float eps,
                  cudaStream_t stream);

/* ------------------------------------------------------------------ */
/* residual_add_ln_fwd -- fused residual add + LayerNorm       [P1 s4] */
/* ------------------------------------------------------------------ */
/*     residual_out = fp16(fp32(residual) + fp32(branch))   (written out)
 *     y            = LN(residual_out)                       (as ln_fwd)
 * The normalisation starts from the ROUNDED fp16 residual_out, the same
 * rounding point as a separate add followed by a separate LayerNorm.
 *   residual, branch, residual_out, y  fp16 [rows, width], 16-byte aligned.
 *   residual_out may equal residual or branch; y may equal residual or
 *   branch; residual_out and y must be distinct; partial overlaps return
 *   WGS_ERR_ALIAS.
 *   width  192 or 384 only. */
wgs_status residual_add_ln_fwd(const void *residual, const void *branch, void *residual_out,
                               void *y, int64_t rows, int32_t width, float eps,
                               cudaStream_t stream);

/* ------------------------------------------------------------------ */
/* window_gather -- shifted-window token gather               [P1 s5] */
/* ------------------------------------------------------------------ */
/* For d in [0, n_idx):
 *     dst[d] = src[idx[d]]   if 0 <= idx[d] < n_src   (bit-exact row copy)
 *     dst[d] = 0             if idx[d] == -1           (all-zero pad row)
 * so padding needs no zero-filled tensor.  An index outside [-1, n_src) is
 * a caller error: its row is written as zeros and the device error word is
 * set (see wgs_check_error); nothing faults.
 *   src  fp16 [n_src, width], dst fp16 [n_idx, width], both 16-byte
 *        aligned; they must not overlap (WGS_ERR_ALIAS).
 *   idx  int32 [n_idx], 4-byte aligned, device memory.  Usually built once
 *        per window shape with wgs_build_window_index and copied to the
 *        device.
 *   width  any multiple of 8 (rows are whole 16-byte chunks); 192 and 384
 *          take a specialised path. */
wgs_status window_gather(const void *src, const int32_t *idx, void *dst, int64_t n_src,
                         int64_t n_idx, int32_t width, cudaStream_t stream);

/* ------------------------------------------------------------------ */
/* norm_gather -- fused LayerNorm then window gather          [P1 s5] */
/* ------------------------------------------------------------------ */
/*     dst[d] = LN(src[idx[d]])  for a valid index, 0 for idx[d] == -1
 * The normalised tensor is never materialised: each gathered row is
 * normalised in registers on its way to dst.  Results equal ln_fwd
 * followed by window_gather bit for bit.  Buffers, index rules and errors
 * as window_gather; width 192 or 384 only. */
wgs_status norm_gather(const void *src, const int32_t *idx, void *dst, int64_t n_src,
                       int64_t n_idx, int32_t width, float eps, cudaStream_t stream);

/* ------------------------------------------------------------------ */
/* window_reverse_add_ln_fwd -- window reverse + residual add + LN     */
/*                                          [P1 s5 inverse, s4, s7]    */
/* ------------------------------------------------------------------ */
/* After window attention the windowed rows return to token order (the
 * inverse of window_gather: crop pads, undo the window order and the
 * cyclic shift), join the residual stream and feed norm2, in one pass.
 * P1 s7 keeps such a "restore path" op; s4 fixes the rounding point:
 *     residual_out[t] = fp16(fp32(residual[t]) + fp32(windows[inv_idx[t]]))
 *     y[t]            = LN(residual_out[t])                   (as ln_fwd)
 *   residual, residual_out, y  fp16 [rows, width], 16-byte aligned;
 *          residual_out and y may each equal residual, must differ from
 *          each other; other overlaps return WGS_ERR_ALIAS.
 *   windows  fp16 [n_windowed, width], 16-byte aligned, read at the rows
 *          inv_idx names; must not overlap the outputs.
 *   inv_idx  int32 [rows]: the windowed row of each token, usually from
 *          wgs_build_window_inverse.  A value outside [0, n_windowed) sets
 *          the device error word and that token takes no branch
 *          (residual_out = residual, bit for bit).
 *   width  192 or 384 only. */
wgs_status window_reverse_add_ln_fwd(const void *residual, const void *windows,
                                     const int32_t *inv_idx, void *residual_out, void *y,
                                     int64_t rows, int64_t n_windowed, int32_t width, float eps,
                                     cudaStream_t stream);

/* ------------------------------------------------------------------ */
/* residual_add_norm_gather -- residual add + norm1 + window gather    */
/*                                                  [P1 s4, s5]        */
/* ------------------------------------------------------------------ */
/* At a block boundary the residual stream is updated and written out (s4)
 * and the next block's norm1 output is consumed only by its window gather
 * (s5); one pass does all three:
 *     residual_out[s] = fp16(fp32(residual[s]) + fp32(branch[s]))
 *     dst[d]          = LN(residual_out[idx[d]])   (zero row for -1)
 * Equal, bit for bit, to residual_add_ln_fwd followed by window_gather of
 * its y.  Each source row s is processed by the destination row that names
 * it: rows of residual_out that idx never names are NOT written (a map from
 * wgs_build_window_index names every token exactly once).
 *   residual, branch, residual_out  fp16 [n_src, width], 16-byte aligned;
 *          residual_out may equal residual or branch (in place is exact
 *          only when idx names each row at most once).
 *   dst    fp16 [n_idx, width], must not overlap anything else.
 *   idx    int32 [n_idx], as for window_gather (bad values: zero row and
 *          the device error word).
 *   width  192 or 384 only. */
wgs_status residual_add_norm_gather(const void *residual, const void *branch, const int32_t *idx,
                                    void *residual_out, void *dst, int64_t n_src, int64_t n_idx,
                                    int32_t width, float eps, cudaStream_t stream);

/* ------------------------------------------------------------------ */
/* bfloat16 forms of the LayerNorm family                               */
/*      [P3 s3 and s12 list BF16 among the formats a hardened op covers] */
/* ------------------------------------------------------------------ */
/* Same arguments, rules and errors as the fp16 entry points above, with
 * every 16-bit tensor in bfloat16: elements widen exactly to FP32, the
 * statistics are FP32, and results round to nearest-even bfloat16.  The
 * residual sum is round_bf16(fp32 a + fp32 b), which equals rounding the
 * exact sum once (binary32 has at least 2 * 8 + 2 significand bits).
 * window_gather copies rows bit for bit and serves both formats. */
wgs_status ln_fwd_bf16(const void *x, void *y, int64_t rows, int32_t width, float eps,
                       cudaStream_t stream);
wgs_status residual_add_ln_fwd_bf16(const void *residual, const void *branch, void *residual_out,
                                    void *y, int64_t rows, int32_t width, float eps,
                                    cudaStream_t stream);
wgs_status norm_gather_bf16(const void *src, const int32_t *idx, void *dst, int64_t n_src,
                            int64_t n_idx, int32_t width, float eps, cudaStream_t stream);
wgs_status window_reverse_add_ln_fwd_bf16(const void *residual, const void *windows,
                                          const int32_t *inv_idx, void *residual_out, void *y,
                                          int64_t rows, int64_t n_windowed, int32_t width,
                                          float eps, cudaStream_t stream);
wgs_status residual_add_norm_gather_bf16(const void *residual, const void *branch,
                                         const int32_t *idx, void *residual_out, void *dst,
                                         int64_t n_src, int64_t n_idx, int32_t width, float eps,
                                         cudaStream_t stream);

/* ------------------------------------------------------------------ */
/* bias_gelu_tanh -- fused bias + tanh-approximate GELU       [P3 s3] */
/* ------------------------------------------------------------------ */
/*     t = x + bias[col]   (rounded once to the tensor dtype)
 *     y = 0.5 t (1 + tanh(sqrt(2/pi) (t + 0.044715 t^3)))
 * evaluated in FP32 and rounded to the tensor dtype.
 *   x, y   [rows, width] of `dtype` (WGS_F32, WGS_F16 or WGS_BF16); y == x allowed,
 *          other overlaps return WGS_ERR_ALIAS.
 *   bias   [width] of `dtype`; must not overlap y.
 *   width  any value >= 1.  A 16-byte vector path runs when width is a
 *          multiple of 4 (f32) or 8 (16-bit types) and all pointers are 16-byte
 *          aligned; otherwise a scalar path runs (same results). */
wgs_status bias_gelu_tanh(const void *x, const void *bias, void *y, int64_t rows, int32_t width,
                          wgs_dtype dtype, cudaStream_t stream);

/* ------------------------------------------------------------------ */
/* bias_gelu_tanh_bwd -- backward of bias + tanh-GELU                   */
/*          [P3 s3: the tutorial op leaves backward out; this adds it]  */
/* ------------------------------------------------------------------ */
/* Gradient of y = gelu_tanh(x + bias) with an eager backward's rounding
 * points:
 *     t         = round(x + bias[c])                         (as forward)
 *     grad_x    = round(grad_y * gelu'(t))   (gelu' evaluated in FP32)
 *     grad_bias = round(sum over rows of grad_x[., c])       (FP32 sum)
 * The column sum is deterministic: per-slab FP32 partial sums go to
 * `workspace`, then one pass adds them in a fixed order; the summation
 * order depends only on rows, width and dtype, so results do not depend on
 * the device.
 *   grad_y, x, grad_x  [rows, width] of `dtype`; grad_x may equal grad_y,
 *          other overlaps return WGS_ERR_ALIAS.
 *   bias, grad_bias    [width] of `dtype`, disjoint from everything else.
 *   workspace  device memory of at least
 *          wgs_bias_gelu_bwd_workspace_bytes(rows, width) bytes (one slab of
 *          width floats when rows == 0), 16-byte aligned, owned by the
 *          caller, disjoint from the tensors; its contents on entry do not
 *          matter.
 *   rows == 0 writes grad_bias = 0 (two small launches); width == 0 returns
 *   WGS_OK and launches nothing.  The 16-byte vector path needs width a
 *   multiple of 4 (f32) or 8 (16-bit types) and aligned tensors; otherwise
 *   a scalar path runs (same results). */
size_t wgs_bias_gelu_bwd_workspace_bytes(int64_t rows, int32_t width);
wgs_status bias_gelu_tanh_bwd(const void *grad_y, const void *x, const void *bias, void *grad_x,
                              void *grad_bias, void *workspace, size_t workspace_bytes,
                              int64_t rows, int32_t width, wgs_dtype dtype, cudaStream_t stream);

/* bias_gelu_tanh_bwd_noalloc -- the same backward without a workspace.
 * The reference pages have no counterpart; it exists for callers that
 * cannot give this library device memory: an op inside a host runtime that
 * owns every allocation and passes its plugins no allocator or workspace,
 * or a hot path that must not call cudaMalloc because that call can
 * synchronise the device.  The partial column sums then live in one array
 * of 1,310,720 floats (5 MiB) built into the library, which every GPU that
 * loads the library keeps until the process exits.
 *   Arguments, results and errors as bias_gelu_tanh_bwd, without
 *   `workspace`.  Sizes whose partial sums would not fit (more than
 *   1,310,720 floats: min(608, ceil(rows / 216)) slabs x width, so any row
 *   count up to width 2048) return WGS_ERR_TOO_LARGE and launch nothing.
 *   Allocates nothing.  Every call looks up the array's device address in
 *   the calling thread's current context (cudaGetSymbolAddress, a host-side
 *   lookup), so a device reset or a second context on the device is safe.
 *   The first call in a context also loads the library's device code there:
 *   make that first call before any stream capture.
 *   All calls on a device share the array, which keeps whatever the last
 *   call left there; nothing in it needs to start at zero, because every
 *   partial sum is written before it is read.  Calls whose work overlaps on
 *   the GPU (other streams, other host threads) race on the array: run one
 *   at a time per device. */
wgs_status bias_gelu_tanh_bwd_noalloc(const void *grad_y, const void *x, const void *bias,
                                      void *grad_x, void *grad_bias, int64_t rows, int32_t width,
                                      wgs_dtype dtype, cudaStream_t stream);

/* ------------------------------------------------------------------ */
/* window_bias_mask_add -- position bias + shift mask before softmax    */
/*                                                          [P1 s6, s7] */
/* ------------------------------------------------------------------ */
/* P1 s7 keeps a "bias-mask" op in the final combination and s6 rejects
 * fusing it with softmax; the pages give no arithmetic.  This library's
 * reading is the shifted-window transformer's general one: the attention
 * logits of every window and head receive a position bias and, in shifted
 * blocks, a mask between rows that the cyclic roll brought together:
 *     t[w,h,i,j]   = fp(scores[w,h,i,j] + bias[type[w],h,i,j])
 *     out[w,h,i,j] = fp(t + (region[w*n+i] == region[w*n+j] ? 0 : m))
 * where fp() rounds to nearest-even in `dtype` and m = fp(mask_value); the
 * mask term is added to every element (so -0 becomes +0 where it is 0).
 * With region == NULL (an unshifted block) out = t.
 *   scores, out  [n_win, heads, n, n] of dtype (WGS_F16 or WGS_BF16);
 *                out may equal scores, other overlaps return WGS_ERR_ALIAS.
 *   bias         [n_types, heads, n, n] of dtype: the position bias already
 *                expanded from its table, one slab per window type.
 *   win_type     int32 [n_win] in [0, n_types), or NULL for type 0 (then
 *                n_types may be 1).  A type outside the range writes that
 *                window's outputs as zeros and sets the device error word
 *                (wgs_check_error); nothing faults.
 *   region       int32 [n_win * n] labels (wgs_build_shift_regions), or NULL.
 * n_win * heads * n must be below 2^31 (else WGS_ERR_SHAPE).  The 16-byte
 * path needs n a multiple of 8 (n <= 2048), scores / bias / out 16-byte
 * aligned and region 16-byte aligned; otherwise a scalar path runs (same
 * results). */
wgs_status window_bias_mask_add(const void *scores, const void *bias, const int32_t *win_type,
                                const int32_t *region, void *out, int64_t n_win, int32_t heads,
                                int32_t n, int32_t n_types, float mask_value, wgs_dtype dtype,
                                cudaStream_t stream);

/* ------------------------------------------------------------------ */
/* Host-side window index map                                 [P1 s5] */
/* ------------------------------------------------------------------ */
/* The page fixes the protocol (INT32 per destination row, >= 0 source
 * token, -1 zero row, precomputed once per window shape); the
 * construction below is this library's reading of it:
 *   - tokens are the row-major flattening of a grid[0] x grid[1] x grid[2]
 *     (Z, H, W) grid;
 *   - the padded grid has extents padded[k] >= grid[k]; padded == NULL
 *     rounds each extent up to a multiple of window[k];
 *   - windows tile the padded grid from the origin, the last one on an axis
 *     cut short when the padded extent is not a window multiple;
 *   - destination rows run window by window (row-major over the window
 *     grid), then row-major over the cells of each window;
 *   - WGS_SHIFT_THEN_PAD: a cell (z,h,w) inside the grid reads token
 *     ((z+s0) mod Z, (h+s1) mod H, (w+s2) mod W) -- a cyclic roll by
 *     -shift -- and every other cell is -1;
 *     WGS_PAD_THEN_SHIFT: the roll runs over the padded grid, and a rolled
 *     position outside the grid is -1.
 * A block feeds one map to its gather, its attention (window_bias_mask_add)
 * and its window reverse, and a batched attention needs equal windows: pass
 * padded extents that are window multiples (padded == NULL does this), e.g.
 * 4 x 96 x 96 for the 4 x 91 x 90 grid at window (2, 6, 12).  A map with a
 * cut last window (4 x 96 x 90 there) is valid for the gathers alone.
 * Host memory only; no CUDA call is made. */

/* Number of destination rows (product of the padded extents), or -1 for
 * invalid extents: grid or window < 1, padded < grid, a rounded-up extent
 * above INT32_MAX, or a product (of the padded extents or of the grid)
 * that does not fit in int64.  The builders below return WGS_ERR_SHAPE for
 * the same extents. */
int64_t wgs_window_index_count(const int32_t grid[3], const int32_t window[3],
                               const int32_t *padded);

/* Fill out_host[0 .. count) with the map.  out_len must be at least the
 * count (else WGS_ERR_SHAPE); the token count must fit in int32. */
wgs_status wgs_build_window_index(const int32_t grid[3], const int32_t window[3],
                                  const int32_t shift[3], const int32_t *padded, int32_t flags,
                                  int32_t *out_host, int64_t out_len);

/* Fill inv_host[0 .. grid[0]*grid[1]*grid[2]) with the inverse map: the
 * windowed row that holds each token (same arguments as
 * wgs_build_window_index; out_len must be at least the token count, else
 * WGS_ERR_SHAPE).  Host memory only; no CUDA call is made. */
wgs_status wgs_build_window_inverse(const int32_t grid[3], const int32_t window[3],
                                    const int32_t shift[3], const int32_t *padded, int32_t flags,
                                    int32_t *inv_host, int64_t out_len);

/* Fill out_host[0 .. count) with the shift-mask region label of every
 * windowed row, in the map's destination order (same arguments as
 * wgs_build_window_index, plus axes_mask).  Along axis k (bit k of
 * axes_mask set) a row's cell c holds the token rolled in from c + s_k of
 * the roll's period (the grid for WGS_SHIFT_THEN_PAD, the padded grid for
 * WGS_PAD_THEN_SHIFT, s_k the shift taken modulo that period); when s_k is
 * not 0 the cell lies past the roll's seam if c + s_k >= period_k.  The
 * label is the sum over masked axes of 2^k * [past the seam along k]; pad
 * cells follow the same rule.  Two rows of a window share a label exactly
 * when the roll put no seam between them along a masked axis, the regions
 * of the classic shifted-window attention mask.  axes_mask = 7 masks every
 * axis; a periodic axis (longitude) can be left out.  Host memory only;
 * out_len must be at least the count, else WGS_ERR_SHAPE. */
wgs_status wgs_build_shift_regions(const int32_t grid[3], const int32_t window[3],
                                   const int32_t shift[3], const int32_t *padded, int32_t flags,
                                   int32_t axes_mask, int32_t *out_host, int64_t out_len);

/* Read and clear the current device's index error words after the work
 * already queued on `stream` has finished.  This call synchronises
 * `stream`.  Returns WGS_ERR_INDEX if any gather since the last check met
 * an index outside [-1, n_src), any window reverse an inverse index outside
 * [0, n_windowed), or any window_bias_mask_add a window type outside
 * [0, n_types); WGS_OK otherwise.  The words are shared by every stream of
 * the device. */
wgs_status wgs_check_error(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* WGS_H */
