// Row kernels of the block glue: no-affine LayerNorm, fused residual add +
// LayerNorm, shifted-window gather, fused norm-then-gather, and the two
// block-boundary fusions (window reverse + residual add + LayerNorm;
// residual add + LayerNorm + window gather), for fp16 and bfloat16 rows
// (sm_103a).
//
// Page "BW1000 gfx936 Pangu-Weather inference profiling":
//   s3  fixed-width (192 / 384) LayerNorm, FP16 in and out, FP32 statistics
//   s4  residual add + norm that keeps the FP16 rounding point
//   s5  INT32-indexed window gather (-1 = zero row) and the fused
//       norm-gather that never writes the normalised tensor
//   s1, s7  the restore path after attention (window reverse)
//
// Design (GB300): all are HBM-bound row streams, so there are no tensor
// cores here.  A row of W 16-bit values is W/8 16-byte chunks; LPR lanes share
// a row (8 lanes at W = 192, 16 at W = 384), each holding CPL = 3 chunks in
// registers, so one warp-wide load instruction moves whole 128-byte lines.
// The row never leaves registers between load, FP32 butterfly reductions and
// store; the statistics use the shifted-data two-pass method (see
// ln_normalize).  Each warp works on U row groups at once, so every lane has
// U * CPL independent 16-byte loads in flight before its first reduction.
// U = 1 measured best: with 40 warps resident per SM there is enough memory
// parallelism, and the smaller CTAs fill the last partial wave better.
#include <atomic>
#include <type_traits>

#include "wgs_common.cuh"

#ifndef WGS_ROW_WARPS
#define WGS_ROW_WARPS 4      // warps per CTA
#endif
#ifndef WGS_ROW_U
#define WGS_ROW_U 1          // row groups per warp per iteration
#endif
#ifndef WGS_ROW_EARLY
#define WGS_ROW_EARLY 1      // L2 prefetch of the first rows before the wait on the previous grid
#endif
#ifndef WGS_ROW_CTAS_PER_SM
#define WGS_ROW_CTAS_PER_SM 64  // grid cap, in CTAs per SM (grid-stride beyond it)
#endif

namespace wgs {

// Set (never cleared by a kernel) when a gather meets an index outside
// [-1, n_src), or the window reverse an inverse index outside
// [0, n_windowed); read and cleared by wgs_check_error().
__device__ unsigned int g_index_error;

// kLN            y[r] = LN(x[r])
// kAddLN         o[r] = fp16(a[r] + b[r]),         y[r] = LN(o[r])
// kGather        y[r] = x[idx[r]]                  (zero row for a pad)
// kNormGather    y[r] = LN(x[idx[r]])              (zero row for a pad)
// kRevAddLN      o[r] = fp16(a[r] + w[inv[r]]),    y[r] = LN(o[r])
// kAddNormGather o[s] = fp16(a[s] + b[s]),         y[r] = LN(o[s]),  s = idx[r]
enum class RowOp : int { kLN, kAddLN, kGather, kNormGather, kRevAddLN, kAddNormGather };

struct RowArgs {
    const uint16_t *in0;  // x / residual / src (16-bit elements)
    const uint16_t *in1;  // branch (add + LN, add + norm + gather), windows (reverse)
    uint16_t *out0;       // y (LN, gathers) or residual_out (the add ops)
    uint16_t *out1;       // y / dst of the add ops
    const int32_t *idx;   // window map (gathers) or its inverse (reverse)
    int64_t rows;         // rows of the launch: tokens, or windowed rows for the gathers
    int64_t n_src;        // bound of idx values: source rows, or windowed rows (reverse)
    float eps;
};

template <int WIDTH> struct RowTiling;
template <> struct RowTiling<192> { static constexpr int kLPR = 8; };
#ifndef WGS_LPR384
#define WGS_LPR384 16  // lanes sharing a 384-wide row
#endif
template <> struct RowTiling<384> { static constexpr int kLPR = WGS_LPR384; };

// No-affine LayerNorm of U rows per lane group, each row held as CPL chunks
// per lane over LPR lanes.  FP32 statistics by the shifted-data two-pass
// method (Chan, Golub & LeVeque, "Algorithms for computing the sample
// variance", 1983): with K the row's first element,
//     m = sum(x - K) / W,  d = (x - K) - m,  var = sum(d^2) / W,
//     y = fp16(d * (1 / sqrt(var + eps))).
// Mathematically d = x - mean.  Numerically, x - K is exact in FP32 when x
// and K lie within a factor of 2^12 of each other (fp16: two 11-bit
// significands fit FP32's 24 bits together; bf16 has 2^15 of room) and
// otherwise carries a single FP32 rounding, far below the output's fp16
// spacing; the summed terms stay at the scale of the row's spread instead
// of its offset, so the error of d no longer grows with |mean|.  Each element is
// converted to FP32 once and kept in registers; each lane sums its part
// with four accumulators (short dependency chains), then the LPR lanes of
// the row combine by butterfly.  The divisions by W are products with 1/W
// and 1/sqrt is the rsqrt instruction: each adds a relative error of a
// few 1e-7 at most, far below what an FP32 LayerNorm carries anyway, and
// saves the long correctly rounded divide / square-root sequences once per
// row.  Every LN kernel calls this one function, so equal inputs give
// equal bits.
template <typename E, int WIDTH, int LPR, int CPL, int U>
__device__ __forceinline__ void ln_normalize(uint4 (&v)[U][CPL], float eps) {
    constexpr int NE = CPL * 8;  // elements of one row held by this lane
    constexpr float kInvWidth = 1.0f / WIDTH;
    const int lead = (threadIdx.x & 31) & ~(LPR - 1);  // lane holding the row's first chunk
    float d[U][NE];
    float mean[U], rstd[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const float shift = __shfl_sync(0xffffffffu, E::to_f2(v[u][0].x).x, lead);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < CPL; ++c)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = E::to_f2(word(v[u][c], j));
                d[u][c * 8 + 2 * j] = f.x - shift;
                d[u][c * 8 + 2 * j + 1] = f.y - shift;
                acc[j] += d[u][c * 8 + 2 * j];
                acc[j] += d[u][c * 8 + 2 * j + 1];
            }
        mean[u] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) mean[u] = group_sum<LPR>(mean[u]) * kInvWidth;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            d[u][e] -= mean[u];
            acc[e & 3] = fmaf(d[u][e], d[u][e], acc[e & 3]);
        }
        rstd[u] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const float var = group_sum<LPR>(rstd[u]) * kInvWidth;
        rstd[u] = rsqrtf(var + eps);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
        for (int c = 0; c < CPL; ++c)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                set_word(v[u][c], j,
                         E::from_f2(d[u][c * 8 + 2 * j] * rstd[u], d[u][c * 8 + 2 * j + 1] * rstd[u]));
}

// residual_out = round(residual + branch) on one 16-byte chunk.
template <typename E>
__device__ __forceinline__ uint4 add_chunk(const uint4 &a, const uint4 &b) {
    uint4 r;
#pragma unroll
    for (int j = 0; j < 4; ++j) set_word(r, j, E::add2(word(a, j), word(b, j)));
    return r;
}

// WGS_ROW_MIN_BLOCKS, when defined: resident CTAs per SM the register
// allocation must allow (otherwise ptxas chooses)
#ifdef WGS_ROW_MIN_BLOCKS
#define WGS_ROW_BOUNDS(T) __launch_bounds__(T, WGS_ROW_MIN_BLOCKS)
#else
#define WGS_ROW_BOUNDS(T) __launch_bounds__(T)
#endif

// Launch shape per op and width.  Most row ops run many short CTAs (the grid
// capped at WGS_ROW_CTAS_PER_SM per SM, so each SM is refilled as CTAs
// finish) and prefetch their first iteration's rows before the wait.
// Norm-gather at width 384 runs one resident wave instead, each CTA
// prefetching the rows of up to 4 grid-stride iterations: measured on GB300
// 8.6 -> 8.3 us at [32760,384] -> 34560 rows and 9.1 -> 8.6 us -> 36864
// rows, while the same shape slowed every other row op by 2-20 %.
// Row groups per warp: one, except bfloat16 norm-gather at width 192, where
// two measured 16.5 -> 16.1 us at 138240 rows (every other op was 1-7 %
// slower with two).
template <RowOp OP, typename E, int WIDTH> struct RowLaunch {
    static constexpr bool kOneWave = OP == RowOp::kNormGather && WIDTH == 384;
    static constexpr int kPrefetchIters = kOneWave ? 4 : 1;
    static constexpr int kRowGroups =
        OP == RowOp::kNormGather && WIDTH == 192 && std::is_same<E, Bf16>::value ? 2 : WGS_ROW_U;
};

template <RowOp OP, typename E, int WIDTH, int U, int WARPS, int PF>
__global__ void WGS_ROW_BOUNDS(WARPS * 32) row_kernel(const RowArgs a) {
#if !WGS_ROW_EARLY
    pdl_prologue();
#endif
    constexpr int LPR = RowTiling<WIDTH>::kLPR;
    constexpr int CPL = WIDTH / 8 / LPR;
    constexpr int RPW = 32 / LPR;                 // rows per warp per group
    constexpr int ROWS_CTA = WARPS * RPW * U;     // rows per CTA per iteration
    // index-driven rows: the launch's rows are windowed rows, read through idx
    constexpr bool kByIndex =
        OP == RowOp::kGather || OP == RowOp::kNormGather || OP == RowOp::kAddNormGather;
    constexpr bool kTwoInputs =
        OP == RowOp::kAddLN || OP == RowOp::kRevAddLN || OP == RowOp::kAddNormGather;
    constexpr bool kNorm = OP != RowOp::kGather;
    static_assert(LPR * CPL * 8 == WIDTH, "row tiling must cover the row");

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int grp = lane / LPR;
    const int sub = lane % LPR;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * ROWS_CTA;
    const int64_t base0 = static_cast<int64_t>(blockIdx.x) * ROWS_CTA;

#if WGS_ROW_EARLY
    // Before waiting for the previous grid, ask L2 for the lines the first
    // PF iterations will load.  The rows of direct ops are known; an
    // index-driven op reads its index first (L2 only) and prefetches the
    // rows it names.  Nothing read here feeds a result: the previous grid may
    // still be writing these buffers, so the index is read again after the
    // wait and every row is loaded after it.  Measured on GB300: the C = 384
    // gather 9.5 -> 8.1 us, its norm-gather 9.7 -> 8.6 us, every row op 2-10 %.
    auto prefetch_rows = [&](const int64_t base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t r = base + static_cast<int64_t>(warp * U + u) * RPW + grp;
            if (r >= a.rows) continue;
            if constexpr (kByIndex || OP == RowOp::kRevAddLN) {
                const int64_t s = ld_cg_i32(a.idx + r);
                if (s >= 0 && s < a.n_src) {
                    const uint16_t *p = kByIndex ? a.in0 : a.in1;
#pragma unroll
                    for (int k = 0; k < CPL; ++k) prefetch_l2(p + s * WIDTH + (sub + k * LPR) * 8);
                    if constexpr (OP == RowOp::kAddNormGather)
#pragma unroll
                        for (int k = 0; k < CPL; ++k)
                            prefetch_l2(a.in1 + s * WIDTH + (sub + k * LPR) * 8);
                }
            }
            if constexpr (!kByIndex) {
#pragma unroll
                for (int k = 0; k < CPL; ++k) prefetch_l2(a.in0 + r * WIDTH + (sub + k * LPR) * 8);
                if constexpr (OP == RowOp::kAddLN)
#pragma unroll
                    for (int k = 0; k < CPL; ++k)
                        prefetch_l2(a.in1 + r * WIDTH + (sub + k * LPR) * 8);
            }
        }
    };
    if constexpr (PF == 1) {
        prefetch_rows(base0);
    } else {
#pragma unroll
        for (int it = 0; it < PF; ++it) prefetch_rows(base0 + it * stride);
    }
    pdl_prologue();
#endif

    for (int64_t base = base0; base < a.rows; base += stride) {
        int64_t row[U], src[U], brow[U];
        bool live[U], valid[U], branch[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            row[u] = base + static_cast<int64_t>(warp * U + u) * RPW + grp;
            live[u] = row[u] < a.rows;
            src[u] = row[u];
            valid[u] = live[u];
            brow[u] = row[u];
            branch[u] = live[u];
        }
        if constexpr (kByIndex || OP == RowOp::kRevAddLN) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t s = live[u] ? __ldg(a.idx + row[u]) : -1;
                const bool ok = s >= 0 && s < a.n_src;
                // a pad (-1) is legal in a window map, never in its inverse
                const bool legal = ok || (kByIndex && s == -1);
                if (live[u] && !legal && sub == 0) atomicOr(&g_index_error, 1u);
                if constexpr (kByIndex) {
                    valid[u] = ok;
                    src[u] = ok ? s : 0;
                    brow[u] = src[u];
                    branch[u] = ok;
                } else {  // reverse: the residual row is always there, the branch row may not be
                    branch[u] = live[u] && ok;
                    brow[u] = ok ? s : 0;
                }
            }
        }

        uint4 v[U][CPL];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int k = 0; k < CPL; ++k)
                v[u][k] = valid[u] ? ld_stream(a.in0 + src[u] * WIDTH + (sub + k * LPR) * 8) : zero;

        if constexpr (kTwoInputs) {
            uint4 b[U][CPL];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int k = 0; k < CPL; ++k)
                    b[u][k] = branch[u] ? ld_stream(a.in1 + brow[u] * WIDTH + (sub + k * LPR) * 8)
                                        : zero;
            // residual_out = fp16(fp32 residual + fp32 branch); a missing
            // branch (bad inverse index) leaves the residual bits unchanged
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (branch[u])
#pragma unroll
                    for (int k = 0; k < CPL; ++k) v[u][k] = add_chunk<E>(v[u][k], b[u][k]);
            // the residual stream is written at its own (source) row
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (valid[u])
#pragma unroll
                    for (int k = 0; k < CPL; ++k)
                        st_stream(a.out0 + src[u] * WIDTH + (sub + k * LPR) * 8, v[u][k]);
        }

        if constexpr (kNorm) ln_normalize<E, WIDTH, LPR, CPL, U>(v, a.eps);

        uint16_t *out = kTwoInputs ? a.out1 : a.out0;
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (live[u])
#pragma unroll
                for (int k = 0; k < CPL; ++k)
                    st_stream(out + row[u] * WIDTH + (sub + k * LPR) * 8, valid[u] ? v[u][k] : zero);
    }
}

// Gather for any width that is a whole number of 16-byte chunks: one warp
// per destination row, lanes striding over the row's chunks.
__global__ void __launch_bounds__(256) gather_any_width_kernel(const uint4 *src, const int32_t *idx,
                                                                uint4 *dst, int64_t n_src,
                                                                int64_t n_idx, int32_t chunks) {
    pdl_prologue();
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t d = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         d < n_idx; d += warps) {
        const int32_t s = __ldg(idx + d);
        const bool valid = s >= 0 && s < n_src;
        if (!valid && s != -1 && lane == 0) atomicOr(&g_index_error, 1u);
        for (int c = lane; c < chunks; c += 32)
            dst[d * chunks + c] = valid ? ld_stream(src + static_cast<int64_t>(s) * chunks + c)
                                        : make_uint4(0u, 0u, 0u, 0u);
    }
}

template <RowOp OP, typename E, int WIDTH>
wgs_status launch_rows(const RowArgs &a, cudaStream_t stream) {
    DeviceInfo dev;
    const wgs_status st = current_device(&dev);
    if (st != WGS_OK) return st;
    using L = RowLaunch<OP, E, WIDTH>;
    constexpr int U = L::kRowGroups, WARPS = WGS_ROW_WARPS;
    constexpr int ROWS_CTA = WARPS * (32 / RowTiling<WIDTH>::kLPR) * U;
    const int64_t iters = ceil_div(a.rows, ROWS_CTA);
    auto kernel = row_kernel<OP, E, WIDTH, U, WARPS, L::kPrefetchIters>;
    int64_t cap = static_cast<int64_t>(dev.sm_count) * WGS_ROW_CTAS_PER_SM;
    if constexpr (L::kOneWave) {
        static std::atomic<int> resident[64];  // per device, for this instantiation
        int per_sm = resident[dev.device].load(std::memory_order_relaxed);
        if (per_sm == 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, WARPS * 32, 0) !=
                    cudaSuccess ||
                per_sm < 1)
                return WGS_ERR_LAUNCH;
            resident[dev.device].store(per_sm, std::memory_order_relaxed);
        }
        cap = static_cast<int64_t>(dev.sm_count) * per_sm;
    }
    const unsigned grid = static_cast<unsigned>(iters < cap ? iters : cap);
    return launch(kernel, dim3(grid), dim3(WARPS * 32), 0, stream, a);
}

template <RowOp OP, typename E = Fp16>
wgs_status dispatch_width(const RowArgs &a, int32_t width, cudaStream_t stream) {
    return width == 192 ? launch_rows<OP, E, 192>(a, stream) : launch_rows<OP, E, 384>(a, stream);
}

bool ln_width(int32_t width) { return width == 192 || width == 384; }

// rows * width 16-bit values must be addressable in bytes.
bool fits(int64_t rows, int32_t width) { return rows <= INT64_MAX / 2 / width; }

}  // namespace wgs

using namespace wgs;

template <typename E>
wgs_status ln_fwd_impl(const void *x, void *y, int64_t rows, int32_t width, float eps,
                             cudaStream_t stream) {
    if (!ln_width(width)) return WGS_ERR_WIDTH;
    if (rows < 0 || !fits(rows, width)) return WGS_ERR_SHAPE;
    if (rows == 0) return WGS_OK;
    if (!x || !y) return WGS_ERR_NULL;
    if (!aligned16(x) || !aligned16(y)) return WGS_ERR_ALIGN;
    const int64_t bytes = rows * width * 2;
    if (!same_or_disjoint(x, y, bytes)) return WGS_ERR_ALIAS;
    RowArgs a{static_cast<const uint16_t *>(x), nullptr, static_cast<uint16_t *>(y), nullptr,
              nullptr, rows, 0, eps};
    return dispatch_width<RowOp::kLN, E>(a, width, stream);
}

template <typename E>
wgs_status residual_add_ln_fwd_impl(const void *residual, const void *branch,
                                          void *residual_out, void *y, int64_t rows,
                                          int32_t width, float eps, cudaStream_t stream) {
    if (!ln_width(width)) return WGS_ERR_WIDTH;
    if (rows < 0 || !fits(rows, width)) return WGS_ERR_SHAPE;
    if (rows == 0) return WGS_OK;
    if (!residual || !branch || !residual_out || !y) return WGS_ERR_NULL;
    if (!aligned16(residual) || !aligned16(branch) || !aligned16(residual_out) || !aligned16(y))
        return WGS_ERR_ALIGN;
    const int64_t bytes = rows * width * 2;
    if (overlap(residual_out, bytes, y, bytes)) return WGS_ERR_ALIAS;
    if (!same_or_disjoint(residual_out, residual, bytes) ||
        !same_or_disjoint(residual_out, branch, bytes) || !same_or_disjoint(y, residual, bytes) ||
        !same_or_disjoint(y, branch, bytes))
        return WGS_ERR_ALIAS;
    RowArgs a{static_cast<const uint16_t *>(residual), static_cast<const uint16_t *>(branch),
              static_cast<uint16_t *>(residual_out), static_cast<uint16_t *>(y), nullptr, rows, 0, eps};
    return dispatch_width<RowOp::kAddLN, E>(a, width, stream);
}

namespace {

wgs_status check_gather(const void *src, const int32_t *idx, void *dst, int64_t n_src,
                        int64_t n_idx, int32_t width) {
    if (n_src < 0 || n_idx < 0 || !fits(n_src, width) || !fits(n_idx, width)) return WGS_ERR_SHAPE;
    if (n_idx == 0) return WGS_OK;
    if (!idx || !dst || (n_src > 0 && !src)) return WGS_ERR_NULL;
    if (!aligned16(dst) || (src && !aligned16(src)) || !aligned4(idx)) return WGS_ERR_ALIGN;
    const int64_t dst_bytes = n_idx * width * 2;
    if (overlap(src, n_src * width * 2, dst, dst_bytes) || overlap(idx, n_idx * 4, dst, dst_bytes))
        return WGS_ERR_ALIAS;
    return WGS_OK;
}

}  // namespace

extern "C" wgs_status window_gather(const void *src, const int32_t *idx, void *dst, int64_t n_src,
                                    int64_t n_idx, int32_t width, cudaStream_t stream) {
    if (width <= 0 || width % 8 != 0) return WGS_ERR_WIDTH;
    wgs_status st = check_gather(src, idx, dst, n_src, n_idx, width);
    if (st != WGS_OK || n_idx == 0) return st;
    RowArgs a{static_cast<const uint16_t *>(src), nullptr, static_cast<uint16_t *>(dst), nullptr, idx,
              n_idx, n_src, 0.f};
    if (ln_width(width)) return dispatch_width<RowOp::kGather>(a, width, stream);

    DeviceInfo dev;
    st = current_device(&dev);
    if (st != WGS_OK) return st;
    const int64_t warps_needed = n_idx;
    const int64_t blocks = ceil_div(warps_needed, 8);
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
    return launch(gather_any_width_kernel, dim3(static_cast<unsigned>(blocks < cap ? blocks : cap)),
                  dim3(256), 0, stream, static_cast<const uint4 *>(src), idx,
                  static_cast<uint4 *>(dst), n_src, n_idx, static_cast<int32_t>(width / 8));
}

template <typename E>
wgs_status norm_gather_impl(const void *src, const int32_t *idx, void *dst, int64_t n_src,
                                  int64_t n_idx, int32_t width, float eps, cudaStream_t stream) {
    if (!ln_width(width)) return WGS_ERR_WIDTH;
    const wgs_status st = check_gather(src, idx, dst, n_src, n_idx, width);
    if (st != WGS_OK || n_idx == 0) return st;
    RowArgs a{static_cast<const uint16_t *>(src), nullptr, static_cast<uint16_t *>(dst), nullptr, idx,
              n_idx, n_src, eps};
    return dispatch_width<RowOp::kNormGather, E>(a, width, stream);
}

template <typename E>
wgs_status window_reverse_add_ln_fwd_impl(const void *residual, const void *windows,
                                                const int32_t *inv_idx, void *residual_out,
                                                void *y, int64_t rows, int64_t n_windowed,
                                                int32_t width, float eps, cudaStream_t stream) {
    if (!ln_width(width)) return WGS_ERR_WIDTH;
    if (rows < 0 || n_windowed < 0 || !fits(rows, width) || !fits(n_windowed, width))
        return WGS_ERR_SHAPE;
    if (rows == 0) return WGS_OK;
    if (!residual || !inv_idx || !residual_out || !y || (n_windowed > 0 && !windows))
        return WGS_ERR_NULL;
    if (!aligned16(residual) || !aligned16(residual_out) || !aligned16(y) ||
        (windows && !aligned16(windows)) || !aligned4(inv_idx))
        return WGS_ERR_ALIGN;
    const int64_t bytes = rows * width * 2;
    const int64_t wbytes = n_windowed * width * 2;
    if (overlap(residual_out, bytes, y, bytes) || !same_or_disjoint(residual_out, residual, bytes) ||
        !same_or_disjoint(y, residual, bytes) || overlap(windows, wbytes, residual_out, bytes) ||
        overlap(windows, wbytes, y, bytes) || overlap(inv_idx, rows * 4, residual_out, bytes) ||
        overlap(inv_idx, rows * 4, y, bytes))
        return WGS_ERR_ALIAS;
    RowArgs a{static_cast<const uint16_t *>(residual), static_cast<const uint16_t *>(windows),
              static_cast<uint16_t *>(residual_out), static_cast<uint16_t *>(y), inv_idx, rows,
              n_windowed, eps};
    return dispatch_width<RowOp::kRevAddLN, E>(a, width, stream);
}

template <typename E>
wgs_status residual_add_norm_gather_impl(const void *residual, const void *branch,
                                               const int32_t *idx, void *residual_out, void *dst,
                                               int64_t n_src, int64_t n_idx, int32_t width,
                                               float eps, cudaStream_t stream) {
    if (!ln_width(width)) return WGS_ERR_WIDTH;
    if (n_src < 0 || n_idx < 0 || !fits(n_src, width) || !fits(n_idx, width)) return WGS_ERR_SHAPE;
    if (n_idx == 0) return WGS_OK;
    if (!idx || !dst || (n_src > 0 && (!residual || !branch || !residual_out))) return WGS_ERR_NULL;
    if (!aligned16(dst) || !aligned4(idx) ||
        (n_src > 0 && (!aligned16(residual) || !aligned16(branch) || !aligned16(residual_out))))
        return WGS_ERR_ALIGN;
    const int64_t bytes = n_src * width * 2;
    const int64_t dbytes = n_idx * width * 2;
    if (!same_or_disjoint(residual_out, residual, bytes) ||
        !same_or_disjoint(residual_out, branch, bytes) || overlap(dst, dbytes, residual, bytes) ||
        overlap(dst, dbytes, branch, bytes) || overlap(dst, dbytes, residual_out, bytes) ||
        overlap(idx, n_idx * 4, dst, dbytes) || overlap(idx, n_idx * 4, residual_out, bytes))
        return WGS_ERR_ALIAS;
    RowArgs a{static_cast<const uint16_t *>(residual), static_cast<const uint16_t *>(branch),
              static_cast<uint16_t *>(residual_out), static_cast<uint16_t *>(dst), idx, n_idx, n_src,
              eps};
    return dispatch_width<RowOp::kAddNormGather, E>(a, width, stream);
}

// ------------------------------------------------ C entry points ------
// Each LayerNorm-family op has an fp16 and a bfloat16 entry point with the
// same arguments; the format only changes how elements widen and round.

extern "C" wgs_status ln_fwd(const void *x, void *y, int64_t rows, int32_t width, float eps,
                             cudaStream_t stream) {
    return ln_fwd_impl<Fp16>(x, y, rows, width, eps, stream);
}
extern "C" wgs_status ln_fwd_bf16(const void *x, void *y, int64_t rows, int32_t width, float eps,
                                  cudaStream_t stream) {
    return ln_fwd_impl<Bf16>(x, y, rows, width, eps, stream);
}

extern "C" wgs_status residual_add_ln_fwd(const void *residual, const void *branch,
                                          void *residual_out, void *y, int64_t rows,
                                          int32_t width, float eps, cudaStream_t stream) {
    return residual_add_ln_fwd_impl<Fp16>(residual, branch, residual_out, y, rows, width, eps,
                                          stream);
}
extern "C" wgs_status residual_add_ln_fwd_bf16(const void *residual, const void *branch,
                                               void *residual_out, void *y, int64_t rows,
                                               int32_t width, float eps, cudaStream_t stream) {
    return residual_add_ln_fwd_impl<Bf16>(residual, branch, residual_out, y, rows, width, eps,
                                          stream);
}

extern "C" wgs_status norm_gather(const void *src, const int32_t *idx, void *dst, int64_t n_src,
                                  int64_t n_idx, int32_t width, float eps, cudaStream_t stream) {
    return norm_gather_impl<Fp16>(src, idx, dst, n_src, n_idx, width, eps, stream);
}
extern "C" wgs_status norm_gather_bf16(const void *src, const int32_t *idx, void *dst,
                                       int64_t n_src, int64_t n_idx, int32_t width, float eps,
                                       cudaStream_t stream) {
    return norm_gather_impl<Bf16>(src, idx, dst, n_src, n_idx, width, eps, stream);
}

extern "C" wgs_status window_reverse_add_ln_fwd(const void *residual, const void *windows,
                                                const int32_t *inv_idx, void *residual_out,
                                                void *y, int64_t rows, int64_t n_windowed,
                                                int32_t width, float eps, cudaStream_t stream) {
    return window_reverse_add_ln_fwd_impl<Fp16>(residual, windows, inv_idx, residual_out, y, rows,
                                                n_windowed, width, eps, stream);
}
extern "C" wgs_status window_reverse_add_ln_fwd_bf16(const void *residual, const void *windows,
                                                     const int32_t *inv_idx, void *residual_out,
                                                     void *y, int64_t rows, int64_t n_windowed,
                                                     int32_t width, float eps,
                                                     cudaStream_t stream) {
    return window_reverse_add_ln_fwd_impl<Bf16>(residual, windows, inv_idx, residual_out, y, rows,
                                                n_windowed, width, eps, stream);
}

extern "C" wgs_status residual_add_norm_gather(const void *residual, const void *branch,
                                               const int32_t *idx, void *residual_out, void *dst,
                                               int64_t n_src, int64_t n_idx, int32_t width,
                                               float eps, cudaStream_t stream) {
    return residual_add_norm_gather_impl<Fp16>(residual, branch, idx, residual_out, dst, n_src,
                                               n_idx, width, eps, stream);
}
extern "C" wgs_status residual_add_norm_gather_bf16(const void *residual, const void *branch,
                                                    const int32_t *idx, void *residual_out,
                                                    void *dst, int64_t n_src, int64_t n_idx,
                                                    int32_t width, float eps,
                                                    cudaStream_t stream) {
    return residual_add_norm_gather_impl<Bf16>(residual, branch, idx, residual_out, dst, n_src,
                                               n_idx, width, eps, stream);
}

extern "C" wgs_status wgs_check_error(cudaStream_t stream) {
    // The error words are read and cleared by symbol, so each copy resolves
    // the word in the context current at this call.
    unsigned int seen = 0, seen_mask = 0;
    static const unsigned int cleared = 0;
    if (cudaMemcpyFromSymbolAsync(&seen, g_index_error, sizeof(seen), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_index_error, &cleared, sizeof(cleared), 0,
                                cudaMemcpyHostToDevice, stream) != cudaSuccess) {
        cudaGetLastError();  // clear this thread's error
        return WGS_ERR_CUDA;
    }
    if (bias_mask_error_take(&seen_mask, stream) != WGS_OK) return WGS_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return WGS_ERR_CUDA;
    }
    return (seen | seen_mask) ? WGS_ERR_INDEX : WGS_OK;
}
