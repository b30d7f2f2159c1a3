// Fused bias + tanh-approximate GELU epilogue (sm_103a).
//
// Page "PyTorch + HIP fused bias + GELU on Hygon DCU", s3: the fused op
// must equal gelu(input + bias, approximate="tanh"), i.e.
//     t = x + bias[col],  y = 0.5 t (1 + tanh(sqrt(2/pi) (t + 0.044715 t^3))).
//
// Evaluation.  0.5 (1 + tanh(u)) = 1 / (1 + exp(-2u)) holds exactly, and
// exp(v) = 2^(v log2 e), so
//     y = t / (1 + 2^w),   w = -2u log2 e = t (c1 + c3 t^2),
//     c1 = -2 sqrt(2/pi) log2 e,  c3 = -2 sqrt(2/pi) 0.044715 log2 e.
// The power of two and the reciprocal are the PTX ex2.approx and
// rcp.approx instructions (one MUFU operation each, relative error near
// 2^-22), and the FP32 arithmetic runs two elements per instruction on the
// packed pipe, so an element costs a handful of instructions: fp16 data carries
// eight elements per 16 bytes, and a full-precision exp / divide would make
// the kernel issue-bound instead of HBM-bound.  The form has no
// cancellation for negative t, where 1 + tanh(u) tends to 0.
//
// Below t = -4, w exceeds 15 and grows like |t|^3, so an FP32 w carries an
// absolute error of |w| times a few ulp, which 2^w turns into a relative
// error of the result approaching 1e-5.  Those inputs (about 3e-5 of an
// N(0,1) tensor) are recomputed from the same formula in FP64.
//
// The op streams 2 x rows x width elements through HBM; the vector path
// moves 16-byte chunks.  Rows of at least 64 chunks run as short CTAs of R
// rows x one column block, a thread per column chunk (16-bit data: two
// steps of R rows, the second staged in shared memory while the first
// computes); narrower rows run a one-wave grid-stride kernel with U chunks
// in flight per thread.  Bias
// chunks come through L1 (the whole bias row is at most a few KB).
#include <atomic>
#include <type_traits>

#include "wgs_common.cuh"

#ifndef WGS_GELU_EARLY
#define WGS_GELU_EARLY 1  // row-block form: L2 prefetch of the first chunks before the wait
#endif
#ifndef WGS_GELU_STAGED_STEPS
#define WGS_GELU_STAGED_STEPS 2  // 16-bit row-block CTAs of this many steps of R rows, staged (0: off)
#endif
#ifndef WGS_GELU_THREADS
#define WGS_GELU_THREADS 256
#endif
#ifndef WGS_GELU_U
#define WGS_GELU_U 4
#endif
#ifndef WGS_GELU_U16
#define WGS_GELU_U16 2  // chunks per thread per pass for 16-bit data, with prefetch
#endif
#ifndef WGS_GELU_R16
#define WGS_GELU_R16 3  // rows per step in the row-block form, 16-bit data
#endif
#ifndef WGS_GELU_R32
#define WGS_GELU_R32 4  // rows per thread in the row-block form, fp32
#endif
#ifndef WGS_GELU_CTAS_PER_SM
#define WGS_GELU_CTAS_PER_SM 0  // grid cap in CTAs per SM; 0: as many as can be resident
#endif
#ifdef WGS_GELU_MIN_CTAS  // optional register cap: resident CTAs per SM to aim for
#define WGS_GELU_BOUNDS(T) __launch_bounds__(T, WGS_GELU_MIN_CTAS)
#else
#define WGS_GELU_BOUNDS(T) __launch_bounds__(T)
#endif

namespace wgs {

constexpr double kSqrt2OverPi = 0.7978845608028654;
constexpr double kLog2e = 1.4426950408889634;
constexpr float kFarLeft = -4.0f;

__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Valid for t >= kFarLeft (and for +inf and NaN).
__device__ __forceinline__ float gelu_tanh_fast(float t) {
    constexpr float c1 = static_cast<float>(-2.0 * kSqrt2OverPi * kLog2e);
    constexpr float c3 = static_cast<float>(-2.0 * kSqrt2OverPi * 0.044715 * kLog2e);
    const float w = t * fmaf(c3, t * t, c1);
    return t * rcp_approx(1.0f + ex2_approx(w));
}

// Two elements at once on the packed FP32 pipe of the sm_100 family
// (__fmul2_rn / __fadd2_rn / __ffma2_rn: each lane is the correctly rounded
// scalar operation), so the pair equals gelu_tanh_fast of each element.
__device__ __forceinline__ float2 gelu_tanh_fast2(float2 t) {
    constexpr float c1 = static_cast<float>(-2.0 * kSqrt2OverPi * kLog2e);
    constexpr float c3 = static_cast<float>(-2.0 * kSqrt2OverPi * 0.044715 * kLog2e);
    const float2 w = __fmul2_rn(t, __ffma2_rn(make_float2(c3, c3), __fmul2_rn(t, t),
                                              make_float2(c1, c1)));
    const float2 d = __fadd2_rn(make_float2(1.0f, 1.0f),
                                make_float2(ex2_approx(w.x), ex2_approx(w.y)));
    return __fmul2_rn(t, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// Any t, in FP64 (taken only for t < kFarLeft).
__device__ __noinline__ float gelu_tanh_far_left(float t) {
    const double td = t;
    const double z = td * (-2.0 * kSqrt2OverPi) * (1.0 + 0.044715 * td * td);
    return static_cast<float>(td / (1.0 + exp(z)));
}

__device__ __forceinline__ float gelu_tanh(float t) {
    return t < kFarLeft ? gelu_tanh_far_left(t) : gelu_tanh_fast(t);
}

// Element formats: F32 here, Fp16 / Bf16 from wgs_common.cuh.
struct F32 {};

// One 16-byte chunk: 4 fp32 or 8 16-bit elements and the matching bias
// chunk.  The fast formula runs on every element; the rare far-left
// elements are redone afterwards behind one branch per chunk.
template <typename E>
__device__ __forceinline__ uint4 gelu_chunk(const uint4 &xv, const uint4 &bv) {
    constexpr bool k16 = !std::is_same<E, F32>::value;
    constexpr int kN = k16 ? 8 : 4;
    float t[kN], y[kN];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if constexpr (k16) {
            // t = round(x + b) in the tensor's 16-bit format, the rounding
            // point of an unfused add in that precision (E::add2 rounds the
            // exact sum once)
            const float2 tf = E::to_f2(E::add2(word(xv, j), word(bv, j)));
            t[2 * j] = tf.x;
            t[2 * j + 1] = tf.y;
        } else {
            t[j] = __uint_as_float(word(xv, j)) + __uint_as_float(word(bv, j));
        }
    }
    float lowest = t[0];  // NaN elements need no redo: the fast form already gives NaN
#pragma unroll
    for (int e = 0; e < kN; e += 2) {
        const float2 v = gelu_tanh_fast2(make_float2(t[e], t[e + 1]));
        y[e] = v.x;
        y[e + 1] = v.y;
        lowest = fminf(lowest, fminf(t[e], t[e + 1]));
    }
    if (lowest < kFarLeft) {
#pragma unroll
        for (int e = 0; e < kN; ++e)
            if (t[e] < kFarLeft) y[e] = gelu_tanh_far_left(t[e]);
    }
    uint4 out;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if constexpr (k16)
            set_word(out, j, E::from_f2(y[2 * j], y[2 * j + 1]));
        else
            set_word(out, j, __float_as_uint(y[j]));
    }
    return out;
}

// Flat grid-stride over 16-byte chunks.  Chunk i belongs to column chunk
// i mod row_vecs; each thread tracks that column incrementally (all steps
// are below row_vecs, so one conditional subtraction keeps it in range).
// With PF the x chunks of the next pass are loaded before this pass's
// arithmetic, so each thread keeps loads in flight while it computes.
template <typename E, int U, int THREADS, bool PF>
__global__ void WGS_GELU_BOUNDS(THREADS)
bias_gelu_vec_kernel(const uint4 *x, const uint4 *bias, uint4 *y, int64_t n_vec, int32_t row_vecs) {
    pdl_prologue();
    constexpr int64_t kTile = static_cast<int64_t>(THREADS) * U;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kTile;
    const int32_t in_tile = THREADS % row_vecs;
    const int32_t per_iter = static_cast<int32_t>(stride % row_vecs);
    int64_t i0 = static_cast<int64_t>(blockIdx.x) * kTile + threadIdx.x;
    int32_t col0 = static_cast<int32_t>(i0 % row_vecs);
    if constexpr (PF) {
        // x chunks of the next pass load while this pass computes
        uint4 nx[U];
        auto fetch = [&](int64_t base, uint4 *dst) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = base + static_cast<int64_t>(u) * THREADS;
                if (i < n_vec) dst[u] = ld_stream(x + i);
            }
        };
        fetch(i0, nx);
        for (; i0 < n_vec; i0 += stride) {
            uint4 xv[U], bv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) xv[u] = nx[u];
            fetch(i0 + stride, nx);
            int32_t col = col0;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                bv[u] = __ldg(bias + col);
                col += in_tile;
                if (col >= row_vecs) col -= row_vecs;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + static_cast<int64_t>(u) * THREADS;
                if (i < n_vec) st_stream(y + i, gelu_chunk<E>(xv[u], bv[u]));
            }
            col0 += per_iter;
            if (col0 >= row_vecs) col0 -= row_vecs;
        }
    } else {
        for (; i0 < n_vec; i0 += stride) {
            uint4 xv[U], bv[U];
            int32_t col = col0;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + static_cast<int64_t>(u) * THREADS;
                if (i < n_vec) {
                    xv[u] = ld_stream(x + i);
                    bv[u] = __ldg(bias + col);
                }
                col += in_tile;
                if (col >= row_vecs) col -= row_vecs;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = i0 + static_cast<int64_t>(u) * THREADS;
                if (i < n_vec) st_stream(y + i, gelu_chunk<E>(xv[u], bv[u]));
            }
            col0 += per_iter;
            if (col0 >= row_vecs) col0 -= row_vecs;
        }
    }
}

// Row-block form, for rows of at least kRowFormMinVecs chunks: CTA (row
// block, column block); thread j owns column chunk blockIdx.y * cv + j of R
// consecutive rows, with its bias chunk loaded once and the R chunks in
// flight together.  The grid holds many short CTAs, so the hardware keeps
// every SM fed as CTAs finish, with no index division anywhere.
constexpr int32_t kRowFormMinVecs = 64;

template <typename E, int R>
__global__ void __launch_bounds__(256)
bias_gelu_rows_kernel(const uint4 *x, const uint4 *bias, uint4 *y, int64_t rows,
                      int32_t row_vecs, int32_t cv) {
    const int32_t c = static_cast<int32_t>(blockIdx.y) * cv + static_cast<int32_t>(threadIdx.x);
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * R;
#if WGS_GELU_EARLY
    // L2 prefetch of this thread's chunks before waiting for the previous
    // grid (a latency hint only: the loads below come after the wait)
    if (c < row_vecs) {
        prefetch_l2(bias + c);
#pragma unroll
        for (int q = 0; q < R; ++q)
            if (r0 + q < rows) prefetch_l2(x + (r0 + q) * row_vecs + c);
    }
#endif
    pdl_prologue();
    if (c >= row_vecs) return;
    const uint4 bv = __ldg(bias + c);
    uint4 xv[R];
#pragma unroll
    for (int q = 0; q < R; ++q)
        if (r0 + q < rows) xv[q] = ld_stream(x + (r0 + q) * row_vecs + c);
#pragma unroll
    for (int q = 0; q < R; ++q)
        if (r0 + q < rows) st_stream(y + (r0 + q) * row_vecs + c, gelu_chunk<E>(xv[q], bv));
}

// Row-block form with STEPS steps of R rows per CTA, for 16-bit data: the
// next step's chunks are copied into shared memory (each thread its own
// slots, cp.async) while this step computes, so a CTA overlaps its own loads
// with its arithmetic without holding the next step in registers.  Eight
// elements a chunk make the arithmetic long; with all of a CTA's rows loaded
// at once (the plain row-block form, 4 rows) the loads of other CTAs did not
// cover it.  Measured on GB300 at [32760,1536]: 32.8 -> 30.5 us with 2 steps
// of 3 rows (4 rows: 30.7; 3 steps: 30.9; 2 rows: 31.4).  fp32, with half
// the arithmetic per chunk, was slower staged (113.2 -> 113.9-114.5 us).
template <typename E, int R, int STEPS>
__global__ void __launch_bounds__(256)
bias_gelu_rows_staged(const uint4 *x, const uint4 *bias, uint4 *y, int64_t rows,
                      int32_t row_vecs, int32_t cv) {
    extern __shared__ uint4 ring[];  // [2][R][blockDim]
    const int tid = threadIdx.x, nt = blockDim.x;
    const int32_t c = static_cast<int32_t>(blockIdx.y) * cv + tid;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * R * STEPS;
#if WGS_GELU_EARLY
    if (c < row_vecs) {
        prefetch_l2(bias + c);
#pragma unroll
        for (int q = 0; q < R; ++q)
            if (r0 + q < rows) prefetch_l2(x + (r0 + q) * row_vecs + c);
    }
#endif
    pdl_prologue();
    if (c >= row_vecs) return;
    auto issue = [&](int st) {
        const int slot = st & 1;
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t r = r0 + st * R + q;
            if (st < STEPS && r < rows) cp_async16(&ring[(slot * R + q) * nt + tid], x + r * row_vecs + c);
        }
        cp_async_commit();
    };
    const uint4 bv = __ldg(bias + c);
    issue(0);
#pragma unroll 1
    for (int st = 0; st < STEPS; ++st) {
        issue(st + 1);
        cp_async_wait<1>();
        const int slot = st & 1;
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t r = r0 + st * R + q;
            if (r < rows)
                st_stream(y + r * row_vecs + c, gelu_chunk<E>(ring[(slot * R + q) * nt + tid], bv));
        }
    }
    cp_async_wait<0>();
}

// Any width, any element alignment: one element per thread per step.
template <typename E>
__global__ void __launch_bounds__(256)
bias_gelu_scalar_kernel(const void *xp, const void *bp, void *yp, int64_t n, int32_t width) {
    pdl_prologue();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t c = static_cast<int32_t>(i % width);
        if constexpr (std::is_same<E, F32>::value) {
            const float *x = static_cast<const float *>(xp);
            const float *b = static_cast<const float *>(bp);
            static_cast<float *>(yp)[i] = gelu_tanh(x[i] + b[c]);
        } else {
            // one 16-bit element in the low half of a word
            const uint16_t *x = static_cast<const uint16_t *>(xp);
            const uint16_t *b = static_cast<const uint16_t *>(bp);
            const float t = E::to_f2(E::add2(x[i], b[c])).x;
            static_cast<uint16_t *>(yp)[i] = static_cast<uint16_t>(E::from_f2(gelu_tanh(t), 0.f));
        }
    }
}

template <typename E>
wgs_status launch_gelu(const void *x, const void *bias, void *y, int64_t rows, int32_t width,
                       int device, int sm_count, cudaStream_t stream) {
    constexpr int kVec = std::is_same<E, F32>::value ? 4 : 8;
    const int64_t n = rows * width;
    const bool vec = width % kVec == 0 && aligned16(x) && aligned16(bias) && aligned16(y);
    if (vec) {
        constexpr bool PF = !std::is_same<E, F32>::value;
        constexpr int R = PF ? WGS_GELU_R16 : WGS_GELU_R32;
        const int32_t row_vecs = static_cast<int32_t>(width / kVec);
        if constexpr (PF && WGS_GELU_STAGED_STEPS > 0) {
            constexpr int ST = WGS_GELU_STAGED_STEPS;
            if (row_vecs >= kRowFormMinVecs &&
                ceil_div(rows, static_cast<int64_t>(R) * ST) <= INT32_MAX) {
                const int32_t cv = row_vecs <= 256 ? row_vecs : 256;
                const dim3 grid(static_cast<unsigned>(ceil_div(rows, static_cast<int64_t>(R) * ST)),
                                static_cast<unsigned>(ceil_div(row_vecs, cv)));
                const size_t smem = static_cast<size_t>(2) * R * cv * sizeof(uint4);
                return launch(bias_gelu_rows_staged<E, R, ST>, grid, dim3(static_cast<unsigned>(cv)),
                              smem, stream, static_cast<const uint4 *>(x),
                              static_cast<const uint4 *>(bias), static_cast<uint4 *>(y), rows,
                              row_vecs, cv);
            }
        }
        if (row_vecs >= kRowFormMinVecs && ceil_div(rows, static_cast<int64_t>(R)) <= INT32_MAX) {
            const int32_t cv = row_vecs <= 256 ? row_vecs : 256;
            const dim3 grid(static_cast<unsigned>(ceil_div(rows, static_cast<int64_t>(R))),
                            static_cast<unsigned>(ceil_div(row_vecs, cv)));
            return launch(bias_gelu_rows_kernel<E, R>, grid, dim3(static_cast<unsigned>(cv)), 0,
                          stream, static_cast<const uint4 *>(x), static_cast<const uint4 *>(bias),
                          static_cast<uint4 *>(y), rows, row_vecs, cv);
        }
        // Narrower rows: one resident wave of grid-stride CTAs.  16-bit data
        // takes fewer chunks per pass, the next pass's loads issued before
        // this pass computes (eight elements a chunk make the compute long
        // enough to hide behind them); fp32 more chunks, no prefetch.
        constexpr int T = WGS_GELU_THREADS, U = PF ? WGS_GELU_U16 : WGS_GELU_U;
        const int64_t n_vec = n / kVec;
        const int64_t need = ceil_div(n_vec, static_cast<int64_t>(T) * U);
        // One resident wave of grid-stride CTAs: a partial second wave
        // would leave SMs idle at the end of this bandwidth-bound stream.
        auto kernel = bias_gelu_vec_kernel<E, U, T, PF>;
        static std::atomic<int> resident[64];  // per device, for this instantiation
        int per_sm = WGS_GELU_CTAS_PER_SM > 0 ? WGS_GELU_CTAS_PER_SM
                                              : resident[device].load(std::memory_order_relaxed);
        if (per_sm == 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, T, 0) != cudaSuccess ||
                per_sm < 1)
                return WGS_ERR_LAUNCH;
            resident[device].store(per_sm, std::memory_order_relaxed);
        }
        const int64_t cap = static_cast<int64_t>(sm_count) * per_sm;
        return launch(kernel,
                      dim3(static_cast<unsigned>(need < cap ? need : cap)), dim3(T), 0, stream,
                      static_cast<const uint4 *>(x), static_cast<const uint4 *>(bias),
                      static_cast<uint4 *>(y), n_vec, static_cast<int32_t>(width / kVec));
    }
    const int64_t need = ceil_div(n, 256);
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    return launch(bias_gelu_scalar_kernel<E>, dim3(static_cast<unsigned>(need < cap ? need : cap)),
                  dim3(256), 0, stream, x, bias, y, n, width);
}

}  // namespace wgs

using namespace wgs;

extern "C" wgs_status bias_gelu_tanh(const void *x, const void *bias, void *y, int64_t rows,
                                     int32_t width, wgs_dtype dtype, cudaStream_t stream) {
    if (dtype != WGS_F32 && dtype != WGS_F16 && dtype != WGS_BF16) return WGS_ERR_DTYPE;
    if (rows < 0 || width < 0) return WGS_ERR_SHAPE;
    const int64_t esz = dtype == WGS_F32 ? 4 : 2;
    if (width > 0 && rows > INT64_MAX / esz / width) return WGS_ERR_SHAPE;
    if (rows == 0 || width == 0) return WGS_OK;
    if (!x || !bias || !y) return WGS_ERR_NULL;
    const uintptr_t mask = static_cast<uintptr_t>(esz - 1);
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(bias) |
         reinterpret_cast<uintptr_t>(y)) & mask)
        return WGS_ERR_ALIGN;
    const int64_t bytes = rows * width * esz;
    if (!same_or_disjoint(x, y, bytes) || overlap(bias, width * esz, y, bytes)) return WGS_ERR_ALIAS;
    DeviceInfo dev;
    const wgs_status st = current_device(&dev);
    if (st != WGS_OK) return st;
    switch (dtype) {
        case WGS_F16:
            return launch_gelu<Fp16>(x, bias, y, rows, width, dev.device, dev.sm_count, stream);
        case WGS_BF16:
            return launch_gelu<Bf16>(x, bias, y, rows, width, dev.device, dev.sm_count, stream);
        default:
            return launch_gelu<F32>(x, bias, y, rows, width, dev.device, dev.sm_count, stream);
    }
}
