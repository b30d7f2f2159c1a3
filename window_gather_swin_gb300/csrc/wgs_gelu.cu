// Fused bias + tanh-approximate GELU epilogue (sm_103a).
//
// Page "PyTorch + HIP fused bias + GELU on Hygon DCU", s3: the fused op
// must equal gelu(input + bias, approximate="tanh"), i.e.
//     t = x + bias[col],  y = 0.5 t (1 + tanh(sqrt(2/pi) (t + 0.044715 t^3))).
//
// Evaluation: 0.5 (1 + tanh(u)) = 1 / (1 + exp(-2u)) holds exactly, so
//     y = t / (1 + exp(z)),   z = -2u = t (k1 + k3 t^2),
//     k1 = -2 sqrt(2/pi),  k3 = -2 sqrt(2/pi) 0.044715.
// This avoids the cancellation of 1 + tanh(u) for negative t (where it
// tends to 0) and costs one exponential and one fast division per element.
//
// The op streams 2 x rows x width elements through HBM; the vector path
// moves 16-byte chunks and keeps U independent chunks in flight per thread.
// Bias chunks come through L1 (the whole bias row is at most a few KB).
#include "wgs_common.cuh"

#ifndef WGS_GELU_THREADS
#define WGS_GELU_THREADS 256
#endif
#ifndef WGS_GELU_U
#define WGS_GELU_U 4
#endif
#ifndef WGS_GELU_CTAS_PER_SM
#define WGS_GELU_CTAS_PER_SM 8
#endif

namespace wgs {

// Below t = -4 the exponent z exceeds ~11 and grows like |t|^3; an FP32 z
// then carries an absolute error of |z| * (a few ulp), which the exponential
// turns into a relative error of the result approaching 1e-5.  Those inputs
// (about 3e-5 of an N(0,1) tensor) take the same formula in FP64 instead.
__device__ __noinline__ float gelu_tanh_far_left(float t) {
    constexpr double kSqrt2OverPi = 0.7978845608028654;
    const double td = t;
    const double z = td * (-2.0 * kSqrt2OverPi) * (1.0 + 0.044715 * td * td);
    return static_cast<float>(td / (1.0 + exp(z)));
}

__device__ __forceinline__ float gelu_tanh(float t) {
    constexpr double kSqrt2OverPi = 0.7978845608028654;
    constexpr float k1 = static_cast<float>(-2.0 * kSqrt2OverPi);
    constexpr float k3 = static_cast<float>(-2.0 * kSqrt2OverPi * 0.044715);
    if (t < -4.0f) return gelu_tanh_far_left(t);
    const float z = t * fmaf(k3, t * t, k1);
    return __fdividef(t, 1.0f + expf(z));
}

// One 16-byte chunk: 4 fp32 or 8 fp16 elements and the matching bias chunk.
template <bool kHalf>
__device__ __forceinline__ uint4 gelu_chunk(const uint4 &xv, const uint4 &bv) {
    uint4 out;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if constexpr (kHalf) {
            const float2 x = half2_to_float2(word(xv, j));
            const float2 b = half2_to_float2(word(bv, j));
            // t is rounded to fp16 first, as an unfused fp16 add would leave it
            const float2 t = half2_to_float2(float2_to_half2(x.x + b.x, x.y + b.y));
            set_word(out, j, float2_to_half2(gelu_tanh(t.x), gelu_tanh(t.y)));
        } else {
            const float t = __uint_as_float(word(xv, j)) + __uint_as_float(word(bv, j));
            set_word(out, j, __float_as_uint(gelu_tanh(t)));
        }
    }
    return out;
}

// Flat grid-stride over 16-byte chunks.  Chunk i belongs to column chunk
// i mod row_vecs; each thread tracks that column incrementally (all steps
// are below row_vecs, so one conditional subtraction keeps it in range).
template <bool kHalf, int U, int THREADS>
__global__ void __launch_bounds__(THREADS)
bias_gelu_vec_kernel(const uint4 *x, const uint4 *bias, uint4 *y, int64_t n_vec, int32_t row_vecs) {
    constexpr int64_t kTile = static_cast<int64_t>(THREADS) * U;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kTile;
    const int32_t in_tile = THREADS % row_vecs;
    const int32_t per_iter = static_cast<int32_t>(stride % row_vecs);
    int64_t i0 = static_cast<int64_t>(blockIdx.x) * kTile + threadIdx.x;
    int32_t col0 = static_cast<int32_t>(i0 % row_vecs);
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
            if (i < n_vec) st_stream(y + i, gelu_chunk<kHalf>(xv[u], bv[u]));
        }
        col0 += per_iter;
        if (col0 >= row_vecs) col0 -= row_vecs;
    }
}

// Any width, any element alignment: one element per thread per step.
template <bool kHalf>
__global__ void __launch_bounds__(256)
bias_gelu_scalar_kernel(const void *xp, const void *bp, void *yp, int64_t n, int32_t width) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t c = static_cast<int32_t>(i % width);
        if constexpr (kHalf) {
            const __half *x = static_cast<const __half *>(xp);
            const __half *b = static_cast<const __half *>(bp);
            const __half t = __float2half_rn(__half2float(x[i]) + __half2float(b[c]));
            static_cast<__half *>(yp)[i] = __float2half_rn(gelu_tanh(__half2float(t)));
        } else {
            const float *x = static_cast<const float *>(xp);
            const float *b = static_cast<const float *>(bp);
            static_cast<float *>(yp)[i] = gelu_tanh(x[i] + b[c]);
        }
    }
}

template <bool kHalf>
wgs_status launch_gelu(const void *x, const void *bias, void *y, int64_t rows, int32_t width,
                       int sm_count, cudaStream_t stream) {
    constexpr int kVec = kHalf ? 8 : 4;
    const int64_t n = rows * width;
    const bool vec = width % kVec == 0 && aligned16(x) && aligned16(bias) && aligned16(y);
    if (vec) {
        constexpr int T = WGS_GELU_THREADS, U = WGS_GELU_U;
        const int64_t n_vec = n / kVec;
        const int64_t need = ceil_div(n_vec, static_cast<int64_t>(T) * U);
        const int64_t cap = static_cast<int64_t>(sm_count) * WGS_GELU_CTAS_PER_SM;
        bias_gelu_vec_kernel<kHalf, U, T><<<static_cast<unsigned>(need < cap ? need : cap), T, 0,
                                            stream>>>(static_cast<const uint4 *>(x),
                                                      static_cast<const uint4 *>(bias),
                                                      static_cast<uint4 *>(y), n_vec, width / kVec);
    } else {
        const int64_t need = ceil_div(n, 256);
        const int64_t cap = static_cast<int64_t>(sm_count) * 8;
        bias_gelu_scalar_kernel<kHalf><<<static_cast<unsigned>(need < cap ? need : cap), 256, 0,
                                         stream>>>(x, bias, y, n, width);
    }
    return launch_status();
}

}  // namespace wgs

using namespace wgs;

extern "C" wgs_status bias_gelu_tanh(const void *x, const void *bias, void *y, int64_t rows,
                                     int32_t width, wgs_dtype dtype, cudaStream_t stream) {
    if (dtype != WGS_F32 && dtype != WGS_F16) return WGS_ERR_DTYPE;
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
    return dtype == WGS_F16 ? launch_gelu<true>(x, bias, y, rows, width, dev.sm_count, stream)
                            : launch_gelu<false>(x, bias, y, rows, width, dev.sm_count, stream);
}
