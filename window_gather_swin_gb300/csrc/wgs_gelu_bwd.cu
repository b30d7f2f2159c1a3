// Backward of the fused bias + tanh-GELU epilogue (sm_103a).
//
// Page "PyTorch + HIP fused bias + GELU on Hygon DCU", s3, leaves backward
// out of its tutorial op; this is the gradient of y = gelu(x + bias) with
// the rounding points of an eager backward:
//     t         = round(x + bias[c])                     (as the forward)
//     grad_x    = round(grad_y * gelu'(t))
//     grad_bias = round(sum over rows of grad_x[., c])
// With s = 1 / (1 + 2^w), w = t (c1 + c3 t^2) as in the forward (so
// s = 0.5 (1 + tanh u)) and 1 - s = 2^w s:
//     gelu'(t) = s + t s (1 - s) (2k + 6k a t^2),   k = sqrt(2/pi), a = 0.044715.
// Below t = -4 the FP64 form runs, as in the forward.
//
// The FP32 arithmetic of gelu' runs two elements per instruction on the
// packed FP32 pipe (__fmul2_rn and friends: each lane is the correctly
// rounded scalar operation), which roughly halves the instructions per
// element; the kernel must stay HBM-bound with eight fp16 elements per
// 16-byte load.
//
// The column sum is deterministic and runs in two passes:
//   1. grid (slab, column block): every thread owns one 16-byte column chunk
//      (or one column on the scalar path), walks rows r0 + g, r0 + g + G, ...
//      of its slab, stores grad_x and accumulates the rounded gradients in
//      FP32 registers; the G row groups of the CTA then combine in shared
//      memory in a fixed order into partial[slab][column];
//   2. per column, 32 lanes sum interleaved slabs in order and then combine
//      in lane order (gelu_bwd_bias).
// The slab count depends only on the row count and G only on the shape and
// format, so results do not depend on the device.  Both passes stream:
// grad_y and x are read once and grad_x is written once; the partials are a
// few MB at most.
#include <atomic>
#include <type_traits>

#include "wgs_common.cuh"

#ifndef WGS_BWD_EARLY
#define WGS_BWD_EARLY 1  // pass 1: L2 prefetch of the first step before the wait
#endif
#ifndef WGS_BWD_ROWS
#define WGS_BWD_ROWS 2  // rows per step per thread (two steps in flight)
#endif
#ifndef WGS_BWD_GROUPS
#define WGS_BWD_GROUPS 4  // most row groups per CTA
#endif
#ifndef WGS_BWD_TARGET_THREADS
// pass-1 threads to aim for when choosing row groups: one 768-thread CTA on
// each of 152 SMs, all that stay resident at the 80-register cap
#define WGS_BWD_TARGET_THREADS 116736
#endif
#ifndef WGS_BWD_MIN_BLOCKS
#define WGS_BWD_MIN_BLOCKS 1  // pass-1 CTAs of the largest size kept resident per SM
#endif
#ifndef WGS_BWD_ASYNC
#define WGS_BWD_ASYNC 1  // 16-bit pass 1 stages its next step in shared memory (cp.async)
#endif
#ifndef WGS_BWD_ASYNC_STAGES
#define WGS_BWD_ASYNC_STAGES 2  // ring slots per thread on that path
#endif
#ifndef WGS_BWD_MIN_SLAB_ROWS
// slab count = min(608, ceil(rows / this)): 32760 rows give 152 slabs, which
// with four row groups fill the resident thread slots exactly
#define WGS_BWD_MIN_SLAB_ROWS 216
#endif

namespace wgs {

namespace {

struct F32 {};

constexpr double kSqrt2OverPi = 0.7978845608028654;
constexpr double kLog2e = 1.4426950408889634;
constexpr float kFarLeft = -4.0f;
constexpr int64_t kMinRowsPerSlab = WGS_BWD_MIN_SLAB_ROWS;
// At most 608 slabs: four 192-thread CTAs (one row group, 80 registers) on
// each of 152 SMs, so a tall shape of 192-chunk rows fills every resident
// slot in one wave (fp32 [131040,768]: 186.9 -> 181.7 us against 512 slabs).
constexpr int64_t kMaxSlabs = 608;
constexpr int kMaxChunksPerBlock = 256;  // column chunks per CTA
// Pass 1 runs at most 768 threads per CTA and keeps one such CTA per SM
// resident (at most 85 registers a thread; the kernels use 78-80, so four
// 192-thread CTAs fit as well), so the usual grids fit in one wave.
constexpr int kMaxThreads = 768;
constexpr int kMinBlocks = WGS_BWD_MIN_BLOCKS;

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

__device__ __noinline__ float gelu_grad_far_left(float t) {
    const double td = t;
    const double k = kSqrt2OverPi;
    const double z = td * (-2.0 * k) * (1.0 + 0.044715 * td * td);  // -2u
    const double e = exp(z);                 // e^{-2u}, may be +inf
    const double s = 1.0 / (1.0 + e);        // 0.5 (1 + tanh u)
    const double one_minus_s = 1.0 / (1.0 + 1.0 / e);
    return static_cast<float>(s + td * s * one_minus_s * (2.0 * k) * (1.0 + 3.0 * 0.044715 * td * td));
}

// Valid for t >= kFarLeft (and +inf / NaN, which give NaN like the FP64 form).
__device__ __forceinline__ float gelu_grad_fast(float t) {
    constexpr float c1 = static_cast<float>(-2.0 * kSqrt2OverPi * kLog2e);
    constexpr float c3 = static_cast<float>(-2.0 * kSqrt2OverPi * 0.044715 * kLog2e);
    constexpr float k1 = static_cast<float>(2.0 * kSqrt2OverPi);
    constexpr float k3 = static_cast<float>(6.0 * kSqrt2OverPi * 0.044715);
    const float t2 = t * t;
    const float e = ex2_approx(t * fmaf(c3, t2, c1));
    const float s = rcp_approx(1.0f + e);
    return fmaf(t * s * (e * s), fmaf(k3, t2, k1), s);
}

// gelu_grad_fast of two elements, on the packed FP32 pipe (each lane is the
// correctly rounded scalar operation, in the same order).
__device__ __forceinline__ float2 gelu_grad_fast2(float2 t) {
    constexpr float c1 = static_cast<float>(-2.0 * kSqrt2OverPi * kLog2e);
    constexpr float c3 = static_cast<float>(-2.0 * kSqrt2OverPi * 0.044715 * kLog2e);
    constexpr float k1 = static_cast<float>(2.0 * kSqrt2OverPi);
    constexpr float k3 = static_cast<float>(6.0 * kSqrt2OverPi * 0.044715);
    const float2 t2 = __fmul2_rn(t, t);
    const float2 w = __fmul2_rn(t, __ffma2_rn(make_float2(c3, c3), t2, make_float2(c1, c1)));
    const float2 e = make_float2(ex2_approx(w.x), ex2_approx(w.y));
    const float2 d = __fadd2_rn(make_float2(1.0f, 1.0f), e);
    const float2 s = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    const float2 ts_es = __fmul2_rn(__fmul2_rn(t, s), __fmul2_rn(e, s));
    return __ffma2_rn(ts_es, __ffma2_rn(make_float2(k3, k3), t2, make_float2(k1, k1)), s);
}

__device__ __forceinline__ float gelu_grad(float t) {
    return t < kFarLeft ? gelu_grad_far_left(t) : gelu_grad_fast(t);
}

// Element pair w of a chunk as FP32: t = round(x + b) and g = grad_y, for
// 16-bit words (one pair per word) or fp32 words (pair = words 2w, 2w + 1).
template <typename E, bool k16>
__device__ __forceinline__ void chunk_pair(const uint4 &gyv, const uint4 &xv, const uint4 &bv,
                                           int w, float2 &t, float2 &g) {
    if constexpr (k16) {
        t = E::to_f2(E::add2(word(xv, w), word(bv, w)));
        g = E::to_f2(word(gyv, w));
    } else {
        t = make_float2(__uint_as_float(word(xv, 2 * w)) + __uint_as_float(word(bv, 2 * w)),
                        __uint_as_float(word(xv, 2 * w + 1)) + __uint_as_float(word(bv, 2 * w + 1)));
        g = make_float2(__uint_as_float(word(gyv, 2 * w)), __uint_as_float(word(gyv, 2 * w + 1)));
    }
}

// Store the pair v = grad_x of pair w into out (rounded for 16-bit words).
template <typename E, bool k16>
__device__ __forceinline__ void put_pair(uint4 &out, int w, float2 v) {
    if constexpr (k16) {
        set_word(out, w, E::from_f2(v.x, v.y));
    } else {
        set_word(out, 2 * w, __float_as_uint(v.x));
        set_word(out, 2 * w + 1, __float_as_uint(v.y));
    }
}

// The chunk with gelu_grad chosen per element (far-left elements in FP64);
// only chunks holding some t < -4 come here.
template <typename E, bool k16>
__device__ __forceinline__ uint4 grad_chunk_exact(uint4 gyv, uint4 xv, uint4 bv) {
    uint4 out;
    for (int w = 0; w < (k16 ? 4 : 2); ++w) {
        float2 t, g;
        chunk_pair<E, k16>(gyv, xv, bv, w, t, g);
        put_pair<E, k16>(out, w, make_float2(g.x * gelu_grad(t.x), g.y * gelu_grad(t.y)));
    }
    return out;
}

// One 16-byte chunk: grad_x = round(gy * gelu'(round(x + b))) for its 4 or
// 8 elements, and the rounded values added to acc.  The packed fast form
// runs on every pair; a chunk with a far-left element is redone by
// grad_chunk_exact, which gives the same bits everywhere else.
template <typename E, bool k16>
__device__ __forceinline__ uint4 grad_chunk(const uint4 &gyv, const uint4 &xv, const uint4 &bv,
                                            float2 *acc) {
    constexpr int kPairs = k16 ? 4 : 2;
    uint4 out;
    float lowest = INFINITY;  // NaN needs no redo: the fast form gives NaN too
#pragma unroll
    for (int w = 0; w < kPairs; ++w) {
        float2 t, g;
        chunk_pair<E, k16>(gyv, xv, bv, w, t, g);
        put_pair<E, k16>(out, w, __fmul2_rn(g, gelu_grad_fast2(t)));
        lowest = fminf(lowest, fminf(t.x, t.y));
    }
    if (lowest < kFarLeft) out = grad_chunk_exact<E, k16>(gyv, xv, bv);
#pragma unroll
    for (int w = 0; w < kPairs; ++w) {
        if constexpr (k16)
            acc[w] = E::widen_add2(word(out, w), acc[w]);
        else
            acc[w] = __fadd2_rn(acc[w], make_float2(__uint_as_float(word(out, 2 * w)),
                                                    __uint_as_float(word(out, 2 * w + 1))));
    }
    return out;
}

// Pass 1, 16-byte chunks.  Block = CVB * G threads: thread (g, j) owns
// column chunk blockIdx.y * CVB + j and walks rows r0 + g, r0 + g + G, ...
// of its slab, R rows a step, accumulating them in increasing row order.
// The next step's loads are issued before this step's arithmetic, so each
// thread keeps loads in flight while it computes.
template <typename E, int R>
__global__ void __launch_bounds__(kMaxThreads, kMinBlocks)
gelu_bwd_chunks(const uint4 *gy, const uint4 *x, const uint4 *bias, uint4 *gx, float *partial,
                int64_t rows, int32_t row_chunks, int32_t width, int32_t cvb, int32_t groups,
                int32_t slabs) {
    constexpr bool k16 = !std::is_same<E, F32>::value;
    constexpr int kN = k16 ? 8 : 4;
    extern __shared__ float red[];  // [groups][cvb][kN]
    const int j = threadIdx.x % cvb, g = threadIdx.x / cvb;
    const int32_t cv = static_cast<int32_t>(blockIdx.y) * cvb + j;
    const bool active = g < groups && cv < row_chunks;
    const int64_t r0 = rows * blockIdx.x / slabs, r1 = rows * (blockIdx.x + 1) / slabs;
#if WGS_BWD_EARLY
    // L2 prefetch of the first step's chunks before waiting for the
    // previous grid (a latency hint only: the loads come after the wait)
    if (active) {
        prefetch_l2(bias + cv);
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t r = r0 + g + static_cast<int64_t>(q) * groups;
            if (r < r1) {
                prefetch_l2(gy + r * row_chunks + cv);
                prefetch_l2(x + r * row_chunks + cv);
            }
        }
    }
#endif
    pdl_prologue();
    float2 acc[kN / 2];
#pragma unroll
    for (int e = 0; e < kN / 2; ++e) acc[e] = make_float2(0.f, 0.f);
    if (active) {
        const uint4 bv = __ldg(bias + cv);
        const int64_t G = groups;
        const int64_t step = G * row_chunks;  // chunks between a thread's rows
        int64_t off = (r0 + g) * row_chunks + cv;
        auto fetch = [&](int64_t r, int64_t o, uint4 *gyv, uint4 *xv) {
#pragma unroll
            for (int q = 0; q < R; ++q) {
                if (r + q * G < r1) {
                    gyv[q] = ld_stream(gy + o + q * step);
                    xv[q] = ld_stream(x + o + q * step);
                }
            }
        };
        // the next R rows load while these R compute
        uint4 ngy[R], nx[R];
        fetch(r0 + g, off, ngy, nx);
        for (int64_t r = r0 + g; r < r1; r += R * G, off += R * step) {
            uint4 gyv[R], xv[R];
#pragma unroll
            for (int q = 0; q < R; ++q) {
                gyv[q] = ngy[q];
                xv[q] = nx[q];
            }
            fetch(r + R * G, off + R * step, ngy, nx);
#pragma unroll
            for (int q = 0; q < R; ++q) {
                if (r + q * G < r1)
                    st_stream(gx + off + q * step, grad_chunk<E, k16>(gyv[q], xv[q], bv, acc));
            }
        }
    }
    // combine the row groups in a fixed order
    if (g < groups)
#pragma unroll
        for (int e = 0; e < kN; ++e) red[(g * cvb + j) * kN + e] = e & 1 ? acc[e / 2].y : acc[e / 2].x;
    __syncthreads();
    if (g == 0 && cv < row_chunks) {
#pragma unroll
        for (int e = 0; e < kN; ++e) {
            float s = red[j * kN + e];
            for (int q = 1; q < groups; ++q) s += red[(q * cvb + j) * kN + e];
            partial[static_cast<int64_t>(blockIdx.x) * width + cv * kN + e] = s;
        }
    }
}

// Pass 1 for 16-bit data with the next step's chunks staged in shared
// memory: the same rows, columns, arithmetic and summation order as
// gelu_bwd_chunks (so the same bits), but each thread copies its own grad_y
// and x chunks S - 1 steps ahead into its own slots of a ring (cp.async: no
// registers held), reads them back after cp.async.wait_group, and needs no
// barrier until the ring is reused for the row-group sums.  With S = 2 (one
// step ahead, as the register form) the 16-bit kernel no longer spills at
// its 80-register cap: [32760,1536] 54.1 -> 52.2 us on GB300.  Deeper rings
// (S = 3: 54.9 us, S = 4: 56.1), three or four rows a step (53.3, 54.4), one
// row a step (53.3) and a third CTA per SM at a 56-register cap (59.3) were
// slower.  One 768-thread CTA per SM (four row groups over 152 slabs of 216
// rows) beat two 384-thread CTAs (two groups, 304 slabs of 108 rows): 51.1
// against 51.5 us, with half as many partial sums for pass 2; five groups at
// a 64-register cap (960 threads) took 51.9 us (one row a step) or 54.4 (two
// rows a step, spilling).
template <typename E, int R, int S>
__global__ void __launch_bounds__(kMaxThreads, kMinBlocks)
gelu_bwd_chunks_async(const uint4 *gy, const uint4 *x, const uint4 *bias, uint4 *gx,
                      float *partial, int64_t rows, int32_t row_chunks, int32_t width, int32_t cvb,
                      int32_t groups, int32_t slabs) {
    constexpr int kN = 8;
    extern __shared__ uint4 ring[];  // [S][R][2][blockDim]; then float red[groups][cvb][kN]
    const int tid = threadIdx.x, nt = blockDim.x;
    const int j = tid % cvb, g = tid / cvb;
    const int32_t cv = static_cast<int32_t>(blockIdx.y) * cvb + j;
    const bool active = g < groups && cv < row_chunks;
    const int64_t r0 = rows * blockIdx.x / slabs, r1 = rows * (blockIdx.x + 1) / slabs;
    const int64_t first = r0 + g;
#if WGS_BWD_EARLY
    if (active) {
        prefetch_l2(bias + cv);
#pragma unroll
        for (int q = 0; q < R; ++q)
            if (first + q * groups < r1) {
                prefetch_l2(gy + (first + q * groups) * row_chunks + cv);
                prefetch_l2(x + (first + q * groups) * row_chunks + cv);
            }
    }
#endif
    pdl_prologue();
    float2 acc[kN / 2];
#pragma unroll
    for (int e = 0; e < kN / 2; ++e) acc[e] = make_float2(0.f, 0.f);
    if (active) {
        const uint4 bv = __ldg(bias + cv);
        // this thread's rows: first, first + G, ... below r1, R a step
        const int32_t n_rows = first < r1 ? static_cast<int32_t>((r1 - first + groups - 1) / groups) : 0;
        const int32_t steps = (n_rows + R - 1) / R;
        const uint4 *gyp = gy + first * row_chunks + cv;
        const uint4 *xp = x + first * row_chunks + cv;
        uint4 *gxp = gx + first * row_chunks + cv;
        const int64_t rstride = static_cast<int64_t>(groups) * row_chunks;  // chunks between rows
        auto issue = [&](int32_t st) {
            const int slot = static_cast<int>(static_cast<uint32_t>(st) % S);
#pragma unroll
            for (int q = 0; q < R; ++q) {
                const int32_t k = st * R + q;  // the thread's k-th row
                if (st < steps && k < n_rows) {
                    cp_async16(&ring[((slot * R + q) * 2 + 0) * nt + tid], gyp + k * rstride);
                    cp_async16(&ring[((slot * R + q) * 2 + 1) * nt + tid], xp + k * rstride);
                }
            }
            cp_async_commit();
        };
#pragma unroll
        for (int st = 0; st < S - 1; ++st) issue(st);
        for (int32_t st = 0; st < steps; ++st) {
            issue(st + S - 1);
            cp_async_wait<S - 1>();  // step st's copies have landed
            const int slot = static_cast<int>(static_cast<uint32_t>(st) % S);
#pragma unroll
            for (int q = 0; q < R; ++q) {
                const int32_t k = st * R + q;
                if (k < n_rows) {
                    const uint4 gyv = ring[((slot * R + q) * 2 + 0) * nt + tid];
                    const uint4 xv = ring[((slot * R + q) * 2 + 1) * nt + tid];
                    st_stream(gxp + k * rstride, grad_chunk<E, true>(gyv, xv, bv, acc));
                }
            }
        }
        cp_async_wait<0>();
    }
    __syncthreads();  // the ring is free: reuse it for the row-group sums
    float *red = reinterpret_cast<float *>(ring);
    if (g < groups)
#pragma unroll
        for (int e = 0; e < kN; ++e) red[(g * cvb + j) * kN + e] = e & 1 ? acc[e / 2].y : acc[e / 2].x;
    __syncthreads();
    if (g == 0 && cv < row_chunks) {
#pragma unroll
        for (int e = 0; e < kN; ++e) {
            float v = red[j * kN + e];
            for (int q = 1; q < groups; ++q) v += red[(q * cvb + j) * kN + e];
            partial[static_cast<int64_t>(blockIdx.x) * width + cv * kN + e] = v;
        }
    }
}

// Pass 1, any width / alignment: thread (g, j) owns column blockIdx.y*CVB + j.
template <typename E>
__global__ void __launch_bounds__(kMaxThreads, kMinBlocks)
gelu_bwd_scalar(const void *gyp, const void *xp, const void *bp, void *gxp, float *partial,
                int64_t rows, int32_t width, int32_t cvb, int32_t groups, int32_t slabs) {
    pdl_prologue();
    constexpr bool k16 = !std::is_same<E, F32>::value;
    extern __shared__ float red[];  // [groups][cvb]
    const int j = threadIdx.x % cvb, g = threadIdx.x / cvb;
    const int32_t c = static_cast<int32_t>(blockIdx.y) * cvb + j;
    const bool active = g < groups && c < width;
    const int64_t r0 = rows * blockIdx.x / slabs, r1 = rows * (blockIdx.x + 1) / slabs;
    float acc = 0.f;
    if (active) {
        for (int64_t r = r0 + g; r < r1; r += groups) {
            const int64_t i = r * width + c;
            if constexpr (k16) {
                const uint16_t *gy = static_cast<const uint16_t *>(gyp);
                const uint16_t *x = static_cast<const uint16_t *>(xp);
                const uint16_t *b = static_cast<const uint16_t *>(bp);
                const float t = E::to_f2(E::add2(x[i], b[c])).x;
                const uint16_t o = static_cast<uint16_t>(E::from_f2(E::to_f2(gy[i]).x * gelu_grad(t), 0.f));
                static_cast<uint16_t *>(gxp)[i] = o;
                acc += E::to_f2(o).x;
            } else {
                const float *gy = static_cast<const float *>(gyp);
                const float *x = static_cast<const float *>(xp);
                const float *b = static_cast<const float *>(bp);
                const float v = gy[i] * gelu_grad(x[i] + b[c]);
                static_cast<float *>(gxp)[i] = v;
                acc += v;
            }
        }
    }
    if (g < groups) red[g * cvb + j] = acc;
    __syncthreads();
    if (g == 0 && c < width) {
        float s = red[j];
        for (int q = 1; q < groups; ++q) s += red[q * cvb + j];
        partial[static_cast<int64_t>(blockIdx.x) * width + c] = s;
    }
}

// Pass 2: grad_bias[c] = round(sum over slabs of partial[slab][c]).  A CTA
// takes 32 columns; its 32 slab lanes (one warp each, reading 32
// consecutive columns of a slab) each sum slabs k, k + 32, ... in order,
// up to 16 loads in flight at any slab count, then the lane sums combine in
// lane order.  The order is fixed, so the result is deterministic.
//
// Unlike the other kernels, it lets the next grid launch before its own
// wait.  That is safe: the next grid's griddepcontrol.wait still waits for
// this grid to complete, and this grid reads nothing before its own wait.
// Pass 2 is short and starts only as pass 1 ends, so releasing the next
// grid after the wait left that grid's launch and first-row prefetches
// outside any overlap: [32760,1536] 52.2 -> 51.5 us, [131040,768] 182.6 ->
// 181.7 us.  (Every kernel of the library signalling first measured the
// same elsewhere.)
constexpr int kBiasCols = 32, kBiasLanes = 32, kBiasUnroll = 16;

template <typename E>
__global__ void __launch_bounds__(kBiasCols * kBiasLanes)
gelu_bwd_bias(const float *partial, void *grad_bias, int32_t width, int32_t slabs) {
#if WGS_PDL
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
    __shared__ float red[kBiasLanes][kBiasCols];
    const int col = threadIdx.x % kBiasCols, lane = threadIdx.x / kBiasCols;
    const int32_t c = static_cast<int32_t>(blockIdx.x) * kBiasCols + col;
    float s = 0.f;
    if (c < width) {
        // up to kBiasUnroll loads in flight, added in slab order
        for (int32_t q = lane; q < slabs; q += kBiasUnroll * kBiasLanes) {
            float v[kBiasUnroll];
#pragma unroll
            for (int u = 0; u < kBiasUnroll; ++u) {
                const int32_t k = q + u * kBiasLanes;
                v[u] = k < slabs ? __ldcg(partial + static_cast<int64_t>(k) * width + c) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kBiasUnroll; ++u)
                if (q + u * kBiasLanes < slabs) s += v[u];
        }
    }
    red[lane][col] = s;
    __syncthreads();
    if (lane == 0 && c < width) {
        float t = red[0][col];
        for (int k = 1; k < kBiasLanes; ++k) t += red[k][col];
        if constexpr (std::is_same<E, F32>::value)
            static_cast<float *>(grad_bias)[c] = t;
        else
            static_cast<uint16_t *>(grad_bias)[c] = static_cast<uint16_t>(E::from_f2(t, 0.f));
    }
}

int64_t slabs_for(int64_t rows) {
    int64_t s = ceil_div(rows, kMinRowsPerSlab);
    return s < 1 ? 1 : (s > kMaxSlabs ? kMaxSlabs : s);
}

template <typename E>
wgs_status launch_bwd(const void *gy, const void *x, const void *bias, void *gx, void *gb,
                      float *partial, int64_t rows, int32_t width, int device,
                      cudaStream_t stream) {
    constexpr bool k16 = !std::is_same<E, F32>::value;
    constexpr int kVec = k16 ? 8 : 4;
    const int32_t slabs = static_cast<int32_t>(slabs_for(rows));
    const bool chunks = width % kVec == 0 && aligned16(gy) && aligned16(x) && aligned16(bias) &&
                        aligned16(gx);
    const int32_t units = chunks ? width / kVec : width;        // column units per row
    const int32_t cvb = units < kMaxChunksPerBlock ? units : kMaxChunksPerBlock;
    const int64_t col_blocks = ceil_div(units, cvb);
    // Row groups: enough threads to cover the GPU's memory latency, chosen
    // from the shape alone (the summation order depends on it).
    int64_t groups64 = WGS_BWD_TARGET_THREADS / (static_cast<int64_t>(slabs) * col_blocks * cvb);
    if (groups64 > WGS_BWD_GROUPS) groups64 = WGS_BWD_GROUPS;
    if (groups64 > kMaxThreads / cvb) groups64 = kMaxThreads / cvb;
    const int32_t groups = groups64 < 1 ? 1 : static_cast<int32_t>(groups64);
    const dim3 grid(static_cast<unsigned>(slabs), static_cast<unsigned>(col_blocks));
    const dim3 block(static_cast<unsigned>(cvb * groups));
    wgs_status st;
    bool staged = false;
    if constexpr (k16 && WGS_BWD_ASYNC) {
        if (chunks) {
            staged = true;
            constexpr int R = WGS_BWD_ROWS, S = WGS_BWD_ASYNC_STAGES;
            auto kernel = gelu_bwd_chunks_async<E, R, S>;
            const size_t ring = static_cast<size_t>(S) * R * 2 * block.x * sizeof(uint4);
            const size_t red = static_cast<size_t>(groups) * cvb * kVec * sizeof(float);
            const size_t smem = ring > red ? ring : red;
            // Shared memory above 48 KB needs an opt-in (two slots of two
            // rows at 768 threads take 96 KB).  The opt-in belongs to the
            // context the kernel is loaded in, so the per-device record only
            // saves the call: a launch the runtime rejects for want of it (in
            // a new context on the device, e.g. after a reset) raises the
            // limit there and is retried once.
            static std::atomic<size_t> opted[64];
            auto opt_in = [&]() {
                if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem)) != cudaSuccess) {
                    cudaGetLastError();
                    return false;
                }
                opted[device].store(smem, std::memory_order_relaxed);
                return true;
            };
            const bool big = smem > 48 * 1024;
            if (big && opted[device].load(std::memory_order_relaxed) < smem && !opt_in())
                return WGS_ERR_LAUNCH;
            auto go = [&]() {
                return launch(kernel, grid, block, smem, stream, static_cast<const uint4 *>(gy),
                              static_cast<const uint4 *>(x), static_cast<const uint4 *>(bias),
                              static_cast<uint4 *>(gx), partial, rows, units, width, cvb, groups,
                              slabs);
            };
            st = go();
            if (st == WGS_ERR_LAUNCH && big && opt_in()) st = go();
        }
    }
    if (staged) {
        // pass 1 is launched
    } else if (chunks) {
        const size_t smem = static_cast<size_t>(groups) * cvb * kVec * sizeof(float);
        st = launch(gelu_bwd_chunks<E, WGS_BWD_ROWS>, grid, block, smem, stream,
                    static_cast<const uint4 *>(gy), static_cast<const uint4 *>(x),
                    static_cast<const uint4 *>(bias), static_cast<uint4 *>(gx), partial, rows,
                    units, width, cvb, groups, slabs);
    } else {
        const size_t smem = static_cast<size_t>(groups) * cvb * sizeof(float);
        st = launch(gelu_bwd_scalar<E>, grid, block, smem, stream, gy, x, bias, gx, partial, rows,
                    width, cvb, groups, slabs);
    }
    if (st != WGS_OK) return st;
    return launch(gelu_bwd_bias<E>, dim3(static_cast<unsigned>(ceil_div(width, kBiasCols))),
                  dim3(kBiasCols * kBiasLanes), 0, stream, static_cast<const float *>(partial), gb,
                  width, slabs);
}

}  // namespace

// Zero rows still take one slab: pass 2 then writes grad_bias = 0.
size_t bwd_workspace_bytes(int64_t rows, int32_t width) {
    if (width <= 0) return 0;
    return static_cast<size_t>(slabs_for(rows > 0 ? rows : 1)) * static_cast<size_t>(width) *
           sizeof(float);
}

wgs_status bias_gelu_bwd_checked(const void *grad_y, const void *x, const void *bias,
                                 void *grad_x, void *grad_bias, float *partial, int64_t rows,
                                 int32_t width, wgs_dtype dtype, cudaStream_t stream) {
    DeviceInfo dev;
    const wgs_status st = current_device(&dev);
    if (st != WGS_OK) return st;
    switch (dtype) {
        case WGS_F16:
            return launch_bwd<Fp16>(grad_y, x, bias, grad_x, grad_bias, partial, rows, width,
                                    dev.device, stream);
        case WGS_BF16:
            return launch_bwd<Bf16>(grad_y, x, bias, grad_x, grad_bias, partial, rows, width,
                                    dev.device, stream);
        default:
            return launch_bwd<F32>(grad_y, x, bias, grad_x, grad_bias, partial, rows, width,
                                   dev.device, stream);
    }
}

// Argument checks shared by the entry points.
wgs_status bias_gelu_bwd_args(const void *grad_y, const void *x, const void *bias, void *grad_x,
                              void *grad_bias, int64_t rows, int32_t width, wgs_dtype dtype) {
    if (dtype != WGS_F32 && dtype != WGS_F16 && dtype != WGS_BF16) return WGS_ERR_DTYPE;
    if (rows < 0 || width < 0) return WGS_ERR_SHAPE;
    const int64_t esz = dtype == WGS_F32 ? 4 : 2;
    if (width > 0 && rows > INT64_MAX / esz / width) return WGS_ERR_SHAPE;
    if (width == 0) return WGS_OK;
    if (!bias || !grad_bias) return WGS_ERR_NULL;
    if (rows > 0 && (!grad_y || !x || !grad_x)) return WGS_ERR_NULL;
    const uintptr_t mask = static_cast<uintptr_t>(esz - 1);
    if ((reinterpret_cast<uintptr_t>(grad_y) | reinterpret_cast<uintptr_t>(x) |
         reinterpret_cast<uintptr_t>(bias) | reinterpret_cast<uintptr_t>(grad_x) |
         reinterpret_cast<uintptr_t>(grad_bias)) & mask)
        return WGS_ERR_ALIGN;
    const int64_t bytes = rows * width * esz, bbytes = width * esz;
    if (!same_or_disjoint(grad_x, grad_y, bytes) || overlap(grad_x, bytes, x, bytes) ||
        overlap(grad_x, bytes, bias, bbytes) || overlap(grad_bias, bbytes, grad_y, bytes) ||
        overlap(grad_bias, bbytes, x, bytes) || overlap(grad_bias, bbytes, grad_x, bytes) ||
        overlap(grad_bias, bbytes, bias, bbytes))
        return WGS_ERR_ALIAS;
    return WGS_OK;
}

}  // namespace wgs

using namespace wgs;

extern "C" size_t wgs_bias_gelu_bwd_workspace_bytes(int64_t rows, int32_t width) {
    return bwd_workspace_bytes(rows, width);
}

extern "C" wgs_status bias_gelu_tanh_bwd(const void *grad_y, const void *x, const void *bias,
                                         void *grad_x, void *grad_bias, void *workspace,
                                         size_t workspace_bytes, int64_t rows, int32_t width,
                                         wgs_dtype dtype, cudaStream_t stream) {
    wgs_status st = bias_gelu_bwd_args(grad_y, x, bias, grad_x, grad_bias, rows, width, dtype);
    if (st != WGS_OK || width == 0) return st;
    const size_t need = bwd_workspace_bytes(rows, width);
    if (!workspace) return WGS_ERR_NULL;
    if (workspace_bytes < need) return WGS_ERR_SHAPE;
    if (!aligned16(workspace)) return WGS_ERR_ALIGN;
    const int64_t esz = dtype == WGS_F32 ? 4 : 2;
    const int64_t bytes = rows * width * esz;
    if (overlap(workspace, static_cast<int64_t>(need), grad_y, bytes) ||
        overlap(workspace, static_cast<int64_t>(need), x, bytes) ||
        overlap(workspace, static_cast<int64_t>(need), grad_x, bytes) ||
        overlap(workspace, static_cast<int64_t>(need), bias, width * esz) ||
        overlap(workspace, static_cast<int64_t>(need), grad_bias, width * esz))
        return WGS_ERR_ALIAS;
    return bias_gelu_bwd_checked(grad_y, x, bias, grad_x, grad_bias, static_cast<float *>(workspace),
                                 rows, width, dtype, stream);
}

// ---------------------------------------------------------------------
// The same backward without a caller workspace.
//
// Some callers cannot hand this library device memory: an op embedded in a
// host runtime that owns every allocation and offers its plugins neither an
// allocator nor a workspace argument, or a hot path that must not call
// cudaMalloc because that call can synchronise the whole device.  For
// them the partial column sums live in a fixed array compiled into the
// library.  Every GPU that loads the library holds the array until the
// process exits, and all calls on that GPU share it.
// ---------------------------------------------------------------------

namespace {

constexpr size_t kNoAllocScratchFloats = size_t{5} << 18;  // 5 MiB per device

static __device__ __align__(256) float g_bwd_scratch[kNoAllocScratchFloats];

// Host code cannot use g_bwd_scratch as a pointer (on the host it names a
// stand-in object, not device memory), so its device address is looked up
// with cudaGetSymbolAddress, in the context current on the calling thread.
// The lookup runs on every call: it is a host-side table lookup that
// allocates nothing, and an address kept from an earlier call could name
// memory of a context that no longer exists (after cudaDeviceReset) or is
// not current (another context on the same device).  The first lookup in a
// context also loads this library's device code there.
wgs_status scratch_address(float **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) {
        cudaGetLastError();  // clear this thread's error
        return WGS_ERR_CUDA;
    }
    *out = static_cast<float *>(p);
    return WGS_OK;
}

}  // namespace

extern "C" wgs_status bias_gelu_tanh_bwd_noalloc(const void *grad_y, const void *x,
                                                 const void *bias, void *grad_x, void *grad_bias,
                                                 int64_t rows, int32_t width, wgs_dtype dtype,
                                                 cudaStream_t stream) {
    const wgs_status st = bias_gelu_bwd_args(grad_y, x, bias, grad_x, grad_bias, rows, width, dtype);
    if (st != WGS_OK || width == 0) return st;
    if (bwd_workspace_bytes(rows, width) > kNoAllocScratchFloats * sizeof(float))
        return WGS_ERR_TOO_LARGE;
    DeviceInfo dev;
    const wgs_status ds = current_device(&dev);
    if (ds != WGS_OK) return ds;
    float *scratch = nullptr;
    const wgs_status ss = scratch_address(&scratch);
    if (ss != WGS_OK) return ss;
    // Pass 1 writes every partial sum that pass 2 reads, in stream order, so
    // nothing in the array needs clearing between calls.
    return bias_gelu_bwd_checked(grad_y, x, bias, grad_x, grad_bias, scratch, rows, width, dtype,
                                 stream);
}
