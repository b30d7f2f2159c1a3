// Shared host and device helpers of the sm_103a block-glue kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <utility>

#include "wgs.h"

#ifndef WGS_PDL
#define WGS_PDL 1  // launch with programmatic dependent launch
#endif

namespace wgs {

// ------------------------------------------------------------ host side --

// Streaming multiprocessors of the current device (cached per device), or
// a negative value on failure.  Also fails unless the device is compute
// capability 10.3, the only target these kernels are built for.
struct DeviceInfo {
    int device;
    int sm_count;
};
wgs_status current_device(DeviceInfo *info);

// Enqueue on `stream` a copy of the bias-mask add's error word into *seen
// and its reset to zero (for wgs_check_error; the caller synchronises).
wgs_status bias_mask_error_take(unsigned int *seen, cudaStream_t stream);

// Launch `kernel` on `stream`.  With WGS_PDL the launch allows programmatic
// dependent launch: the grid may be scheduled while the previous kernel on
// the stream drains, and every kernel of this library starts with
// pdl_prologue(), whose griddepcontrol.wait holds it until the previous
// grid has completed and its writes are visible.  Kernels that do not use
// these controls (other libraries') keep the usual full serialisation.
template <typename... Params, typename... Args>
wgs_status launch(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                  cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = WGS_PDL ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) != cudaSuccess) {
        cudaGetLastError();  // clear this thread's launch error
        return WGS_ERR_LAUNCH;
    }
    return WGS_OK;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// True when [a, a + na) and [b, b + nb) share a byte.
inline bool overlap(const void *a, int64_t na, const void *b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + static_cast<uintptr_t>(nb) &&
           y < x + static_cast<uintptr_t>(na);
}

// Same buffer exactly, or no shared byte at all.
inline bool same_or_disjoint(const void *a, const void *b, int64_t n) {
    return a == b || !overlap(a, n, b, n);
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------- device side --

// First statement of every kernel: wait until the grid launched before this
// one on the stream has completed (its outputs may be this grid's inputs),
// then let the next grid start its launch.  Both are no-ops for a launch
// without programmatic dependent launch.
__device__ __forceinline__ void pdl_prologue() {
#if WGS_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// Ask L2 to fetch the 128-byte line holding p.  No data reaches the
// thread, so a prefetch issued before griddepcontrol.wait cannot feed a
// result with a stale value: L2 is the coherence point for every SM, and a
// line that the previous grid writes afterwards is updated in L2.  Only a
// latency hint; p must lie inside a live allocation.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// 4-byte global load cached in L2 only (never in the SM's L1), so a value
// read before griddepcontrol.wait leaves no stale copy in L1 for a later
// load of the same address.
__device__ __forceinline__ int32_t ld_cg_i32(const int32_t *p) { return __ldcg(p); }

// 16-byte asynchronous copy global -> shared (cp.async; the executing
// thread reads the slot after cp_async_wait).  cg: cached in L2 only; ca:
// also in L1, for data other CTAs of the SM reread.  Both addresses must be
// 16-byte aligned.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async16_ca(void *smem, const void *gmem) {
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(gmem) : "memory");
}
// Close the group of copies issued since the last commit.
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's committed groups are in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 16-byte global load that skips L1 (each byte is read exactly once).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    return __ldcg(reinterpret_cast<const uint4 *>(p));
}

// 16-byte global store.
__device__ __forceinline__ void st_stream(void *p, const uint4 &v) {
    *reinterpret_cast<uint4 *>(p) = v;
}

__device__ __forceinline__ float2 half2_to_float2(uint32_t bits) {
    __half2 h;
    memcpy(&h, &bits, sizeof(h));
    return __half22float2(h);
}

__device__ __forceinline__ uint32_t float2_to_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);  // round to nearest even
    uint32_t bits;
    memcpy(&bits, &h, sizeof(bits));
    return bits;
}

__device__ __forceinline__ uint32_t word(const uint4 &v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

__device__ __forceinline__ void set_word(uint4 &v, int j, uint32_t w) {
    if (j == 0) v.x = w; else if (j == 1) v.y = w; else if (j == 2) v.z = w; else v.w = w;
}

// 16-bit element formats of the row kernels: two elements per 32-bit word.
// to_f2 widens exactly; widen_add2 widens and adds an FP32 pair (one
// rounding); from_f2 rounds to nearest even; add2 returns
// round(a + b) for each pair with one native add.  For both formats that
// also equals rounding the binary32 sum once more (binary32 carries at
// least 2p + 2 bits for a p-bit format, so the double rounding is
// innocuous), which is how the residual sum is specified.
// (lo + c.x, hi + c.y) for the two 16-bit values of word w, each widened
// exactly and added in FP32 with one rounding: PTX add.rn.f32.f16 / .bf16
// (widen and add in one instruction).
#define WGS_WIDEN_ADD2(FMT)                                                              \
    __device__ static float2 widen_add2(uint32_t w, float2 c) {                        \
        float2 r;                                                                       \
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"                       \
            "add.rn.f32." FMT " %0, lo, %3;\n\tadd.rn.f32." FMT " %1, hi, %4;\n\t}"         \
            : "=f"(r.x), "=f"(r.y)                                                      \
            : "r"(w), "f"(c.x), "f"(c.y));                                              \
        return r;                                                                       \
    }

struct Fp16 {
    WGS_WIDEN_ADD2("f16")
    __device__ static float2 to_f2(uint32_t w) { return half2_to_float2(w); }
    __device__ static uint32_t from_f2(float a, float b) { return float2_to_half2(a, b); }
    __device__ static uint32_t add2(uint32_t a, uint32_t b) {
        __half2 x, y;
        memcpy(&x, &a, 4);
        memcpy(&y, &b, 4);
        const __half2 z = __hadd2(x, y);
        uint32_t r;
        memcpy(&r, &z, 4);
        return r;
    }
};

struct Bf16 {
    WGS_WIDEN_ADD2("bf16")
    __device__ static float2 to_f2(uint32_t w) {
        __nv_bfloat162 h;
        memcpy(&h, &w, 4);
        return __bfloat1622float2(h);
    }
    __device__ static uint32_t from_f2(float a, float b) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        uint32_t r;
        memcpy(&r, &h, 4);
        return r;
    }
    // one correctly rounded bf16x2 add (PTX add.rn.bf16x2, sm_90 and later)
    __device__ static uint32_t add2(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
};

// Sum over the LPR consecutive lanes that share a row (LPR a power of two,
// groups aligned to LPR), by butterfly exchange; every lane of the group
// ends with the total.  All 32 lanes must call it together.
template <int LPR>
__device__ __forceinline__ float group_sum(float s) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

}  // namespace wgs
