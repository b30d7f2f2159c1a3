// Position bias + shift mask added to the pre-softmax attention logits of a
// shifted-window transformer (sm_103a).
//
// Page "BW1000 gfx936 Pangu-Weather inference profiling", s7 keeps a
// "bias-mask" op in the final combination and s6 rejects fusing it with
// softmax; the pages do not give its arithmetic.  The reading here is the
// shifted-window transformer's general one, with the rounding points of an
// eager "attn + bias; attn + mask" sequence in the tensor's format:
//     t   = fp(scores[w,h,i,j] + bias[type[w],h,i,j])
//     out = fp(t + (region[w,i] == region[w,j] ? 0 : m))      (region given)
// The logits tensor is streamed once (read, written); the bias slabs
// (n_types x heads x n x n, a few hundred KB per type) and the region labels
// are re-read by every window and stay in L2 / L1.
//
// Layout: a logits row is n 16-bit elements = n/8 16-byte chunks.  A CTA of
// RP x (n/8) threads gives every thread one fixed chunk column and RP rows
// per pass, U passes in flight.  A CTA takes one unit, a contiguous run of
// rows of one (window, head) tile: a tile's passes are split into the
// fewest parts of at most WGS_BM_PART_PASSES passes, evened out (n = 144,
// RP = 7, U = 2: 11 passes in parts of 56, 56 and 32 rows).
// A unit's window and head come from two
// divisions by invariant integers done as multiply-high (Granlund &
// Montgomery 1994); its window type and column labels are loaded once.
#include "wgs_common.cuh"

#ifndef WGS_BM_EARLY
#define WGS_BM_EARLY 1  // L2 prefetch of the first unit's logits before the wait
#endif
#ifndef WGS_BM_U
#define WGS_BM_U 2  // rows in flight per thread
#endif
#ifndef WGS_BM_PART_PASSES
#define WGS_BM_PART_PASSES 4  // passes of RP x U rows per unit, at most
#endif
#ifndef WGS_BM_STAGED
#define WGS_BM_STAGED 1  // stage a unit's next pass of logits and bias in shared memory
#endif
#ifndef WGS_BM_THREADS
#define WGS_BM_THREADS 128  // threads per CTA to aim for (vector path)
#endif

namespace wgs {

namespace {

// Set (never cleared by a kernel) when a window type lies outside
// [0, n_types); read and cleared by wgs_check_error through
// bias_mask_error_take.  Kernels name it directly, so no device address is
// kept on the host.
__device__ unsigned int g_mask_error;

}  // namespace

// Enqueue on `stream` a copy of the bias-mask error word into *seen and a
// reset of the word to zero; the caller synchronises the stream.
wgs_status bias_mask_error_take(unsigned int *seen, cudaStream_t stream) {
    static const unsigned int cleared = 0;
    if (cudaMemcpyFromSymbolAsync(seen, g_mask_error, sizeof(*seen), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_mask_error, &cleared, sizeof(cleared), 0,
                                cudaMemcpyHostToDevice, stream) != cudaSuccess) {
        cudaGetLastError();  // clear this thread's error
        return WGS_ERR_CUDA;
    }
    return WGS_OK;
}

namespace {

// Vector-path CTAs: RP = max(1, WGS_BM_THREADS / (n/8)) rows of n/8 threads,
// so at most 256 threads for the widest row the path takes (n = 2048).
constexpr int kMaxChunksPerRow = 256;

// x / d for 0 <= x < 2^31 and 1 <= d < 2^31 with one multiply-high
// (Granlund & Montgomery, "Division by invariant integers using
// multiplication", 1994, s4): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, x / d = (mulhi(x, m) + x) >> l.  The
// sum stays below 2^32 because mulhi(x, m) <= x < 2^31.
struct FastDiv {
    uint32_t m, l;
};

FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((uint64_t{1} << l) < d) ++l;
    const uint64_t m = ((uint64_t{1} << 32) * ((uint64_t{1} << l) - d)) / d + 1;
    return {static_cast<uint32_t>(m), l};
}

__device__ __forceinline__ uint32_t div_by(uint32_t x, FastDiv f) {
    return (__umulhi(x, f.m) + x) >> f.l;
}

// The mask term of one 32-bit word (two elements): m in each half whose
// column label differs from the row label, +0 elsewhere.
__device__ __forceinline__ uint32_t mask_word(int32_t row, int32_t c_lo, int32_t c_hi,
                                              uint32_t mask2) {
    return (c_lo != row ? (mask2 & 0xffffu) : 0u) | (c_hi != row ? (mask2 & 0xffff0000u) : 0u);
}

// A unit is one (window, head) tile's rows [part * part_rows, (part + 1) *
// part_rows); the launch gives each CTA one (the loop also serves a smaller
// grid).  A unit's window type, column labels and base addresses are found
// once; its rows then stream with plain offsets in passes of RP x U rows,
// the next pass's logits and bias chunks copied into shared memory
// (cp.async, each thread its own two slots) while this pass computes:
// 73.9 -> 72.9 us at [960,6] and 41.0 -> 40.4 us at [256,12] on GB300
// against loading each pass after the previous one.
template <typename E, int U>
__global__ void __launch_bounds__(kMaxChunksPerRow > WGS_BM_THREADS ? kMaxChunksPerRow : WGS_BM_THREADS)
bias_mask_vec(const uint4 *scores, const uint4 *bias, const int32_t *win_type,
                const int32_t *region, uint4 *out, uint32_t units, int32_t n,
                int32_t heads, int32_t n_types, int32_t cpr, int32_t rp, int32_t part_rows,
                int32_t parts, FastDiv by_parts, FastDiv by_heads, uint32_t mask2) {
    const int jc = static_cast<int>(threadIdx.x) % cpr, lr = static_cast<int>(threadIdx.x) / cpr;
#if WGS_BM_EARLY
    // L2 prefetch of the first unit's logits before waiting for the previous
    // grid (a latency hint only: the loads come after the wait)
    if (lr < rp && blockIdx.x < units) {
        const uint32_t tile = div_by(blockIdx.x, by_parts);
        const int32_t part = static_cast<int32_t>(blockIdx.x - tile * static_cast<uint32_t>(parts));
        const int32_t i1 = (part + 1) * part_rows < n ? (part + 1) * part_rows : n;
        const uint4 *sp = scores + static_cast<int64_t>(tile) * n * cpr + jc;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int32_t ii = part * part_rows + lr + u * rp;
            if (ii < i1) prefetch_l2(sp + static_cast<int64_t>(ii) * cpr);
        }
    }
#endif
    pdl_prologue();
    if (lr >= rp) return;
    for (uint32_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const uint32_t tile = div_by(unit, by_parts);
        const int32_t part = static_cast<int32_t>(unit - tile * static_cast<uint32_t>(parts));
        const uint32_t w = div_by(tile, by_heads), h = tile - w * heads;
        const int32_t type = win_type ? __ldg(win_type + w) : 0;
        const bool ok = type >= 0 && type < n_types;
        const int32_t *lab = region + static_cast<int64_t>(w) * n;
        int4 c0 = make_int4(0, 0, 0, 0), c1 = c0;
        if (region) {
            c0 = __ldg(reinterpret_cast<const int4 *>(lab) + 2 * jc);
            c1 = __ldg(reinterpret_cast<const int4 *>(lab) + 2 * jc + 1);
        }
        const int32_t i1 = (part + 1) * part_rows < n ? (part + 1) * part_rows : n;
        const uint4 *sp = scores + static_cast<int64_t>(tile) * n * cpr + jc;
        const uint4 *bp = bias + (static_cast<int64_t>(ok ? type : 0) * heads + h) * n * cpr + jc;
        uint4 *op = out + static_cast<int64_t>(tile) * n * cpr + jc;
#if WGS_BM_STAGED
        // passes of RP x U rows; each thread copies its chunks of the next
        // pass (logits, and the bias unless the type is bad) into its own two
        // ring slots while this pass computes
        extern __shared__ uint4 ring[];  // [2][U][2][blockDim]
        const int tid = static_cast<int>(threadIdx.x), nt = static_cast<int>(blockDim.x);
        const int32_t i0 = part * part_rows + lr;
        const int32_t npass = (i1 - part * part_rows + rp * U - 1) / (rp * U);
        auto issue = [&](int32_t pass) {
            const int slot = pass & 1;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t ii = i0 + pass * rp * U + u * rp;
                if (pass < npass && ii < i1) {
                    cp_async16(&ring[((slot * U + u) * 2 + 0) * nt + tid], sp + static_cast<int64_t>(ii) * cpr);
                    if (ok) cp_async16_ca(&ring[((slot * U + u) * 2 + 1) * nt + tid], bp + static_cast<int64_t>(ii) * cpr);
                }
            }
            cp_async_commit();
        };
        issue(0);
        for (int32_t pass = 0; pass < npass; ++pass) {
            issue(pass + 1);
            cp_async_wait<1>();
            const int slot = pass & 1;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t ii = i0 + pass * rp * U + u * rp;
                if (ii >= i1) continue;
                const uint4 sv = ring[((slot * U + u) * 2 + 0) * nt + tid];
                uint4 o = make_uint4(0u, 0u, 0u, 0u);
                if (ok) {
                    const uint4 bv = ring[((slot * U + u) * 2 + 1) * nt + tid];
                    const int32_t li = region ? __ldg(lab + ii) : 0;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t t = E::add2(word(sv, k), word(bv, k));
                        if (region) {
                            const int4 &c = k < 2 ? c0 : c1;
                            const int32_t lo = (k & 1) ? c.z : c.x, hi = (k & 1) ? c.w : c.y;
                            t = E::add2(t, mask_word(li, lo, hi, mask2));
                        }
                        set_word(o, k, t);
                    }
                } else {
                    atomicOr(&g_mask_error, 1u);
                }
                st_stream(op + static_cast<int64_t>(ii) * cpr, o);
            }
        }
        cp_async_wait<0>();  // the ring is free for the next unit
#else
        for (int32_t i = part * part_rows + lr; i < i1; i += rp * U) {
            uint4 sv[U], bv[U];
            int32_t li[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t ii = i + u * rp;
                if (ii < i1) {
                    sv[u] = ld_stream(sp + static_cast<int64_t>(ii) * cpr);
                    if (ok) bv[u] = __ldg(bp + static_cast<int64_t>(ii) * cpr);
                    if (region) li[u] = __ldg(lab + ii);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t ii = i + u * rp;
                if (ii >= i1) continue;
                uint4 o = make_uint4(0u, 0u, 0u, 0u);
                if (ok) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t t = E::add2(word(sv[u], k), word(bv[u], k));
                        if (region) {
                            const int4 &c = k < 2 ? c0 : c1;
                            const int32_t lo = (k & 1) ? c.z : c.x, hi = (k & 1) ? c.w : c.y;
                            t = E::add2(t, mask_word(li[u], lo, hi, mask2));
                        }
                        set_word(o, k, t);
                    }
                } else {
                    atomicOr(&g_mask_error, 1u);
                }
                st_stream(op + static_cast<int64_t>(ii) * cpr, o);
            }
        }
#endif
    }
}

// Any n or alignment: one element per thread per step.
template <typename E>
__global__ void __launch_bounds__(256)
bias_mask_scalar(const uint16_t *scores, const uint16_t *bias, const int32_t *win_type,
                 const int32_t *region, uint16_t *out, int64_t total, int32_t n,
                 int32_t heads, int32_t n_types, uint32_t mask2) {
    pdl_prologue();
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = e / n, tile = r / n, w = tile / heads;
        const int32_t j = static_cast<int32_t>(e - r * n), i = static_cast<int32_t>(r - tile * n);
        const int32_t h = static_cast<int32_t>(tile - w * heads);
        const int32_t type = win_type ? win_type[w] : 0;
        uint16_t o = 0;
        if (type >= 0 && type < n_types) {
            uint32_t t = E::add2(scores[e], bias[((type * static_cast<int64_t>(heads) + h) * n + i) * n + j]);
            if (region) {
                const int32_t *lab = region + w * n;
                t = E::add2(t, lab[i] != lab[j] ? (mask2 & 0xffffu) : 0u);
            }
            o = static_cast<uint16_t>(t);
        } else {
            atomicOr(&g_mask_error, 1u);
        }
        out[e] = o;
    }
}

template <typename E>
wgs_status launch_bias_mask(const void *scores, const void *bias, const int32_t *win_type,
                            const int32_t *region, void *out, int64_t n_win,
                            int32_t heads, int32_t n, int32_t n_types, uint32_t mask2,
                            const DeviceInfo &dev, cudaStream_t stream) {
    const int64_t rows = n_win * heads * n;
    const int32_t cpr = n / 8;
    const bool vec = n % 8 == 0 && cpr <= kMaxChunksPerRow && aligned16(scores) &&
                     aligned16(bias) && aligned16(out) && (!region || aligned16(region));
    if (vec) {
        constexpr int U = WGS_BM_U;
        const int32_t rp = cpr < WGS_BM_THREADS ? WGS_BM_THREADS / cpr : 1;
        auto kernel = bias_mask_vec<E, U>;
        // the fewest parts of at most WGS_BM_PART_PASSES passes, evened out
        const int32_t passes = static_cast<int32_t>(ceil_div(n, rp * U));
        const int32_t part_passes = static_cast<int32_t>(
            ceil_div(passes, ceil_div(passes, WGS_BM_PART_PASSES)));
        const int32_t part_rows = part_passes * rp * U;
        const int32_t parts = static_cast<int32_t>(ceil_div(n, part_rows));
        const int64_t units = n_win * heads * parts;
        // a CTA per unit: the hardware refills each SM as CTAs finish (one
        // resident wave striding over units left its last round part-empty)
        const size_t smem = WGS_BM_STAGED ? static_cast<size_t>(2) * U * 2 * rp * cpr * sizeof(uint4) : 0;
        return launch(kernel, dim3(static_cast<unsigned>(units)),
                      dim3(static_cast<unsigned>(rp * cpr)), smem, stream,
                      static_cast<const uint4 *>(scores), static_cast<const uint4 *>(bias),
                      win_type, region, static_cast<uint4 *>(out),
                      static_cast<uint32_t>(units), n, heads, n_types, cpr, rp, part_rows, parts,
                      make_fastdiv(static_cast<uint32_t>(parts)),
                      make_fastdiv(static_cast<uint32_t>(heads)), mask2);
    }
    const int64_t total = rows * n;
    const int64_t need = ceil_div(total, 256);
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
    return launch(bias_mask_scalar<E>, dim3(static_cast<unsigned>(need < cap ? need : cap)),
                  dim3(256), 0, stream, static_cast<const uint16_t *>(scores),
                  static_cast<const uint16_t *>(bias), win_type, region,
                  static_cast<uint16_t *>(out), total, n, heads, n_types, mask2);
}

}  // namespace

}  // namespace wgs

using namespace wgs;

extern "C" wgs_status window_bias_mask_add(const void *scores, const void *bias,
                                           const int32_t *win_type, const int32_t *region,
                                           void *out, int64_t n_win, int32_t heads, int32_t n,
                                           int32_t n_types, float mask_value, wgs_dtype dtype,
                                           cudaStream_t stream) {
    if (dtype != WGS_F16 && dtype != WGS_BF16) return WGS_ERR_DTYPE;
    if (n_win < 0 || heads < 0 || n < 0 || n_types < 0) return WGS_ERR_SHAPE;
    if (n_win == 0 || heads == 0 || n == 0) return WGS_OK;
    if (n_types < 1) return WGS_ERR_SHAPE;
    if (n_win > (int64_t{1} << 31) / heads / n ||
        n_win * heads * n >= (int64_t{1} << 31))
        return WGS_ERR_SHAPE;
    if (!scores || !bias || !out) return WGS_ERR_NULL;
    if (((reinterpret_cast<uintptr_t>(scores) | reinterpret_cast<uintptr_t>(bias) |
          reinterpret_cast<uintptr_t>(out)) & 1u) ||
        !aligned4(win_type) || !aligned4(region))
        return WGS_ERR_ALIGN;
    const int64_t nn = static_cast<int64_t>(n) * n;
    const int64_t bytes = n_win * heads * nn * 2, bbytes = static_cast<int64_t>(n_types) * heads * nn * 2;
    if (!same_or_disjoint(out, scores, bytes) || overlap(out, bytes, bias, bbytes) ||
        (win_type && overlap(out, bytes, win_type, n_win * 4)) ||
        (region && overlap(out, bytes, region, n_win * n * 4)))
        return WGS_ERR_ALIAS;
    DeviceInfo dev;
    wgs_status st = current_device(&dev);
    if (st != WGS_OK) return st;
    // the mask value rounded once to the tensor's format, in both halves
    uint16_t m16;
    if (dtype == WGS_F16) {
        const __half h = __float2half_rn(mask_value);
        memcpy(&m16, &h, 2);
    } else {
        const __nv_bfloat16 h = __float2bfloat16_rn(mask_value);
        memcpy(&m16, &h, 2);
    }
    const uint32_t mask2 = static_cast<uint32_t>(m16) | (static_cast<uint32_t>(m16) << 16);
    if (dtype == WGS_F16)
        return launch_bias_mask<Fp16>(scores, bias, win_type, region, out, n_win, heads, n,
                                      n_types, mask2, dev, stream);
    return launch_bias_mask<Bf16>(scores, bias, win_type, region, out, n_win, heads, n,
                                  n_types, mask2, dev, stream);
}
