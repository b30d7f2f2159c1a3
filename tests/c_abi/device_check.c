/*
 * The library driven from plain C99 on a GPU: device buffers from
 * cudaMalloc, work on a stream the program creates, results read back
 * with cudaMemcpy.  No Python is involved.  Checks, each against a value
 * fixed by the definition of the op:
 *   - window_gather through the map of a padded 3 x 11 x 20 grid: every
 *     source row carries its own number in every element, so each
 *     destination row must hold the number its index names, and pad rows
 *     must be all-zero bits;
 *   - ln_fwd of rows of alternating +1 / -1: the mean is 0 and the variance
 *     1, so y = +-1 / sqrt(1 + 1e-5), which rounds to exactly +-1.0 in fp16;
 *   - bias_gelu_tanh in fp32 at t = 0 (gives 0) and at t = 30 (gives 30:
 *     tanh saturates to 1 in binary32);
 *   - bias_gelu_tanh_bwd_noalloc gives the same bits as bias_gelu_tanh_bwd
 *     with a caller workspace;
 *   - an index outside [-1, n_src) makes wgs_check_error report
 *     WGS_ERR_INDEX, and the next check reports WGS_OK;
 *   - after cudaDeviceReset the fp16 backward (with and without a
 *     workspace) gives the bits it gave before the reset.
 * Prints "device ok" and exits 0, or names the first failed check and
 * exits 1 (2 when no usable device is present).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "wgs.h"

static int fails = 0;
#define CHECK(cond)                                                           \
    do {                                                                      \
        if (!(cond)) {                                                        \
            fprintf(stderr, "check failed (line %d): %s\n", __LINE__, #cond); \
            ++fails;                                                          \
        }                                                                     \
    } while (0)
#define CUDA(call)                                                            \
    do {                                                                      \
        if ((call) != cudaSuccess) {                                          \
            fprintf(stderr, "CUDA call failed (line %d): %s\n", __LINE__, #call); \
            return 1;                                                         \
        }                                                                     \
    } while (0)

enum { W = 192 };

/* The fp16 backward at [rows, width] through both entry points, on buffers
 * and a stream made here and released before returning.  Returns 0, or 1
 * when a CUDA call failed. */
static int bwd16(int64_t rows, int32_t width, const uint16_t *gy, const uint16_t *x,
                 const uint16_t *b, uint16_t *gx_ws, uint16_t *gb_ws, uint16_t *gx_na,
                 uint16_t *gb_na, wgs_status *st_ws, wgs_status *st_na) {
    const size_t n = (size_t)(rows * width) * 2, nb = (size_t)width * 2;
    const size_t ws = wgs_bias_gelu_bwd_workspace_bytes(rows, width);
    cudaStream_t s;
    void *d_gy, *d_x, *d_b, *d_gx, *d_gb, *d_ws;
    CUDA(cudaStreamCreate(&s));
    CUDA(cudaMalloc(&d_gy, n));
    CUDA(cudaMalloc(&d_x, n));
    CUDA(cudaMalloc(&d_b, nb));
    CUDA(cudaMalloc(&d_gx, n));
    CUDA(cudaMalloc(&d_gb, nb));
    CUDA(cudaMalloc(&d_ws, ws));
    CUDA(cudaMemcpy(d_gy, gy, n, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_x, x, n, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_b, b, nb, cudaMemcpyHostToDevice));
    *st_ws = bias_gelu_tanh_bwd(d_gy, d_x, d_b, d_gx, d_gb, d_ws, ws, rows, width, WGS_F16, s);
    CUDA(cudaStreamSynchronize(s));
    CUDA(cudaMemcpy(gx_ws, d_gx, n, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(gb_ws, d_gb, nb, cudaMemcpyDeviceToHost));
    CUDA(cudaMemset(d_gx, 0xFF, n));
    CUDA(cudaMemset(d_gb, 0xFF, nb));
    *st_na = bias_gelu_tanh_bwd_noalloc(d_gy, d_x, d_b, d_gx, d_gb, rows, width, WGS_F16, s);
    CUDA(cudaStreamSynchronize(s));
    CUDA(cudaMemcpy(gx_na, d_gx, n, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(gb_na, d_gb, nb, cudaMemcpyDeviceToHost));
    cudaFree(d_gy); cudaFree(d_x); cudaFree(d_b); cudaFree(d_gx); cudaFree(d_gb); cudaFree(d_ws);
    cudaStreamDestroy(s);
    return 0;
}

/* A binary16 value in [2^-4, 4) with a random sign and significand. */
static uint16_t rand_half(void) {
    const unsigned sign = (unsigned)(rand() & 1), ex = 11u + (unsigned)(rand() % 6);
    return (uint16_t)((sign << 15) | (ex << 10) | (unsigned)(rand() & 0x3FF));
}

int main(void) {
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count < 1) {
        fprintf(stderr, "no CUDA device\n");
        return 2;
    }
    cudaStream_t s;
    CUDA(cudaStreamCreate(&s));

    /* ---- window_gather over the padded tiny grid ---- */
    const int32_t grid[3] = {3, 11, 20}, win[3] = {2, 6, 12}, shift[3] = {1, 3, 6};
    const int64_t n_src = 3 * 11 * 20;
    const int64_t n_idx = wgs_window_index_count(grid, win, NULL);
    CHECK(n_idx == 4 * 12 * 24);
    int32_t *idx = (int32_t *)malloc((size_t)n_idx * sizeof(int32_t));
    uint16_t *src = (uint16_t *)malloc((size_t)(n_src * W) * 2);
    uint16_t *dst = (uint16_t *)malloc((size_t)(n_idx * W) * 2);
    if (!idx || !src || !dst) return 1;
    CHECK(wgs_build_window_index(grid, win, shift, NULL, WGS_SHIFT_THEN_PAD, idx, n_idx) == WGS_OK);
    for (int64_t r = 0; r < n_src; ++r)
        for (int c = 0; c < W; ++c) src[r * W + c] = (uint16_t)(r + 1); /* never 0 */
    void *d_src, *d_dst, *d_idx;
    CUDA(cudaMalloc(&d_src, (size_t)(n_src * W) * 2));
    CUDA(cudaMalloc(&d_dst, (size_t)(n_idx * W) * 2));
    CUDA(cudaMalloc(&d_idx, (size_t)n_idx * sizeof(int32_t)));
    CUDA(cudaMemcpy(d_src, src, (size_t)(n_src * W) * 2, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_idx, idx, (size_t)n_idx * sizeof(int32_t), cudaMemcpyHostToDevice));
    CHECK(window_gather(d_src, (const int32_t *)d_idx, d_dst, n_src, n_idx, W, s) == WGS_OK);
    CUDA(cudaStreamSynchronize(s));
    CUDA(cudaMemcpy(dst, d_dst, (size_t)(n_idx * W) * 2, cudaMemcpyDeviceToHost));
    int64_t pads = 0, bad_rows = 0;
    for (int64_t d = 0; d < n_idx; ++d) {
        const uint16_t want = idx[d] < 0 ? 0 : (uint16_t)(idx[d] + 1);
        pads += idx[d] < 0;
        for (int c = 0; c < W; ++c)
            if (dst[d * W + c] != want) {
                ++bad_rows;
                break;
            }
    }
    CHECK(pads == n_idx - n_src);
    CHECK(bad_rows == 0);
    CHECK(wgs_check_error(s) == WGS_OK);

    /* ---- ln_fwd of alternating rows: exactly +-1.0 ---- */
    const int64_t rows = 37;
    uint16_t *x = (uint16_t *)malloc((size_t)(rows * W) * 2);
    uint16_t *y = (uint16_t *)malloc((size_t)(rows * W) * 2);
    if (!x || !y) return 1;
    for (int64_t i = 0; i < rows * W; ++i) x[i] = (i & 1) ? 0xBC00u : 0x3C00u; /* -1, +1 */
    void *d_x, *d_y;
    CUDA(cudaMalloc(&d_x, (size_t)(rows * W) * 2));
    CUDA(cudaMalloc(&d_y, (size_t)(rows * W) * 2));
    CUDA(cudaMemcpy(d_x, x, (size_t)(rows * W) * 2, cudaMemcpyHostToDevice));
    CHECK(ln_fwd(d_x, d_y, rows, W, 1e-5f, s) == WGS_OK);
    CUDA(cudaStreamSynchronize(s));
    CUDA(cudaMemcpy(y, d_y, (size_t)(rows * W) * 2, cudaMemcpyDeviceToHost));
    CHECK(memcmp(x, y, (size_t)(rows * W) * 2) == 0);

    /* ---- bias_gelu_tanh fp32 at closed-form points ---- */
    float gx_in[8] = {0.f, 0.f, 30.f, 30.f, 0.f, 0.f, 30.f, 30.f};
    float gb_in[4] = {0.f, 0.f, 0.f, 0.f}, gy_out[8];
    void *d_gx, *d_gb, *d_gy;
    CUDA(cudaMalloc(&d_gx, sizeof gx_in));
    CUDA(cudaMalloc(&d_gb, sizeof gb_in));
    CUDA(cudaMalloc(&d_gy, sizeof gy_out));
    CUDA(cudaMemcpy(d_gx, gx_in, sizeof gx_in, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_gb, gb_in, sizeof gb_in, cudaMemcpyHostToDevice));
    CHECK(bias_gelu_tanh(d_gx, d_gb, d_gy, 2, 4, WGS_F32, s) == WGS_OK);
    CUDA(cudaStreamSynchronize(s));
    CUDA(cudaMemcpy(gy_out, d_gy, sizeof gy_out, cudaMemcpyDeviceToHost));
    for (int i = 0; i < 8; ++i) CHECK(gy_out[i] == gx_in[i]);

    /* ---- the backward without a workspace equals the one with it ---- */
    const int64_t br = 300;
    const int32_t bw = 768;
    float *bx = (float *)malloc((size_t)(br * bw) * 4), *bg = (float *)malloc((size_t)(br * bw) * 4);
    float *bb = (float *)malloc((size_t)bw * 4);
    float *o1 = (float *)malloc((size_t)(br * bw) * 4), *o2 = (float *)malloc((size_t)(br * bw) * 4);
    float gb1[768], gb2[768];
    if (!bx || !bg || !bb || !o1 || !o2) return 1;
    srand(7);
    for (int64_t i = 0; i < br * bw; ++i) {
        bx[i] = (float)(rand() % 2001 - 1000) / 250.0f;
        bg[i] = (float)(rand() % 2001 - 1000) / 1000.0f;
    }
    for (int i = 0; i < bw; ++i) bb[i] = (float)(rand() % 201 - 100) / 5000.0f;
    void *d_bx, *d_bg, *d_bb, *d_o, *d_gbias, *d_ws;
    const size_t ws = wgs_bias_gelu_bwd_workspace_bytes(br, bw);
    CUDA(cudaMalloc(&d_bx, (size_t)(br * bw) * 4));
    CUDA(cudaMalloc(&d_bg, (size_t)(br * bw) * 4));
    CUDA(cudaMalloc(&d_bb, (size_t)bw * 4));
    CUDA(cudaMalloc(&d_o, (size_t)(br * bw) * 4));
    CUDA(cudaMalloc(&d_gbias, (size_t)bw * 4));
    CUDA(cudaMalloc(&d_ws, ws));
    CUDA(cudaMemcpy(d_bx, bx, (size_t)(br * bw) * 4, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_bg, bg, (size_t)(br * bw) * 4, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_bb, bb, (size_t)bw * 4, cudaMemcpyHostToDevice));
    CHECK(bias_gelu_tanh_bwd(d_bg, d_bx, d_bb, d_o, d_gbias, d_ws, ws, br, bw, WGS_F32, s) == WGS_OK);
    CUDA(cudaStreamSynchronize(s));
    CUDA(cudaMemcpy(o1, d_o, (size_t)(br * bw) * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(gb1, d_gbias, (size_t)bw * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemset(d_o, 0xFF, (size_t)(br * bw) * 4));
    CUDA(cudaMemset(d_gbias, 0xFF, (size_t)bw * 4));
    CHECK(bias_gelu_tanh_bwd_noalloc(d_bg, d_bx, d_bb, d_o, d_gbias, br, bw, WGS_F32, s) == WGS_OK);
    CUDA(cudaStreamSynchronize(s));
    CUDA(cudaMemcpy(o2, d_o, (size_t)(br * bw) * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(gb2, d_gbias, (size_t)bw * 4, cudaMemcpyDeviceToHost));
    CHECK(memcmp(o1, o2, (size_t)(br * bw) * 4) == 0);
    CHECK(memcmp(gb1, gb2, (size_t)bw * 4) == 0);
    CHECK(isfinite(gb1[0]));

    /* ---- a bad index sets the error word; the check clears it ---- */
    idx[5] = (int32_t)n_src; /* one past the last source row */
    CUDA(cudaMemcpy(d_idx, idx, (size_t)n_idx * sizeof(int32_t), cudaMemcpyHostToDevice));
    CHECK(window_gather(d_src, (const int32_t *)d_idx, d_dst, n_src, n_idx, W, s) == WGS_OK);
    CHECK(wgs_check_error(s) == WGS_ERR_INDEX);
    CHECK(wgs_check_error(s) == WGS_OK);

    cudaFree(d_src); cudaFree(d_dst); cudaFree(d_idx); cudaFree(d_x); cudaFree(d_y);
    cudaFree(d_gx); cudaFree(d_gb); cudaFree(d_gy); cudaFree(d_bx); cudaFree(d_bg);
    cudaFree(d_bb); cudaFree(d_o); cudaFree(d_gbias); cudaFree(d_ws);
    cudaStreamDestroy(s);
    free(idx); free(src); free(dst); free(x); free(y); free(bx); free(bg); free(bb);
    free(o1); free(o2);

    /* ---- the same results in a new context after a device reset: the fp16
     * backward at [4000, 1536] runs 768-thread CTAs whose shared-memory limit
     * is raised per context, and the no-alloc form looks its array up in
     * the current context ---- */
    {
        const int64_t hr = 4000;
        const int32_t hw = 1536;
        const size_t hn = (size_t)(hr * hw);
        uint16_t *h_gy = (uint16_t *)malloc(hn * 2), *h_x = (uint16_t *)malloc(hn * 2);
        uint16_t h_b[1536];
        uint16_t *r[4], *rb[4];
        wgs_status sw[2], sn[2];
        if (!h_gy || !h_x) return 1;
        for (size_t i = 0; i < hn; ++i) {
            h_gy[i] = rand_half();
            h_x[i] = rand_half();
        }
        for (int i = 0; i < hw; ++i) h_b[i] = rand_half();
        for (int k = 0; k < 4; ++k) {
            r[k] = (uint16_t *)malloc(hn * 2);
            rb[k] = (uint16_t *)malloc((size_t)hw * 2);
            if (!r[k] || !rb[k]) return 1;
        }
        if (bwd16(hr, hw, h_gy, h_x, h_b, r[0], rb[0], r[1], rb[1], &sw[0], &sn[0])) return 1;
        CUDA(cudaDeviceReset());
        if (bwd16(hr, hw, h_gy, h_x, h_b, r[2], rb[2], r[3], rb[3], &sw[1], &sn[1])) return 1;
        CHECK(sw[0] == WGS_OK && sn[0] == WGS_OK && sw[1] == WGS_OK && sn[1] == WGS_OK);
        for (int k = 1; k < 4; ++k) {
            CHECK(memcmp(r[0], r[k], hn * 2) == 0);
            CHECK(memcmp(rb[0], rb[k], (size_t)hw * 2) == 0);
        }
        for (int k = 0; k < 4; ++k) {
            free(r[k]);
            free(rb[k]);
        }
        free(h_gy);
        free(h_x);
    }
    if (fails) return 1;
    printf("device ok\n");
    return 0;
}
