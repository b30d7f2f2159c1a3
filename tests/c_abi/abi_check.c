/*
 * The C ABI used from plain C99: include/wgs.h compiles as C, links against
 * libwgs.so, and the host-side entry points behave as declared.  Only calls
 * that need no GPU are made (host builders, status strings, and argument
 * errors that every device entry point reports before touching a device).
 * Prints "abi ok" and exits 0, or names the first failed check and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "wgs.h"

static int fails = 0;
#define CHECK(cond)                                                     \
    do {                                                                \
        if (!(cond)) {                                                  \
            fprintf(stderr, "check failed (line %d): %s\n", __LINE__, #cond); \
            ++fails;                                                    \
        }                                                               \
    } while (0)

int main(void) {
    const int32_t grid[3] = {2, 12, 24}, win[3] = {2, 6, 12}, shift[3] = {1, 3, 6};
    static int32_t idx[576], inv[576], lab[576];
    int64_t i;

    CHECK(wgs_abi_version() == WGS_ABI_VERSION);
    CHECK(strcmp(wgs_status_string(WGS_OK), "ok") == 0);
    CHECK(strstr(wgs_status_string(WGS_ERR_INDEX), "index") != NULL);

    /* the tiny grid: 576 rows, no pads; destination 0 reads token
       (1*12 + 3)*24 + 6 = 366 (roll by -shift), destination 150 wraps in W */
    CHECK(wgs_window_index_count(grid, win, NULL) == 576);
    CHECK(wgs_build_window_index(grid, win, shift, NULL, WGS_SHIFT_THEN_PAD, idx, 576) == WGS_OK);
    CHECK(idx[0] == 366);
    CHECK(idx[150] == 360);
    CHECK(idx[575] == 53);
    CHECK(wgs_build_window_inverse(grid, win, shift, NULL, WGS_SHIFT_THEN_PAD, inv, 576) == WGS_OK);
    for (i = 0; i < 576; ++i) CHECK(inv[idx[i]] == i);
    CHECK(wgs_build_shift_regions(grid, win, shift, NULL, WGS_SHIFT_THEN_PAD, 7, lab, 576) == WGS_OK);
    CHECK(lab[0] == 0);
    CHECK(wgs_build_window_index(grid, win, shift, NULL, WGS_SHIFT_THEN_PAD, idx, 575) == WGS_ERR_SHAPE);

    /* argument errors come back before any device work */
    CHECK(ln_fwd(NULL, NULL, 10, 192, 1e-5f, 0) == WGS_ERR_NULL);
    CHECK(ln_fwd(NULL, NULL, 0, 192, 1e-5f, 0) == WGS_OK);
    CHECK(residual_add_ln_fwd(NULL, NULL, NULL, NULL, 10, 100, 1e-5f, 0) == WGS_ERR_WIDTH);
    CHECK(window_gather(NULL, NULL, NULL, 10, 0, 192, 0) == WGS_OK);
    CHECK(bias_gelu_tanh(NULL, NULL, NULL, 4, 8, (wgs_dtype)7, 0) == WGS_ERR_DTYPE);
    CHECK(window_bias_mask_add(NULL, NULL, NULL, NULL, NULL, 4, 6, 144, 1, -100.0f, WGS_F32, 0) ==
          WGS_ERR_DTYPE);
    CHECK(wgs_bias_gelu_bwd_workspace_bytes(0, 768) == 768 * 4);

    if (fails) return 1;
    printf("abi ok\n");
    return 0;
}
