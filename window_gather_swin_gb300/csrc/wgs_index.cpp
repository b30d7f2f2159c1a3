// Host-side construction of the shifted-window INT32 index map.
//
// Page "BW1000 gfx936 Pangu-Weather inference profiling", s5: the window
// gather reads one precomputed INT32 per destination row; a value >= 0 names
// the source token and -1 asks for a zero row, so shift, padding and the
// window-major reordering all live in one array built once per window shape.
// The construction (see wgs.h) walks the destination in order: window by
// window, then cell by cell inside each window, writing each cell's source.
#include "wgs.h"

#include <cstdint>

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t wrap(int64_t a, int64_t m) {
    int64_t r = a % m;
    return r < 0 ? r + m : r;
}

// a * b for positive a, b, or false when the product passes INT64_MAX.
bool mul_fits(int64_t a, int64_t b, int64_t *out) {
    if (a > INT64_MAX / b) return false;
    *out = a * b;
    return true;
}

// Padded extents (given, or the grid rounded up to whole windows), the cell
// count of the padded grid and of the grid.  False for a non-positive grid
// or window, a padded extent below the grid or above INT32_MAX, or a cell
// count past INT64_MAX.
bool padded_extents(const int32_t grid[3], const int32_t window[3], const int32_t *padded,
                    int64_t ext[3], int64_t *cells, int64_t *grid_cells) {
    int64_t n = 1, g = 1;
    for (int k = 0; k < 3; ++k) {
        if (grid[k] < 1 || window[k] < 1) return false;
        ext[k] = padded ? padded[k] : ceil_div(grid[k], window[k]) * window[k];
        if (ext[k] < grid[k] || ext[k] > INT32_MAX) return false;
        if (!mul_fits(n, ext[k], &n) || !mul_fits(g, grid[k], &g)) return false;
    }
    *cells = n;
    *grid_cells = g;
    return true;
}

}  // namespace

extern "C" int64_t wgs_window_index_count(const int32_t grid[3], const int32_t window[3],
                                          const int32_t *padded) {
    if (!grid || !window) return -1;
    int64_t ext[3], cells, grid_cells;
    if (!padded_extents(grid, window, padded, ext, &cells, &grid_cells)) return -1;
    return cells;
}

extern "C" wgs_status wgs_build_window_index(const int32_t grid[3], const int32_t window[3],
                                             const int32_t shift[3], const int32_t *padded,
                                             int32_t flags, int32_t *out_host, int64_t out_len) {
    if (!grid || !window || !shift || !out_host) return WGS_ERR_NULL;
    if (flags != WGS_SHIFT_THEN_PAD && flags != WGS_PAD_THEN_SHIFT) return WGS_ERR_SHAPE;
    int64_t ext[3], cells, grid_cells;
    if (!padded_extents(grid, window, padded, ext, &cells, &grid_cells)) return WGS_ERR_SHAPE;
    const int64_t G[3] = {grid[0], grid[1], grid[2]};
    if (grid_cells > INT32_MAX) return WGS_ERR_SHAPE;  // source tokens are INT32
    if (out_len < cells) return WGS_ERR_SHAPE;

    // The roll is taken modulo the grid (shift then pad) or the padded grid
    // (pad then shift).
    const bool roll_padded = flags == WGS_PAD_THEN_SHIFT;
    int64_t period[3], s[3];
    for (int k = 0; k < 3; ++k) {
        period[k] = roll_padded ? ext[k] : G[k];
        s[k] = wrap(shift[k], period[k]);
    }

    int64_t d = 0;
    for (int64_t z0 = 0; z0 < ext[0]; z0 += window[0])
        for (int64_t h0 = 0; h0 < ext[1]; h0 += window[1])
            for (int64_t w0 = 0; w0 < ext[2]; w0 += window[2]) {
                const int64_t z1 = z0 + window[0] < ext[0] ? z0 + window[0] : ext[0];
                const int64_t h1 = h0 + window[1] < ext[1] ? h0 + window[1] : ext[1];
                const int64_t w1 = w0 + window[2] < ext[2] ? w0 + window[2] : ext[2];
                for (int64_t z = z0; z < z1; ++z)
                    for (int64_t h = h0; h < h1; ++h)
                        for (int64_t w = w0; w < w1; ++w) {
                            int32_t v = -1;
                            const bool inside = z < G[0] && h < G[1] && w < G[2];
                            if (roll_padded || inside) {
                                int64_t zs = z + s[0], hs = h + s[1], ws = w + s[2];
                                if (zs >= period[0]) zs -= period[0];
                                if (hs >= period[1]) hs -= period[1];
                                if (ws >= period[2]) ws -= period[2];
                                if (zs < G[0] && hs < G[1] && ws < G[2])
                                    v = static_cast<int32_t>((zs * G[1] + hs) * G[2] + ws);
                            }
                            out_host[d++] = v;
                        }
            }
    return WGS_OK;
}

// Inverse of the map above: inv[t] = the windowed row that holds token t.
// Computed in closed form per token: the destination cell is the token's
// coordinates rolled back by the shift (modulo the grid, or the padded grid
// for pad-then-shift), and a cell's position in the window-major order is
// the cells of all earlier window slabs / bands / windows plus its row-major
// offset inside its own (possibly cut) window.
extern "C" wgs_status wgs_build_window_inverse(const int32_t grid[3], const int32_t window[3],
                                               const int32_t shift[3], const int32_t *padded,
                                               int32_t flags, int32_t *inv_host, int64_t out_len) {
    if (!grid || !window || !shift || !inv_host) return WGS_ERR_NULL;
    if (flags != WGS_SHIFT_THEN_PAD && flags != WGS_PAD_THEN_SHIFT) return WGS_ERR_SHAPE;
    int64_t P[3], cells, grid_cells;
    if (!padded_extents(grid, window, padded, P, &cells, &grid_cells)) return WGS_ERR_SHAPE;
    const int64_t G[3] = {grid[0], grid[1], grid[2]};
    if (cells > INT32_MAX) return WGS_ERR_SHAPE;  // windowed rows are INT32
    if (out_len < grid_cells) return WGS_ERR_SHAPE;
    const bool roll_padded = flags == WGS_PAD_THEN_SHIFT;
    int64_t period[3], s[3], w[3];
    for (int k = 0; k < 3; ++k) {
        period[k] = roll_padded ? P[k] : G[k];
        s[k] = wrap(shift[k], period[k]);
        w[k] = window[k];
    }
    int64_t t = 0;
    for (int64_t z = 0; z < G[0]; ++z)
        for (int64_t h = 0; h < G[1]; ++h)
            for (int64_t x = 0; x < G[2]; ++x) {
                // destination cell c with c + shift = (z, h, x) modulo the period
                const int64_t c[3] = {wrap(z - s[0], period[0]), wrap(h - s[1], period[1]),
                                      wrap(x - s[2], period[2])};
                int64_t b[3], e[3], i[3];
                for (int k = 0; k < 3; ++k) {
                    b[k] = c[k] / w[k];
                    i[k] = c[k] % w[k];
                    e[k] = P[k] - b[k] * w[k] < w[k] ? P[k] - b[k] * w[k] : w[k];
                }
                const int64_t start = b[0] * w[0] * P[1] * P[2] + e[0] * b[1] * w[1] * P[2] +
                                      e[0] * e[1] * b[2] * w[2];
                inv_host[t++] = static_cast<int32_t>(start + (i[0] * e[1] + i[1]) * e[2] + i[2]);
            }
    return WGS_OK;
}

// Shift-mask region labels in the destination order of the map above: the
// same window walk, with each cell labelled by the axes along which it lies
// past the roll's seam.
extern "C" wgs_status wgs_build_shift_regions(const int32_t grid[3], const int32_t window[3],
                                              const int32_t shift[3], const int32_t *padded,
                                              int32_t flags, int32_t axes_mask, int32_t *out_host,
                                              int64_t out_len) {
    if (!grid || !window || !shift || !out_host) return WGS_ERR_NULL;
    if (flags != WGS_SHIFT_THEN_PAD && flags != WGS_PAD_THEN_SHIFT) return WGS_ERR_SHAPE;
    if (axes_mask < 0 || axes_mask > 7) return WGS_ERR_SHAPE;
    int64_t ext[3], cells, grid_cells;
    if (!padded_extents(grid, window, padded, ext, &cells, &grid_cells)) return WGS_ERR_SHAPE;
    if (out_len < cells) return WGS_ERR_SHAPE;
    // seam[k]: first cell past the seam along k (ext[k] when the axis is
    // not masked or not moved, so no cell is past it)
    int64_t seam[3];
    for (int k = 0; k < 3; ++k) {
        const int64_t period = flags == WGS_PAD_THEN_SHIFT ? ext[k] : grid[k];
        const int64_t s = wrap(shift[k], period);
        seam[k] = ((axes_mask >> k) & 1) && s != 0 ? period - s : ext[k];
    }
    int64_t d = 0;
    for (int64_t z0 = 0; z0 < ext[0]; z0 += window[0])
        for (int64_t h0 = 0; h0 < ext[1]; h0 += window[1])
            for (int64_t w0 = 0; w0 < ext[2]; w0 += window[2]) {
                const int64_t z1 = z0 + window[0] < ext[0] ? z0 + window[0] : ext[0];
                const int64_t h1 = h0 + window[1] < ext[1] ? h0 + window[1] : ext[1];
                const int64_t w1 = w0 + window[2] < ext[2] ? w0 + window[2] : ext[2];
                for (int64_t z = z0; z < z1; ++z)
                    for (int64_t h = h0; h < h1; ++h)
                        for (int64_t w = w0; w < w1; ++w)
                            out_host[d++] = (z >= seam[0] ? 1 : 0) | (h >= seam[1] ? 2 : 0) |
                                            (w >= seam[2] ? 4 : 0);
            }
    return WGS_OK;
}
