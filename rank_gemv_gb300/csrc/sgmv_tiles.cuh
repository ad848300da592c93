// sgmv_tiles.cuh -- numbering of tiles over segments, done on the device.
//
// A tile is up to `rows` consecutive sorted positions of one segment.  The
// tiles of the segments a launch handles (adapter >= 0, or also -1 when
// asked; length in [min_len, max_len]) are numbered in segment order, and
// grid.y is the tile number.  Every CTA derives its tile from seg_ptr, so
// metadata built on the host or by the device grouping kernel both work.
#pragma once

#include "sgmv_device.cuh"

namespace sgmv {

// Warp 0 finds tile `tile`.  out = {segment or -1, first position, rows,
// adapter}.  With `report` the warp scans every segment and records malformed
// ones in the error word (one CTA per launch reports).
__device__ __forceinline__ void find_tile(const int32_t *seg_ptr, const int32_t *idx, int S,
                                          int T, int L, int rows, int min_len, int max_len,
                                          int *err, int tile, bool with_no_adapter, bool report,
                                          int *out) {
    const int lane = threadIdx.x & 31;
    int base = 0;
    int f_s = -1, f_p0 = 0, f_n = 0, f_a = -1;
    for (int s0 = 0; s0 < S; s0 += 32) {
        const int s = s0 + lane;
        int n = 0, b = 0, e = 0, a = -1;
        if (s < S) {
            b = seg_ptr[s];
            e = seg_ptr[s + 1];
            a = idx[s];
            const bool seg_ok = b >= 0 && e >= b && e <= T;
            const bool idx_ok = a >= -1 && a < L;
            if (report && !seg_ok) set_error(err, kErrBadSegments);
            if (report && seg_ok && !idx_ok) set_error(err, kErrBadIndex);
            const int len = e - b;
            if (seg_ok && idx_ok && len > 0 && (a >= 0 || with_no_adapter) && len >= min_len &&
                len <= max_len)
                n = (len + rows - 1) / rows;
        }
        int incl = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        const int excl = incl - n;
        const bool mine = f_s < 0 && n > 0 && tile >= base + excl && tile < base + incl;
        const unsigned m = __ballot_sync(0xffffffffu, mine);
        if (m) {
            const int src = __ffs(m) - 1;
            int p0 = 0, nr = 0;
            if (lane == src) {
                p0 = b + (tile - base - excl) * rows;
                nr = min(rows, e - p0);
            }
            f_s = __shfl_sync(0xffffffffu, s, src);
            f_p0 = __shfl_sync(0xffffffffu, p0, src);
            f_n = __shfl_sync(0xffffffffu, nr, src);
            f_a = __shfl_sync(0xffffffffu, a, src);
            if (!report) break;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
        out[0] = f_s;
        out[1] = f_p0;
        out[2] = f_n;
        out[3] = f_a;
    }
}

}  // namespace sgmv
