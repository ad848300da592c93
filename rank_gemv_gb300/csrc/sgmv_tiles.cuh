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

// Tiles of segment s (as find_tile counts them) with its first and end
// positions and adapter; 0 for a segment the launch does not handle.
__device__ __forceinline__ int seg_tiles(const int32_t *seg_ptr, const int32_t *idx, int s, int T,
                                         int L, int rows, int min_len, int max_len, int *err,
                                         bool report, int &b, int &e, int &a) {
    b = seg_ptr[s];
    e = seg_ptr[s + 1];
    a = idx[s];
    const bool seg_ok = b >= 0 && e >= b && e <= T;
    const bool idx_ok = a >= -1 && a < L;
    if (report && !seg_ok) set_error(err, kErrBadSegments);
    if (report && seg_ok && !idx_ok) set_error(err, kErrBadIndex);
    const int len = e - b;
    if (seg_ok && idx_ok && len > 0 && a >= 0 && len >= min_len && len <= max_len)
        return (len + rows - 1) / rows;
    return 0;
}

// Warp 0 of CTA c of G finds the CTA's share of the launch.  Tiles are
// numbered as in find_tile (segments with an adapter only); tile t weighs
// w_t = rows_t + kw, and the G CTAs are dealt to the tiles in proportion to
// weight, at least one each: tile t gets CTAs [start_t, start_t+1) with
//   start_t = t + floor((G - ntiles) * W_t / W),
// W_t the weight of the tiles before t and W the total, so start_0 = 0 and
// start_ntiles = G.  out = {segment or -1, first position, rows, adapter,
// index of the CTA among its tile's CTAs, CTAs of the tile}.  G below the
// number of tiles is an error (kErrBadSegments) and every CTA gets nothing.
__device__ __forceinline__ void find_share(const int32_t *seg_ptr, const int32_t *idx, int S,
                                           int T, int L, int rows, int kw, int min_len,
                                           int max_len, int *err, int c, int G, bool report,
                                           int *out) {
    const int lane = threadIdx.x & 31;
    // pass 1: number of tiles and total weight
    int ntiles = 0;
    long long wsum = 0;
    for (int s0 = 0; s0 < S; s0 += 32) {
        const int s = s0 + lane;
        int n = 0, b = 0, e = 0, a = -1;
        if (s < S) n = seg_tiles(seg_ptr, idx, s, T, L, rows, min_len, max_len, err, report, b, e, a);
        long long w = n > 0 ? (long long)(e - b) + (long long)kw * n : 0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            n += __shfl_xor_sync(0xffffffffu, n, off);
            w += __shfl_xor_sync(0xffffffffu, w, off);
        }
        ntiles += n;
        wsum += w;
    }
    int f_s = -1, f_p0 = 0, f_n = 0, f_a = -1, f_i = 0, f_c = 0;
    const long long E = (long long)G - ntiles;
    if (E < 0 && report && lane == 0) set_error(err, kErrBadSegments);
    if (E >= 0 && ntiles > 0) {
        // pass 2: the segment, then the tile, whose CTAs include c
        auto start = [&](long long t, long long wpre) { return t + E * wpre / wsum; };
        int tbase = 0;
        long long wbase = 0;
        for (int s0 = 0; s0 < S; s0 += 32) {
            const int s = s0 + lane;
            int n = 0, b = 0, e = 0, a = -1;
            if (s < S) n = seg_tiles(seg_ptr, idx, s, T, L, rows, min_len, max_len, err, false, b, e, a);
            const long long w = n > 0 ? (long long)(e - b) + (long long)kw * n : 0;
            int in = n;
            long long iw = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int vn = __shfl_up_sync(0xffffffffu, in, off);
                const long long vw = __shfl_up_sync(0xffffffffu, iw, off);
                if (lane >= off) {
                    in += vn;
                    iw += vw;
                }
            }
            const int t0 = tbase + in - n;       // first tile of segment s
            const long long w0 = wbase + iw - w;  // weight before it
            const bool mine = n > 0 && c >= start(t0, w0) && c < start(t0 + n, w0 + w);
            const unsigned m = __ballot_sync(0xffffffffu, mine);
            if (m) {
                if (mine) {
                    // last tile j of the segment with start <= c (all but the
                    // segment's last tile have `rows` rows)
                    const long long wf = (long long)rows + kw;
                    int lo = 0, hi = n - 1;
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (start(t0 + mid, w0 + mid * wf) <= c) lo = mid;
                        else hi = mid - 1;
                    }
                    const int p0 = b + lo * rows, nr = min(rows, e - p0);
                    const long long st = start(t0 + lo, w0 + lo * wf);
                    const long long nx = start(t0 + lo + 1, w0 + lo * wf + nr + kw);
                    f_s = s;
                    f_p0 = p0;
                    f_n = nr;
                    f_a = a;
                    f_i = (int)(c - st);
                    f_c = (int)(nx - st);
                }
                const int src = __ffs(m) - 1;
                f_s = __shfl_sync(0xffffffffu, f_s, src);
                f_p0 = __shfl_sync(0xffffffffu, f_p0, src);
                f_n = __shfl_sync(0xffffffffu, f_n, src);
                f_a = __shfl_sync(0xffffffffu, f_a, src);
                f_i = __shfl_sync(0xffffffffu, f_i, src);
                f_c = __shfl_sync(0xffffffffu, f_c, src);
                break;
            }
            tbase += __shfl_sync(0xffffffffu, in, 31);
            wbase += __shfl_sync(0xffffffffu, iw, 31);
        }
    }
    if (lane == 0) {
        out[0] = f_s;
        out[1] = f_p0;
        out[2] = f_n;
        out[3] = f_a;
        out[4] = f_i;
        out[5] = f_c;
    }
}

}  // namespace sgmv
