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

// Most pieces in one CTA's run (find_run): three, see there.
constexpr int kMaxPieces = 3;

// A CTA's run: pieces of consecutive column blocks, each of one tile.
struct Run {
    int n;                      // pieces (0: nothing to do)
    int k0[kMaxPieces + 1];     // first block of piece i in the CTA's sequence; k0[n] = blocks
    int p0[kMaxPieces];         // tile's first sorted position
    int rows[kMaxPieces];       // tile's rows
    int a[kMaxPieces];          // adapter
    int b0[kMaxPieces];         // first column block
};

// The blocks claimed at run time (find_run): the tiles from the first one with
// a block past the static part of the line to the last, at most kMaxDyn.
constexpr int kMaxDyn = 32;
struct DynTable {
    int n;                  // tiles (0: every block is dealt statically)
    int d0[kMaxDyn + 1];    // first claimed block of tile i; d0[n] = claimed blocks
    int p0[kMaxDyn];        // tile's first sorted position
    int rows[kMaxDyn];      // tile's rows
    int a[kMaxDyn];         // adapter
    int b0[kMaxDyn];        // first claimed column block of the tile
};

// Warp 0 of CTA c of G finds the CTA's run.  Tiles are numbered as in
// find_tile (segments with an adapter only), each cut into nblk column
// blocks; block b of tile t weighs rows_t + kw.  The blocks are laid end to
// end in (tile, block) order on a line of total weight W.  The blocks that
// start before Ws = W sfrac / 64 are dealt statically: CTA c takes those that
// start in [c Ws / G, (c+1) Ws / G), equal shares of weight, so a run may end
// inside one tile and go on into the next.  With G >= ntiles a share weighs
// at most nblk (rows + kw) + 1, a tile at least nblk (1 + kw); with
// kw > rows - 2 no share holds two whole tiles, so a run has at most three
// pieces (the end of one tile, a whole one, the start of the next).  The
// blocks from Ws on, in the same order, are listed in *dyn for the CTAs to
// claim at run time; when they span more than kMaxDyn tiles (or sfrac is 64)
// the whole line is dealt statically and dyn->n is 0.  G below the number of
// tiles is an error (kErrBadSegments) and every CTA gets nothing.
__device__ __forceinline__ void find_run(const int32_t *seg_ptr, const int32_t *idx, int S, int T,
                                         int L, int rows, int kw, int nblk, int min_len,
                                         int max_len, int *err, int c, int G, bool report,
                                         int sfrac, Run *out, DynTable *dyn) {
    const int lane = threadIdx.x & 31;
    // pass 1: number of tiles and total weight per column block
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
    int np = 0, nd = 0;
    if (ntiles > G && report && lane == 0) set_error(err, kErrBadSegments);
    if (ntiles > 0 && ntiles <= G) {
        const long long W = (long long)nblk * wsum;
        const long long full = (long long)nblk * (rows + kw);  // weight of a full tile
        long long Ws = W;
        if (sfrac < 64) {
            // the claimed part: tiles j >= jd of each segment, jd the first
            // whose last block starts at or after Wd
            const long long Wd = W * sfrac / 64;
            long long wbase = 0;
            for (int s0 = 0; s0 < S && nd <= kMaxDyn; s0 += 32) {
                const int s = s0 + lane;
                int n = 0, b = 0, e = 0, a = -1;
                if (s < S) n = seg_tiles(seg_ptr, idx, s, T, L, rows, min_len, max_len, err, false, b, e, a);
                const long long w = n > 0 ? (long long)nblk * ((long long)(e - b) + (long long)kw * n) : 0;
                long long iw = w;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const long long v = __shfl_up_sync(0xffffffffu, iw, off);
                    if (lane >= off) iw += v;
                }
                const long long ws = wbase + iw - w;
                int jd = n, f0 = 0;
                if (n > 0 && ws + w > Wd) {
                    jd = Wd > ws ? (int)min((long long)(n - 1), (Wd - ws) / full) : 0;
                    const long long wt = ws + (long long)jd * full;
                    const long long wb = (long long)(min(rows, (e - b) - jd * rows) + kw);
                    const long long f = Wd > wt ? (Wd - wt + wb - 1) / wb : 0;
                    if (f >= nblk) ++jd;
                    else f0 = (int)f;
                }
                const int cnt = n - jd;
                int ic = cnt;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, ic, off);
                    if (lane >= off) ic += v;
                }
                for (int q = 0; q < cnt && nd + ic - cnt + q < kMaxDyn; ++q) {
                    const int slot = nd + ic - cnt + q, j = jd + q;
                    dyn->p0[slot] = b + j * rows;
                    dyn->rows[slot] = min(rows, (e - b) - j * rows);
                    dyn->a[slot] = a;
                    dyn->b0[slot] = q == 0 ? f0 : 0;
                }
                nd += __shfl_sync(0xffffffffu, ic, 31);
                wbase += __shfl_sync(0xffffffffu, iw, 31);
            }
            if (nd > 0 && nd <= kMaxDyn) Ws = Wd;
            else nd = 0;
        }
        const long long lo = (long long)c * Ws / G, hi = (long long)(c + 1) * Ws / G;
        long long wbase = 0;  // weight of the segments before this batch
        for (int s0 = 0; s0 < S && lo < hi; s0 += 32) {
            const int s = s0 + lane;
            int n = 0, b = 0, e = 0, a = -1;
            if (s < S) n = seg_tiles(seg_ptr, idx, s, T, L, rows, min_len, max_len, err, false, b, e, a);
            const long long w = n > 0 ? (long long)nblk * ((long long)(e - b) + (long long)kw * n) : 0;
            long long iw = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const long long v = __shfl_up_sync(0xffffffffu, iw, off);
                if (lane >= off) iw += v;
            }
            const long long ws = wbase + iw - w;  // where segment s starts on the line
            // this segment's pieces: tiles j whose blocks start in [lo, hi)
            // (one entry more than a run holds, so that an overflow is seen)
            int cnt = 0, pj[kMaxPieces + 1], pb[kMaxPieces + 1], pn[kMaxPieces + 1];
            if (n > 0 && ws < hi && ws + w > lo) {
                int j = lo > ws ? (int)min((long long)(n - 1), (lo - ws) / full) : 0;
                for (; j < n && cnt <= kMaxPieces; ++j) {
                    const long long wt = ws + (long long)j * full;  // tiles before j are full
                    if (wt >= hi) break;
                    const int nr = min(rows, (e - b) - j * rows);
                    const long long wb = (long long)(nr + kw);
                    const long long f = lo > wt ? (lo - wt + wb - 1) / wb : 0;
                    const long long l = min((long long)nblk, (hi - wt + wb - 1) / wb);
                    if (f < l) {
                        pj[cnt] = j;
                        pb[cnt] = (int)f;
                        pn[cnt] = (int)(l - f);
                        ++cnt;
                    }
                }
            }
            int ic = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, ic, off);
                if (lane >= off) ic += v;
            }
            for (int q = 0; q < cnt; ++q) {
                const int slot = np + ic - cnt + q;
                if (slot < kMaxPieces) {
                    out->p0[slot] = b + pj[q] * rows;
                    out->rows[slot] = min(rows, (e - b) - pj[q] * rows);
                    out->a[slot] = a;
                    out->b0[slot] = pb[q];
                    out->k0[slot + 1] = pn[q];  // a count here; prefix sums below
                }
            }
            np += __shfl_sync(0xffffffffu, ic, 31);
            wbase += __shfl_sync(0xffffffffu, iw, 31);
            // segments after this batch start at or beyond wbase
            if (wbase >= hi) break;
        }
        if (np > kMaxPieces) {
            if (lane == 0) set_error(err, kErrBadSegments);
            np = 0;
        }
    }
    __syncwarp();
    if (lane == 0) {
        out->n = np;
        out->k0[0] = 0;
        for (int q = 0; q < np; ++q) out->k0[q + 1] += out->k0[q];
        dyn->n = nd;
        dyn->d0[0] = 0;
        for (int q = 0; q < nd; ++q) dyn->d0[q + 1] = dyn->d0[q] + (nblk - dyn->b0[q]);
    }
    __syncwarp();
}

}  // namespace sgmv
