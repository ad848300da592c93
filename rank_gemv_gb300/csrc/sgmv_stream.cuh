// sgmv_stream.cuh -- persistent streaming CUDA-core SGMV kernel for
// decode-sized segments (rank r <= 64, r a multiple of 4).
//
// Method ("Punica: when LoRA fine-tuned models need multi-tenant serving",
// omica.com.cn article, §2.2): for every row of a segment, shrink
// v = x . A[idx] with A gathered out of the stacked adapters, then expand
// y += scale * v . B[idx].  Decode rows do about one flop per weight byte, so
// the kernel is built to keep HBM busy rather than the arithmetic units.
//
// Work decomposition:
//   * a tile is up to `trows` (1..8) consecutive rows of one segment;
//   * CL CTAs form a cluster (CL = 1, 2, 4 or 8, fewer for larger batches);
//     CTA `rank` owns the slice [rank*hc, ...) of H1 and [rank*jc, ...) of H2;
//   * one launch may carry up to four problems with the same rows, segments
//     and shapes but their own x, A, B and y (the projections of a layer
//     that read the same rows); a unit is a (problem, tile) pair, numbered
//     problem by problem;
//   * cluster c walks the units c, c + G, c + 2G, ...: the kernel is
//     persistent over units, and each CTA streams its slices of every unit's
//     A and B through a ring of shared-memory stages, 32 KB of weights per
//     chunk at the rank bound: one 1-D bulk (TMA) copy per A chunk
//     (contiguous in A[a]), tiled tensor (TMA) boxes of 256 columns x r rows
//     per B chunk, one bulk copy per x or y row.  One warp
//     only issues copies; eight warps compute.  The ring order is A(0); A(1) B(0); A(2) B(1); ...: the shrink of tile m runs
//     before the expand of tile m-1, so the cluster exchange of tile m-1's v
//     is hidden behind it, and the copies never wait for an exchange;
//   * partial v of a CTA's H1 slice goes to every CTA of the cluster through
//     distributed shared memory (double-buffered by tile parity, one mbarrier
//     per buffer with one release-arrive per CTA), and each CTA sums the
//     partials in rank order: the same bits in every CTA.
// Summation order of every output element: fixed by (H1, H2, r, CL) alone --
// not by the number of rows in a tile, the chunking or the tile assignment --
// so cutting a segment into tiles differently changes no bit.
// Programmatic dependent launch: segment metadata and weights are read before
// griddepcontrol.wait; x and y only after it.
#pragma once

#include <climits>

#include "sgmv_device.cuh"
#include "sgmv_internal.h"

namespace sgmv {

constexpr int kTileRows = 8;

// Barrier of the CW compute warps (the copy warp does not take part).
template <int CW> __device__ __forceinline__ void consumers_sync() { named_sync<1, CW * 32>(); }

// Walks a CTA's ring in order: A(0); then for m = 1 .. nt-1: A(m), B(m-1);
// then B(nt-1).  Chunk = A(blk, i) when !isB, else B(blk - 1, i).
struct RingIter {
    int blk, isB, i, nt, nA, nB;
    __device__ __forceinline__ void start(int nt_, int nA_, int nB_) {
        nt = nt_;
        nA = nA_;
        nB = nB_;
        blk = 0;
        isB = 0;
        i = 0;
        settle();
    }
    __device__ __forceinline__ void settle() {
        for (;;) {
            if (blk > nt) return;
            if (!isB) {
                if (blk < nt && i < nA) return;
                isB = 1;
                i = 0;
            }
            if (blk >= 1 && i < nB) return;
            ++blk;
            isB = 0;
            i = 0;
        }
    }
    __device__ __forceinline__ void next() {
        ++i;
        settle();
    }
    __device__ __forceinline__ int tile() const { return isB ? blk - 1 : blk; }
};

// Bounded wait of a compute thread; after a timeout the error word is set, the
// wait is repeated once with the full limit (copies still in flight land
// before the CTA moves on) and the thread stops writing y.  `fail` takes the
// timeout path without polling first (the injected timeout of a diagnostic
// launch); the repeated wait is the same as after a real timeout.
__device__ __forceinline__ void stream_wait(uint64_t *bar, uint32_t parity, bool &lost, int *err,
                                            bool fail = false) {
    if (fail || !mbar_wait(bar, parity)) {
        set_error(err, kErrTimeout);
        mbar_wait(bar, parity);
        lost = true;
    }
}

// Shrink of one tile with R rows (R >= the tile's rows): the CTA's partial of
// v over its H1 slice, one warp partial per warp written to red[warp][t][k].
// Thread (warp, lane) owns k-quad kq = lane % (RK/4) and the columns
// h = warp*HL + lane/(RK/4) + HSTR*j of the slice, summed in increasing h;
// the HL lanes of a k-quad are then summed by a butterfly in a fixed order.
template <typename Tin, int RK, int R, int CW>
__device__ __forceinline__ void stream_shrink(uint8_t *sm, uint32_t stage_bytes, uint32_t act_off,
                                              int nst, int &q, int nA, int hlen, int hn, int rk,
                                              uint64_t *full, uint64_t *empty, float *red,
                                              bool &lost, int *err, bool inject) {
    constexpr int KQ = RK / 4, HL = 32 / KQ, HSTR = CW * HL;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int kq = lane % KQ, hl = lane / KQ;
    const int hoff = warp * HL + hl;
    const bool kact = 4 * kq < rk;
    float acc[R][4];
#pragma unroll
    for (int t = 0; t < R; ++t)
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[t][u] = 0.f;
    for (int i = 0; i < nA; ++i, ++q) {
        const int s = q % nst;
        stream_wait(&full[s], (uint32_t)((q / nst) & 1), lost, err, inject && q == 0);
        const int nh = min(hn, hlen - i * hn);
        const uint8_t *base = sm + (size_t)s * stage_bytes;
        const Tin *As = reinterpret_cast<const Tin *>(base);
        const Tin *Xs = reinterpret_cast<const Tin *>(base + act_off);
        if (kact) {
#pragma unroll 2
            for (int h = hoff; h < nh; h += HSTR) {
                const uint2 av = lds64(As + h * rk + 4 * kq);
                const unsigned short a[4] = {(unsigned short)(av.x & 0xffffu),
                                             (unsigned short)(av.x >> 16),
                                             (unsigned short)(av.y & 0xffffu),
                                             (unsigned short)(av.y >> 16)};
#pragma unroll
                for (int t = 0; t < R; ++t) {
                    const unsigned short xb = lds16(Xs + t * hn + h);
#pragma unroll
                    for (int u = 0; u < 4; ++u) acc[t][u] = fma16<Tin>(xb, a[u], acc[t][u]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
#pragma unroll
    for (int off = 16; off >= KQ; off >>= 1)
#pragma unroll
        for (int t = 0; t < R; ++t)
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[t][u] += __shfl_xor_sync(0xffffffffu, acc[t][u], off);
    if (hl == 0 && kact)
#pragma unroll
        for (int t = 0; t < R; ++t)
            sts128(red + (warp * kTileRows + t) * RK + 4 * kq,
                   make_uint4(__float_as_uint(acc[t][0]), __float_as_uint(acc[t][1]),
                              __float_as_uint(acc[t][2]), __float_as_uint(acc[t][3])));
}

// Expand of one tile with R rows: y[row, j] += scale * v . B[a][:, j] for the
// CTA's H2 slice; each thread owns JN / (64 CW) pairs (at least one) of adjacent
// columns of a chunk and runs the r-sum in increasing k.
template <typename Tin, typename Ty, int RK, int R, int CW>
__device__ __forceinline__ void stream_expand(uint8_t *sm, uint32_t stage_bytes, uint32_t act_off,
                                              int nst, int &q, int nB, int jlen, int j0, int rk,
                                              const float *sv, const int (&row)[kTileRows],
                                              Ty *gY, int H2, float scale, uint64_t *full,
                                              uint64_t *empty, bool &lost, int *err) {
    constexpr int JN = kStreamChunkElems / RK;
    constexpr int PP = JN / (2 * CW * 32) > 0 ? JN / (2 * CW * 32) : 1;
    const int tid = threadIdx.x;
    for (int i = 0; i < nB; ++i, ++q) {
        const int s = q % nst;
        stream_wait(&full[s], (uint32_t)((q / nst) & 1), lost, err);
        const int nj = min(JN, jlen - i * JN);
        const uint8_t *base = sm + (size_t)s * stage_bytes;
        const Tin *Bs = reinterpret_cast<const Tin *>(base);
        const Ty *Ys = reinterpret_cast<const Ty *>(base + act_off);
#pragma unroll
        for (int pp = 0; pp < PP; ++pp) {
            const int c = 2 * (tid + pp * CW * 32);
            if (c >= nj) break;
            // B chunk in shared memory: boxes of 256 columns, [box][k][256]
            const Tin *bcol = Bs + (c >> 8) * rk * 256 + (c & 255);
            float acc[R][2];
#pragma unroll
            for (int t = 0; t < R; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll
            for (int kk = 0; kk < RK; kk += 4) {
                if (kk < rk) {
                    float v[R][4];
#pragma unroll
                    for (int t = 0; t < R; ++t) {
                        const uint4 u = lds128(sv + t * RK + kk);
                        v[t][0] = __uint_as_float(u.x);
                        v[t][1] = __uint_as_float(u.y);
                        v[t][2] = __uint_as_float(u.z);
                        v[t][3] = __uint_as_float(u.w);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float b0, b1;
                        unpack2<Tin>(lds32(bcol + (kk + e) * 256), b0, b1);
#pragma unroll
                        for (int t = 0; t < R; ++t) fma2(v[t][e], b0, b1, acc[t][0], acc[t][1]);
                    }
                }
            }
            if (!lost) {
                const int jg = j0 + i * JN + c;
#pragma unroll
                for (int t = 0; t < R; ++t) {
                    if (row[t] < 0) continue;
                    float y0, y1;
                    lds2<Ty>(Ys + t * JN + c, y0, y1);
                    st2<Ty>(gY + (size_t)row[t] * H2 + jg, fmaf(scale, acc[t][0], y0),
                            fmaf(scale, acc[t][1], y1));
                }
            }
        }
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(&empty[s]);
    }
}

// MULTI: the launch may carry several problems (P.np).  Single-problem
// launches use the instantiation without it, where every problem number is
// the constant 0: with a run-time problem number in the copy warp's tensor-map
// address and in the tile numbering, single calls measured 2-4 % slower.
template <typename Tin, typename Ty, int RK, bool GROUPED, int CW, bool MULTI = false>
__global__ void __launch_bounds__(CW * 32 + 32, CW == 8 ? 2 : 1)
    sgmv_stream_kernel(const __grid_constant__ StreamParamsT<MULTI ? kStreamMaxProblems : 1> P) {
    constexpr int kStreamConsumers = CW * 32, kStreamWarps = CW, kStreamThreads = CW * 32 + 32;
    // Parameters read once into registers (see sgmv_cc.cuh).
    const int T = P.T, L = P.L, H1 = P.H1, H2 = P.H2, rk = P.r;
    const int ncl = P.cl, G = P.G, hn = P.hn, nst = P.nst;
    const int min_len = P.min_len, max_len = P.max_len;
    const int trows = P.trows;  // rows per tile, 1..8
    const uint32_t stage_bytes = P.stage_bytes, act_off = P.act_off;
    const float scale = P.scale;
    int *const err = P.err;
    // diagnostic launches only: the first ring wait of every compute thread
    // reports a timeout (the chunk is still awaited before it is used)
    const bool inject = P.inject != 0;

    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ __align__(8) uint64_t full[kStreamMaxStages], empty[kStreamMaxStages], vfull[2];
    __shared__ int s_wsum[kStreamThreads / 32];
    __shared__ int s_total;
    constexpr int kG = GROUPED ? kGroupMaxT : 4;
    __shared__ __align__(16) int g_key[kG];
    __shared__ int g_pn[kG], g_pkey[kG], g_flag[kG], g_sperm[kG];
    __shared__ int g_nseg_s;
    // A, x and y of every problem (copied out of the parameters with
    // constant indices)
    __shared__ const void *s_pp[3][kStreamMaxProblems];
    const int np = MULTI ? P.np : 1;

    float *const red = reinterpret_cast<float *>(sm + P.red_off);    // [8 warps][8][RK]
    float *const recv = reinterpret_cast<float *>(sm + P.recv_off);  // [2][cl][8][RK]
    float *const s_v = reinterpret_cast<float *>(sm + P.v_off);      // [2][8][RK]
    int *const tab = reinterpret_cast<int *>(sm + P.tab_off);        // [tiles][4]: p0, n, a, problem
    int *const trow = tab + 4 * kStreamMaxTiles;                     // [tiles][8] rows

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = (int)blockIdx.x, cid = (int)blockIdx.y;
    const bool report = rank == 0 && cid == 0;

    // The next kernel on the stream may start as soon as every CTA of this
    // one has: it reads nothing this kernel writes before its own
    // griddepcontrol.wait, which still waits for this grid to finish.
    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 2);  // weights, then the x / y rows
            mbar_init(&empty[s], kStreamWarps);
        }
        mbar_init(&vfull[0], 1);  // armed once per tile with the bytes the peers push
        mbar_init(&vfull[1], 1);
        mbar_init_fence();
        s_total = 0;
        if constexpr (MULTI) {
#pragma unroll
            for (int q = 0; q < kStreamMaxProblems; ++q) {
                s_pp[0][q] = P.A[q];
                s_pp[1][q] = P.x[q];
                s_pp[2][q] = P.y[q];
            }
        }
    }

    // ---- this cluster's tiles: tab[m] = global tile cid + m*G ---------------
    int g_less = 0, g_nseg = 0, gkey = -1, grank = 0;
    if (!GROUPED) {
        // Tiles per segment, block-scanned over the segments in order.
        const int S = P.S;
        const int32_t *seg_ptr = P.seg_ptr;
        const int32_t *idx = P.idx;
        auto seg = [&](int s, int &b, int &len, int &a, bool rep) {
            b = seg_ptr[s];
            const int e = seg_ptr[s + 1];
            a = idx[s];
            if (b < 0 || e < b || e > T) {
                if (rep) set_error(err, kErrBadSegments);
                return 0;
            }
            len = e - b;
            if (len == 0 || a == -1 || len < min_len || len > max_len) return 0;
            if (a < -1 || a >= L) {
                if (rep) set_error(err, kErrBadIndex);
                return 0;
            }
            return (len + trows - 1) / trows;
        };
        const int per = (S + kStreamThreads - 1) / kStreamThreads;
        const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
        int own = 0;
        for (int s = s0; s < s1; ++s) {
            int b, len, a;
            own += seg(s, b, len, a, report);
        }
        int incl = own;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            constexpr int NW = kStreamThreads / 32;
            const int w = lane < NW ? s_wsum[lane] : 0;
            int wi = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, wi, off);
                if (lane >= off) wi += o;
            }
            if (lane < NW) s_wsum[lane] = wi - w;
            if (lane == NW - 1) s_total = wi;
        }
        __syncthreads();
        int gbase = s_wsum[warp] + incl - own;  // first global tile of this thread's segments
        const int ntile = s_total;               // tiles of one problem
        for (int s = s0; s < s1; ++s) {
            int b = 0, len = 0, a = 0;
            const int n = seg(s, b, len, a, false);
            // unit u = problem * ntile + tile: tiles j of this segment with
            // (u0 + j) % G == cid, u0 the unit of the segment's first tile
            for (int pb = 0; pb < np; ++pb) {
                const int u0 = pb * ntile + gbase;
                for (int j = ((cid - u0 % G) % G + G) % G; j < n; j += G) {
                    const int m = (u0 + j) / G;
                    if (m < kStreamMaxTiles) {
                        tab[4 * m] = b + trows * j;
                        tab[4 * m + 1] = min(trows, len - trows * j);
                        tab[4 * m + 2] = a;
                        tab[4 * m + 3] = pb;
                    }
                }
            }
            gbase += n;
        }
    } else {
        // Every CTA groups the batch itself (T <= kGroupMaxT).  Row t's sorted
        // position is p = (#rows with a smaller id) + (#earlier rows with its
        // id).  Each row then marks, at its position, whether it starts a
        // segment and whether it starts a tile (every trows-th row of an id,
        // ids >= 0 only); one scan over the positions numbers both.
        // Keys past T are INT_MAX, so that padded entries count for nothing.
        const int32_t *ra = P.row_adapter;
        const int T4 = (T + 3) & ~3;
        if (tid < T4) {
            if (tid < T) {
                gkey = ra[tid];
                if (gkey < -1 || gkey >= L) {
                    if (report) set_error(err, kErrBadIndex);
                    gkey = -1;
                }
            }
            g_key[tid] = tid < T ? gkey : INT_MAX;
        }
        __syncthreads();
        if (tid < T) {
            int cnt = 0;
            for (int u = 0; u < T4; u += 4) {
                const uint4 k4 = lds128(g_key + u);
                const int ku[4] = {(int)k4.x, (int)k4.y, (int)k4.z, (int)k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    g_less += ku[e] < gkey;
                    cnt += ku[e] == gkey;
                    grank += (ku[e] == gkey) & (u + e < tid);
                }
            }
            const int p = g_less + grank;
            g_sperm[p] = tid;
            g_pn[p] = min(trows, cnt - grank);  // rows of the tile starting here
            g_pkey[p] = gkey;                   // id at sorted position p
            // bit 0..15: starts a tile; bit 16..: starts a segment
            g_flag[p] = ((gkey >= 0 && (grank & (trows - 1)) == 0) ? 1 : 0) | (grank == 0 ? 0x10000 : 0);
        }
        __syncthreads();
        // Exclusive scan of the flags over positions 0 .. T-1 (two warps).
        const int f = tid < T ? g_flag[tid] : 0;
        int inc = f;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += o;
        }
        if (lane == 31 && warp < 2) s_wsum[warp] = inc;
        __syncthreads();
        const int before = (warp == 1 ? s_wsum[0] : 0) + inc - f;  // warps 0, 1 hold positions
        if (tid < T) {
            if (f & 1) {
                const int gt = before & 0xffff;
                if (gt % G == cid && gt / G < kStreamMaxTiles) {
                    const int m = gt / G;
                    tab[4 * m] = tid;
                    tab[4 * m + 1] = g_pn[tid];
                    tab[4 * m + 2] = g_pkey[tid];
                    tab[4 * m + 3] = 0;  // one problem
                }
            }
            g_flag[tid] = before;  // segment number (high half) of position tid
        }
        if (tid == 0) {
            const int tot = s_wsum[0] + (T > 32 ? s_wsum[1] : 0);
            s_total = tot & 0xffff;
            g_nseg_s = tot >> 16;
        }
        __syncthreads();
        g_nseg = g_nseg_s;
    }
    __syncthreads();
    const int ntot = s_total * np;  // units: tiles of every problem
    int nt = ntot > cid ? (ntot - 1 - cid) / G + 1 : 0;
    if (nt > kStreamMaxTiles) {
        if (rank == 0) set_error(err, kErrBadSegments);
        nt = kStreamMaxTiles;
    }
    // Grouped form, CTA (0,0): the grouping is written out for later calls,
    // after the previous kernel on the stream (which may still read it).
    auto write_meta = [&]() {  // thread p < T: sorted position p
        if (tid < T) {
            P.perm_out[tid] = g_sperm[tid];
            const int sg = g_flag[tid] >> 16;  // segments before position p
            if (tid == 0 || g_pkey[tid] != g_pkey[tid - 1]) {
                P.seg_out[sg] = tid;
                P.idx_out[sg] = g_pkey[tid];
            }
        }
        if (tid == 0) {
            P.seg_out[g_nseg] = T;
            *P.S_out = g_nseg;
        }
        for (int sidx = g_nseg + tid; sidx < P.S_max; sidx += kStreamThreads) {
            P.idx_out[sidx] = -1;
            P.seg_out[sidx + 1] = T;
        }
    };
    const bool meta_out = GROUPED && report && P.perm_out != nullptr;
    if (nt == 0) {  // the same for every CTA of the cluster
        if (meta_out) {
            pdl_wait();
            write_meta();
        }
        return;
    }
    if (ncl > 1) cluster_arrive_relaxed();  // waited on before the first peer access

    const int h0 = min(H1, rank * P.hc), h1 = min(H1, h0 + P.hc);
    const int j0 = min(H2, rank * P.jc), j1 = min(H2, j0 + P.jc);
    const int nA = (h1 - h0 + hn - 1) / hn;
    constexpr int JN = kStreamChunkElems / RK;
    const int nB = (j1 - j0 + JN - 1) / JN;
    const int total = nt * (nA + nB);

    if (warp == kStreamWarps) {
        // ---- copy warp: fills the ring in the order the compute warps use it.
        // Weights need only the adapter ids, so they are requested while the
        // compute warps look up the tiles' rows.
        // the unit's problem picks its A, B (tensor map), x and y
        const CUtensorMap *const tmb0 = &P.tmap_b[0];
        const Tin *gA = static_cast<const Tin *>(P.A[0]);
        const Tin *gX = static_cast<const Tin *>(P.x[0]);
        const Ty *gY = static_cast<const Ty *>(P.y[0]);
        const CUtensorMap *tmb = tmb0;
        const uint32_t bbox = (uint32_t)rk * 256u * (uint32_t)sizeof(Tin);
        const bool b4d = P.b4d != 0;
        RingIter it;
        int cur_a = -1, cur_r = -1, a = 0, row = -1;
        uint32_t nvalid = 0;
        auto issue_w = [&](int s) {  // weights of chunk `it` into stage s
            if (it.tile() != cur_a) {
                cur_a = it.tile();
                a = (int)lds32(tab + 4 * cur_a + 2);
                if (MULTI) {
                    const int pb = (int)lds32(tab + 4 * cur_a + 3);
                    gA = static_cast<const Tin *>(s_pp[0][pb]);
                    tmb = tmb0 + pb;
                }
            }
            uint8_t *dst = sm + (size_t)s * stage_bytes;
            if (lane == 0) {
                if (!it.isB) {
                    const int hlo = h0 + it.i * hn, n = min(hn, h1 - hlo);
                    const uint32_t bytes = (uint32_t)(n * rk) * (uint32_t)sizeof(Tin);
                    mbar_arrive_expect_tx(&full[s], bytes);
                    bulk_g2s(dst, gA + ((size_t)a * H1 + hlo) * rk, bytes, &full[s]);
                } else {
                    const int jlo = j0 + it.i * JN;
                    if (b4d && j1 - jlo >= JN) {  // a whole chunk in one copy
                        mbar_arrive_expect_tx(&full[s], bbox * (uint32_t)(JN / 256));
                        tma_load_4d(dst, tmb, 0, 0, jlo >> 8, a, &full[s]);
                    }
                }
            }
            if (it.isB && !(b4d && j1 - (j0 + it.i * JN) >= JN)) {  // one box of 256 columns per lane
                const int jlo = j0 + it.i * JN, n = min(JN, j1 - jlo);
                const int nbox = (n + 255) >> 8;
                if (lane == 0) mbar_arrive_expect_tx(&full[s], bbox * (uint32_t)nbox);
                __syncwarp();
                if (lane < nbox)
                    tma_load_3d(dst + lane * bbox, tmb, jlo + 256 * lane, 0, a, &full[s]);
            }
        };
        auto issue_act = [&](int s) {  // x or y rows of chunk `it` into stage s
            if (it.tile() != cur_r) {
                cur_r = it.tile();
                row = lane < kTileRows ? (int)lds32(trow + kTileRows * cur_r + lane) : -1;
                nvalid = (uint32_t)__popc(__ballot_sync(0xffffffffu, row >= 0));
                if (MULTI) {
                    const int pb = (int)lds32(tab + 4 * cur_r + 3);
                    gX = static_cast<const Tin *>(s_pp[1][pb]);
                    gY = static_cast<const Ty *>(s_pp[2][pb]);
                }
            }
            uint8_t *dst = sm + (size_t)s * stage_bytes + act_off;
            if (!it.isB) {
                const int hlo = h0 + it.i * hn, n = min(hn, h1 - hlo);
                const uint32_t rowb = (uint32_t)n * (uint32_t)sizeof(Tin);
                if (lane == 0) mbar_arrive_expect_tx(&full[s], rowb * nvalid);
                __syncwarp();
                if (row >= 0)
                    bulk_g2s(dst + (size_t)lane * hn * sizeof(Tin), gX + (size_t)row * H1 + hlo,
                             rowb, &full[s]);
            } else {
                const int jlo = j0 + it.i * JN, n = min(JN, j1 - jlo);
                const uint32_t rowb = (uint32_t)n * (uint32_t)sizeof(Ty);
                if (lane == 0) mbar_arrive_expect_tx(&full[s], rowb * nvalid);
                __syncwarp();
                if (row >= 0)
                    bulk_g2s(dst + (size_t)lane * JN * sizeof(Ty),
                             gY + (size_t)row * H2 + jlo, rowb, &full[s]);
            }
        };
        // The first `pre` chunks fill stages 0 .. pre-1 with one chunk per lane:
        // lane q requests chunk q's weights now and, after griddepcontrol.wait,
        // its x / y rows, so each phase leaves in one instruction.
        const int pre = min(nst, total);
        {
            RingIter mine;
            mine.start(nt, nA, nB);
            for (int k = 0; k < lane && k < pre; ++k) mine.next();
            const bool own = lane < pre;
            const int tile = own ? mine.tile() : 0;
            uint8_t *dst = sm + (size_t)lane * stage_bytes;
            uint64_t *bar = &full[own ? lane : 0];
            const int mp = MULTI && own ? (int)lds32(tab + 4 * tile + 3) : 0;  // the chunk's problem
            if (own) {
                const int ma = (int)lds32(tab + 4 * tile + 2);
                if (!mine.isB) {
                    const int hlo = h0 + mine.i * hn, n = min(hn, h1 - hlo);
                    const uint32_t bytes = (uint32_t)(n * rk) * (uint32_t)sizeof(Tin);
                    mbar_arrive_expect_tx(bar, bytes);
                    bulk_g2s(dst,
                             static_cast<const Tin *>(MULTI ? s_pp[0][mp] : P.A[0]) +
                                 ((size_t)ma * H1 + hlo) * rk,
                             bytes, bar);
                } else {
                    const int jlo = j0 + mine.i * JN, n = min(JN, j1 - jlo);
                    if (b4d && n >= JN) {
                        mbar_arrive_expect_tx(bar, bbox * (uint32_t)(JN / 256));
                        tma_load_4d(dst, tmb0 + mp, 0, 0, jlo >> 8, ma, bar);
                    } else {
                        const int nbox = (n + 255) >> 8;
                        mbar_arrive_expect_tx(bar, bbox * (uint32_t)nbox);
                        for (int bx = 0; bx < nbox; ++bx)
                            tma_load_3d(dst + bx * bbox, tmb0 + mp, jlo + 256 * bx, 0, ma, bar);
                    }
                }
            }
            named_sync<2, kStreamThreads>();  // the rows table is complete
            pdl_wait();
            if (own) {
                int rows_[kTileRows];
                uint32_t nv = 0;
#pragma unroll
                for (int t = 0; t < kTileRows; ++t) {
                    rows_[t] = t < trows ? (int)lds32(trow + kTileRows * tile + t) : -1;
                    nv += rows_[t] >= 0;
                }
                uint8_t *adst = dst + act_off;
                if (!mine.isB) {
                    const int hlo = h0 + mine.i * hn, n = min(hn, h1 - hlo);
                    const uint32_t rowb = (uint32_t)n * (uint32_t)sizeof(Tin);
                    mbar_arrive_expect_tx(bar, rowb * nv);
#pragma unroll
                    for (int t = 0; t < kTileRows; ++t)
                        if (rows_[t] >= 0)
                            bulk_g2s(adst + (size_t)t * hn * sizeof(Tin),
                                     static_cast<const Tin *>(MULTI ? s_pp[1][mp] : P.x[0]) +
                                         (size_t)rows_[t] * H1 + hlo,
                                     rowb, bar);
                } else {
                    const int jlo = j0 + mine.i * JN, n = min(JN, j1 - jlo);
                    const uint32_t rowb = (uint32_t)n * (uint32_t)sizeof(Ty);
                    mbar_arrive_expect_tx(bar, rowb * nv);
#pragma unroll
                    for (int t = 0; t < kTileRows; ++t)
                        if (rows_[t] >= 0)
                            bulk_g2s(adst + (size_t)t * JN * sizeof(Ty),
                                     static_cast<const Ty *>(MULTI ? s_pp[2][mp] : P.y[0]) +
                                         (size_t)rows_[t] * H2 + jlo,
                                     rowb, bar);
                }
            }
        }
        it.start(nt, nA, nB);
        for (int q = 0; q < pre; ++q) it.next();
        for (int q = pre, s = pre % nst; q < total; ++q, it.next()) {
            if (!mbar_wait(&empty[s], (uint32_t)((q / nst - 1) & 1))) set_error(err, kErrTimeout);
            __syncwarp();
            issue_w(s);
            issue_act(s);
            if (++s == nst) s = 0;
        }
        if (ncl > 1) cluster_wait();
    } else {
        // ---- compute warps -------------------------------------------------
        // Physical rows of the tiles; invalid perm entries are skipped and reported.
        for (int e = tid; e < nt * kTileRows; e += kStreamConsumers) {
            const int m = e / kTileRows, t = e % kTileRows;
            int row = -1;
            if (t < tab[4 * m + 1]) {
                const int p = tab[4 * m] + t;
                row = GROUPED ? g_sperm[p] : (P.perm ? P.perm[p] : p);
                if (row < 0 || row >= T) {
                    if (rank == 0) set_error(err, kErrBadIndex);
                    row = -1;
                }
            }
            trow[e] = row;
        }
        named_sync<2, kStreamThreads>();
        pdl_wait();  // y is written below: only after the previous kernel
        if (meta_out) write_meta();
        if (ncl > 1) cluster_wait();  // every CTA of the cluster has started
        bool lost = false;
        int q = 0;
        float4 part;  // elements (t, 4q .. 4q+3) of this CTA's partial v, tid = t * (rk/4) + q
        for (int m = 0; m <= nt; ++m) {
            if (m < nt) {
                const int n = (int)lds32(tab + 4 * m + 1);
                if (n <= 1)
                    stream_shrink<Tin, RK, 1, CW>(sm, stage_bytes, act_off, nst, q, nA, h1 - h0, hn, rk,
                                              full, empty, red, lost, err, inject);
                else if (n <= 2)
                    stream_shrink<Tin, RK, 2, CW>(sm, stage_bytes, act_off, nst, q, nA, h1 - h0, hn, rk,
                                              full, empty, red, lost, err, inject);
                else if (n <= 4)
                    stream_shrink<Tin, RK, 4, CW>(sm, stage_bytes, act_off, nst, q, nA, h1 - h0, hn, rk,
                                              full, empty, red, lost, err, inject);
                else
                    stream_shrink<Tin, RK, 8, CW>(sm, stage_bytes, act_off, nst, q, nA, h1 - h0, hn, rk,
                                              full, empty, red, lost, err, inject);
                consumers_sync<CW>();
                // this CTA's partial of v, four consecutive k per thread
                part = make_float4(0.f, 0.f, 0.f, 0.f);
                if (tid < n * (rk / 4)) {
                    const int t = tid / (rk / 4), k = 4 * (tid - t * (rk / 4));
#pragma unroll
                    for (int w = 0; w < kStreamWarps; ++w) {
                        const uint4 u = lds128(red + (w * kTileRows + t) * RK + k);
                        part.x += __uint_as_float(u.x);
                        part.y += __uint_as_float(u.y);
                        part.z += __uint_as_float(u.z);
                        part.w += __uint_as_float(u.w);
                    }
                    if (ncl == 1)
                        sts128(s_v + ((m & 1) * kTileRows + t) * RK + k,
                               make_uint4(__float_as_uint(part.x), __float_as_uint(part.y),
                                          __float_as_uint(part.z), __float_as_uint(part.w)));
                }
            }
            if (ncl > 1) {
                if (m >= 1) {
                    // v of tile m-1: every CTA's partial has arrived
                    const int b = (m - 1) & 1;
                    if (!mbar_wait_cluster(&vfull[b], (uint32_t)(((m - 1) >> 1) & 1))) {
                        set_error(err, kErrTimeout);
                        mbar_wait_cluster(&vfull[b], (uint32_t)(((m - 1) >> 1) & 1));
                        lost = true;
                    }
                    const int n1 = (int)lds32(tab + 4 * (m - 1) + 1);
                    for (int e = tid; e < n1 * rk; e += kStreamConsumers) {
                        const int t = e / rk, k = e - (e / rk) * rk;
                        float sum = 0.f;
                        for (int c = 0; c < ncl; ++c)
                            sum += ldsf(recv + ((b * ncl + c) * kTileRows + t) * RK + k);
                        stsf(s_v + (b * kTileRows + t) * RK + k, sum);
                    }
                }
                if (m < nt) {
                    // Push this CTA's partial of tile m into slot (m & 1, rank)
                    // of every CTA with st.async, which counts the bytes on
                    // the owner's vfull[m & 1]; each CTA expects ncl partials.
                    // The slot was last read for tile m-2: its owner had read
                    // it (and passed the barrier below) before pushing tile
                    // m-1, which the wait above saw.
                    const int b = m & 1;
                    const int n = (int)lds32(tab + 4 * m + 1);
                    consumers_sync<CW>();  // this CTA's reads of its own slots are done
                    if (tid == 0)
                        mbar_arrive_expect_tx(&vfull[b], (uint32_t)(ncl * n * rk) * 4u);
                    if (tid < n * (rk / 4)) {
                        const int t = tid / (rk / 4), k = 4 * (tid - t * (rk / 4));
                        float *slot = recv + ((b * ncl + rank) * kTileRows + t) * RK + k;
                        for (int c = 0; c < ncl; ++c)
                            st_async4(peer_addr(slot, (uint32_t)c), part.x, part.y, part.z, part.w,
                                      peer_addr(&vfull[b], (uint32_t)c));
                    }
                }
            }
            consumers_sync<CW>();  // s_v of tile m-1 is complete
            if (m >= 1) {
                const int mm = m - 1;
                const int n = (int)lds32(tab + 4 * mm + 1);
                int row[kTileRows];
#pragma unroll
                for (int t = 0; t < kTileRows; ++t) row[t] = (int)lds32(trow + kTileRows * mm + t);
                const float *sv = s_v + (mm & 1) * kTileRows * RK;
                Ty *gY = static_cast<Ty *>(
                    MULTI ? const_cast<void *>(s_pp[2][(int)lds32(tab + 4 * mm + 3)]) : P.y[0]);
                if (n <= 1)
                    stream_expand<Tin, Ty, RK, 1, CW>(sm, stage_bytes, act_off, nst, q, nB, j1 - j0, j0,
                                                  rk, sv, row, gY, H2, scale, full, empty, lost, err);
                else if (n <= 2)
                    stream_expand<Tin, Ty, RK, 2, CW>(sm, stage_bytes, act_off, nst, q, nB, j1 - j0, j0,
                                                  rk, sv, row, gY, H2, scale, full, empty, lost, err);
                else if (n <= 4)
                    stream_expand<Tin, Ty, RK, 4, CW>(sm, stage_bytes, act_off, nst, q, nB, j1 - j0, j0,
                                                  rk, sv, row, gY, H2, scale, full, empty, lost, err);
                else
                    stream_expand<Tin, Ty, RK, 8, CW>(sm, stage_bytes, act_off, nst, q, nB, j1 - j0, j0,
                                                  rk, sv, row, gY, H2, scale, full, empty, lost, err);
            }
        }
    }
    // No closing cluster barrier: the only accesses to another CTA's shared
    // memory are the st.async pushes of partial v, and every CTA waits for all
    // pushes addressed to it (its vfull barriers) before it gets here.
}

// ---- host-side launcher for one input type ----------------------------------
template <typename Tin, typename Ty, int RK>
static void *stream_pick(bool grouped, int cw, bool multi) {
    if (grouped) return (void *)sgmv_stream_kernel<Tin, Ty, RK, true, 8>;
    if (multi) return (void *)sgmv_stream_kernel<Tin, Ty, RK, false, 16, true>;
    return cw == 16 ? (void *)sgmv_stream_kernel<Tin, Ty, RK, false, 16>
                    : (void *)sgmv_stream_kernel<Tin, Ty, RK, false, 8>;
}

template <typename Tin, typename Ty>
static void *stream_pick_rk(int rk, bool grouped, int cw, bool multi) {
    switch (rk) {
        case 16: return stream_pick<Tin, Ty, 16>(grouped, cw, multi);
        case 32: return stream_pick<Tin, Ty, 32>(grouped, cw, multi);
        default: return stream_pick<Tin, Ty, 64>(grouped, cw, multi);
    }
}

template <typename Tin>
static int stream_launch_impl(const StreamLaunch &l) {
    void *fn;
    switch (l.y_dtype) {
        case 0: fn = stream_pick_rk<Tin, __half>(l.rk, l.grouped, l.cw, l.multi); break;
        case 1: fn = stream_pick_rk<Tin, __nv_bfloat16>(l.rk, l.grouped, l.cw, l.multi); break;
        default: fn = stream_pick_rk<Tin, float>(l.rk, l.grouped, l.cw, l.multi); break;
    }
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)l.p.smem_bytes);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)l.p.cl, (unsigned)l.p.G, 1);
    cfg.blockDim = dim3((unsigned)(l.cw * 32 + 32), 1, 1);
    cfg.dynamicSmemBytes = l.p.smem_bytes;
    cfg.stream = l.stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (l.p.cl > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)l.p.cl;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = (unsigned)na;
    if (l.multi) {
        void *args[] = {(void *)&l.p};
        return (int)cudaLaunchKernelExC(&cfg, fn, args);
    }
    // one problem: the smaller parameter block of that instantiation
    StreamParams1 p1;
    static_cast<StreamCommon &>(p1) = static_cast<const StreamCommon &>(l.p);
    p1.tmap_b[0] = l.p.tmap_b[0];
    p1.y[0] = l.p.y[0];
    p1.x[0] = l.p.x[0];
    p1.A[0] = l.p.A[0];
    p1.B[0] = l.p.B[0];
    void *args[] = {(void *)&p1};
    return (int)cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace sgmv
