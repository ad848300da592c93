// sgmv_cc.cuh -- CUDA-core SGMV kernels for decode-sized segments.
//
// Method ("Punica: when LoRA fine-tuned models need multi-tenant serving",
// omica.com.cn article, §2.2): for every row of a segment, shrink
// v = x . A[idx] (A gathered out of the stacked adapters), then expand
// y += scale * v . B[idx].  Both steps stream one adapter's weights and do
// about one flop per byte, so they are bound by HBM bandwidth and run on the
// CUDA cores; the tensor-core path takes long segments.
//
// Work decomposition (one launch, no device-memory intermediate in kFused):
//   * a tile is up to kRowsMax consecutive rows of one segment; tiles are
//     numbered on the device from seg_ptr (grid.y = tile slot), so the same
//     kernel serves metadata built on the host or on the device;
//   * the CL CTAs of one tile form a thread-block cluster; CTA c owns the
//     H1 slice [c*hc, (c+1)*hc) for the shrink and the H2 slice [c*jc, ...)
//     for the expand;
//   * each CTA issues 1-D bulk (TMA) copies of its A slice (one contiguous
//     block), its B slice (r rows) and the tile's X rows into shared memory,
//     all at kernel start, so the whole working set is in flight at once;
//   * partial v from the CTA's H1 slice is summed over the cluster through
//     distributed shared memory in a fixed order (deterministic, identical in
//     every CTA), then each CTA expands its H2 slice and updates y in place.
// Programmatic dependent launch: A, B and the segment metadata are requested
// before griddepcontrol.wait; x, y and v only after it.
#pragma once

#include "sgmv_device.cuh"
#include "sgmv_internal.h"
#include "sgmv_tiles.cuh"

namespace sgmv {

template <typename Tin, typename Ty, int RMAX, int MODE>
__global__ void __launch_bounds__(kThreads) sgmv_cc_kernel(const __grid_constant__ CCParams P) {
    // Kernel parameters, read once into registers: touching the parameter
    // struct inside loops or lambdas makes the compiler address it in memory
    // and reload its fields on every use.
    const int nseg = P.S, nrows_all = P.T, nadapters = P.L, H1 = P.H1, H2 = P.H2, rk = P.r;
    const int tile_rows = P.rows, hc = P.hc, jc = P.jc, hs = P.hs, js = P.js;
    const int ax_stages = P.ax_stages, b_stages = P.b_stages, ncl = P.cl;
    const int min_len = P.min_len, max_len = P.max_len, y_pref_on = P.y_pref;
    const float scale = P.scale;
    int *const err = P.err;
    const int32_t *const perm = P.perm;
    const int32_t *const seg_ptr = P.seg_ptr;
    const int32_t *const idx = P.idx;
    const float *const v_in = P.v_in;
    float *const v_out = P.v_out;
    const void *const xptr = P.x;
    const void *const Aptr = P.A;
    const void *const Bptr = P.B;
    void *const yptr = P.y;
    const CCSmem lay = cc_smem_layout(P, (int)sizeof(Tin), MODE);

    extern __shared__ __align__(128) uint8_t dsmem[];
    // 0,1: (A, X) stages, two arrivals each (A, then X); 2,3: B stages; 4: y rows
    __shared__ __align__(8) uint64_t bars[5];
    __shared__ int s_info[4];
    __shared__ int s_row[kRowsMax];
    __shared__ __align__(16) float s_v[kRowsMax * RMAX];
    __shared__ float s_red[(MODE == kExpand) ? 1 : kRowsMax * RMAX * (kThreads / (RMAX / 16)) / 32];
    constexpr int kKeys = MODE == kGrouped ? kGroupMaxT : 1;
    __shared__ int s_key[kKeys], s_cnt[kKeys], s_rank[kKeys];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const bool report = blockIdx.x == 0 && blockIdx.y == 0;

    // kGrouped: this thread's row (t = tid) in the stable grouping by adapter id
    int g_key = -1, g_less = 0, g_rank = 0, g_dless = 0, g_nseg = 0;
    if (MODE == kGrouped) {
        // Every CTA groups the batch itself (T <= kGroupMaxT): no metadata to
        // read from device memory and no separate grouping launch.  Sorted
        // position of row t = (#rows with a smaller id) + (#earlier rows with
        // the same id); tiles are numbered over ids in ascending order.
        const int32_t *ra = P.row_adapter;
        if (tid < nrows_all) {
            g_key = ra[tid];
            if (g_key < -1 || g_key >= nadapters) {
                if (report) set_error(err, kErrBadIndex);
                g_key = -1;
            }
            s_key[tid] = g_key;
        }
        if (tid == 0) {
            s_info[0] = -1;
            mbar_init(&bars[0], 2);
            mbar_init(&bars[1], 2);
            mbar_init(&bars[2], 1);
            mbar_init(&bars[3], 1);
            mbar_init(&bars[4], 1);
            mbar_init_fence();
        }
        __syncthreads();
        int cnt = 0;
        if (tid < nrows_all) {
            for (int u = 0; u < nrows_all; ++u) {
                const int ku = s_key[u];
                g_less += ku < g_key;
                cnt += ku == g_key;
                g_rank += (ku == g_key) & (u < tid);
            }
            s_cnt[tid] = cnt;
            s_rank[tid] = g_rank;
        }
        __syncthreads();
        if (tid < nrows_all) {
            int tb = 0;  // tiles of the adapters with a smaller id
            for (int u = 0; u < nrows_all; ++u) {
                const int ku = s_key[u];
                if (s_rank[u] == 0 && ku < g_key) {
                    ++g_dless;
                    if (ku >= 0) tb += (s_cnt[u] + kRowsMax - 1) / kRowsMax;
                }
            }
            if (g_key >= 0 && tb + g_rank / kRowsMax == (int)blockIdx.y) {
                const int slot = g_rank % kRowsMax;
                s_row[slot] = tid;
                if (slot == 0) {
                    s_info[0] = 0;
                    s_info[1] = g_less + g_rank;
                    s_info[2] = min(kRowsMax, cnt - g_rank);
                    s_info[3] = g_key;
                }
            }
        }
        g_nseg = __syncthreads_count(tid < nrows_all && g_rank == 0);
    } else {
        if (tid < 32) {
            find_tile(seg_ptr, idx, nseg, nrows_all, nadapters, tile_rows, min_len, max_len, err,
                      blockIdx.y, MODE == kShrink, report, s_info);
            if (tid == 0) {
                mbar_init(&bars[0], 2);
                mbar_init(&bars[1], 2);
                mbar_init(&bars[2], 1);
                mbar_init(&bars[3], 1);
                mbar_init(&bars[4], 1);
                mbar_init_fence();
            }
        }
        __syncthreads();
    }
    if (MODE == kGrouped && report && P.perm_out) {
        // CTA (0,0) writes the grouping out for later calls: after the
        // previous kernel on the stream, which may still read these arrays.
        pdl_wait();
        if (tid < nrows_all) {
            P.perm_out[g_less + g_rank] = tid;
            if (g_rank == 0) {
                P.seg_out[g_dless] = g_less;
                P.idx_out[g_dless] = g_key;
            }
        }
        if (tid == 0) {
            P.seg_out[g_nseg] = nrows_all;
            *P.S_out = g_nseg;
        }
        for (int sidx = g_nseg + tid; sidx < P.S_max; sidx += kThreads) {
            P.idx_out[sidx] = -1;
            P.seg_out[sidx + 1] = nrows_all;
        }
    }
    if (s_info[0] < 0) return;  // no tile for this slot (same for the whole cluster)
    const int p0 = s_info[1];
    const int nrows = s_info[2];
    const int a = s_info[3];

    if (MODE == kShrink && a < 0) {  // no adapter: v = 0 for these rows
        pdl_wait();
        pdl_trigger();
        if (blockIdx.x == 0)
            for (int e = tid; e < nrows * rk; e += kThreads)
                v_out[(size_t)(p0 + e / rk) * rk + e % rk] = 0.f;
        return;
    }
    const bool clustered = MODE != kExpand && ncl > 1;
    if (clustered) cluster_arrive_relaxed();  // waited on just before the first peer access

    const Tin *gA = static_cast<const Tin *>(Aptr);
    const Tin *gB = static_cast<const Tin *>(Bptr);
    const Tin *gX = static_cast<const Tin *>(xptr);
    Ty *gY = static_cast<Ty *>(yptr);

    // Slices owned by this CTA.
    int h0 = 0, h1 = 0, j0 = 0, j1 = 0;
    if (MODE != kExpand) {
        h0 = min(H1, (int)blockIdx.x * hc);
        h1 = min(H1, h0 + hc);
    }
    if (MODE != kShrink) {
        j0 = min(H2, (int)blockIdx.x * jc);
        j1 = min(H2, j0 + jc);
    }
    const int nA = (MODE != kExpand && h1 > h0) ? (h1 - h0 + hs - 1) / hs : 0;
    const int nB = (MODE != kShrink && j1 > j0) ? (j1 - j0 + js - 1) / js : 0;
    const bool y_pref = MODE != kShrink && y_pref_on && nB > 0;

    auto ax_buf = [&](int st) {
        return reinterpret_cast<Tin *>(dsmem + lay.ax_off + st * lay.ax_stage_bytes);
    };
    auto b_buf = [&](int st) {
        return reinterpret_cast<Tin *>(dsmem + lay.b_off + st * lay.b_stage_bytes);
    };
    Ty *ybuf = reinterpret_cast<Ty *>(dsmem + lay.y_off);
    float *recv = reinterpret_cast<float *>(dsmem + lay.recv_off);

    // Chunk i of A: first of the two arrivals on its stage barrier.
    auto issue_a = [&](int i) {  // lane 0 of warp 0
        const int st = i % ax_stages;
        const int hlo = h0 + i * hs;
        const int hn = min(hs, h1 - hlo);
        const uint32_t ab = (uint32_t)(hn * rk) * sizeof(Tin);
        mbar_arrive_expect_tx(&bars[st], ab);
        bulk_g2s(ax_buf(st), gA + ((size_t)a * H1 + hlo) * rk, ab, &bars[st]);
    };
    // Chunk i of the tile's X rows: second arrival.  Needs s_row and nvalid.
    auto issue_x = [&](int i, int nvalid) {  // all lanes of warp 0
        const int st = i % ax_stages;
        const int hlo = h0 + i * hs;
        const int hn = min(hs, h1 - hlo);
        if (lane == 0) mbar_arrive_expect_tx(&bars[st], (uint32_t)(nvalid * hn) * sizeof(Tin));
        __syncwarp();
        Tin *xs = ax_buf(st) + hs * rk;
        if (lane < nrows && s_row[lane] >= 0)
            bulk_g2s(xs + lane * hs, gX + (size_t)s_row[lane] * H1 + hlo,
                     (uint32_t)hn * sizeof(Tin), &bars[st]);
    };
    auto issue_b = [&](int i) {  // all lanes of warp 0
        const int st = i % b_stages;
        const int jlo = j0 + i * js;
        const int jn = min(js, j1 - jlo);
        if (lane == 0) mbar_arrive_expect_tx(&bars[2 + st], (uint32_t)(rk * jn) * sizeof(Tin));
        __syncwarp();
        for (int k = lane; k < rk; k += 32)
            bulk_g2s(b_buf(st) + k * js, gB + ((size_t)a * rk + k) * H2 + jlo,
                     (uint32_t)jn * sizeof(Tin), &bars[2 + st]);
    };

    // Weights first: they do not depend on the previous kernel on the stream,
    // and nothing waits for the row permutation before they are requested.
    if (tid < 32) {
        if (lane == 0)
            for (int i = 0; i < min(nA, ax_stages); ++i) issue_a(i);
        for (int i = 0; i < min(nB, b_stages); ++i) issue_b(i);
    } else if (MODE != kGrouped && tid < 32 + nrows) {
        // Physical rows of the tile; invalid perm entries are skipped and reported.
        const int t = tid - 32;
        int row = perm ? perm[p0 + t] : p0 + t;
        if (row < 0 || row >= nrows_all) {
            set_error(err, kErrBadIndex);
            row = -1;
        }
        s_row[t] = row;
    }
    pdl_wait();
    __syncthreads();
    unsigned vmask = 0;  // tile rows with a valid physical row
    int nvalid = 0;
#pragma unroll
    for (int t = 0; t < kRowsMax; ++t)
        if (t < nrows && s_row[t] >= 0) {
            vmask |= 1u << t;
            ++nvalid;
        }
    // Activations and outputs: only after the previous kernel has finished.
    if (tid < 32) {
        for (int i = 0; i < min(nA, ax_stages); ++i) issue_x(i, nvalid);
        if (y_pref) {
            const uint32_t yb = (uint32_t)(j1 - j0) * sizeof(Ty);
            if (lane == 0) mbar_arrive_expect_tx(&bars[4], yb * nvalid);
            __syncwarp();
            if (lane < nrows && s_row[lane] >= 0)
                bulk_g2s(ybuf + lane * jc, gY + (size_t)s_row[lane] * H2 + j0, yb, &bars[4]);
        }
    }
    pdl_trigger();

    bool lost = false;  // a bounded wait ran out: this thread writes nothing
    // Every thread polls the mbarrier itself: no CTA barrier per wait.
    auto cta_wait = [&](uint64_t *bar, uint32_t par) {
        if (!mbar_wait(bar, par)) {
            set_error(err, kErrTimeout);
            mbar_wait(bar, par);
            lost = true;
        }
    };
    if (MODE == kExpand) {
        for (int e = tid; e < nrows * rk; e += kThreads) {
            const int t = e / rk, k = e - (e / rk) * rk;
            s_v[t * RMAX + k] = v_in[(size_t)(p0 + t) * rk + k];
        }
    } else {
        // ---- shrink: partial v over this CTA's H1 slice -----------------
        // Thread -> (k-group of 16 columns of r, h-group); each thread reads
        // two 16-byte vectors of A per h and one X value per row, and the
        // 32 h-groups of a warp are summed by a reduce-scatter butterfly.
        constexpr int KG = RMAX / 16;        // k-groups: 1, 2, 4, 8
        constexpr int HG = kThreads / KG;    // h-groups per k-group (>= 32)
        constexpr int WPG = HG / 32;         // warps per k-group
        const int kg = tid / HG, hg = tid - (tid / HG) * HG;
        const int kbase = kg * 16;
        const int wig = hg >> 5;             // warp within the k-group
        const bool kact = kbase < rk;       // same for the whole warp
        const bool vec = (rk & 7) == 0;     // A rows are 16-byte aligned in smem
        for (int i = 0; i < nA; ++i) {
            const int st = i % ax_stages;
            const uint32_t par = (uint32_t)((i / ax_stages) & 1);
            cta_wait(&bars[st], par);
            const int hn = min(hs, h1 - (h0 + i * hs));
            const Tin *As = ax_buf(st);
            const Tin *Xs = As + hs * rk;
            if (kact) {
                for (int t = 0; t < nrows; ++t) {
                    if (!(vmask & (1u << t))) continue;
                    float acc[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
                    for (int h = hg; h < hn; h += HG) {
                        const unsigned short xb = lds16(Xs + t * hs + h);
                        const float x = to_f<Tin>(*reinterpret_cast<const Tin *>(&xb));
                        float av[16];
                        const Tin *arow = As + h * rk + kbase;
                        if (vec) {
                            float lo[8], hi[8];
                            unpack8<Tin>(lds128(arow), lo);
                            unpack8<Tin>(lds128(arow + 8), hi);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                av[j] = lo[j];
                                av[8 + j] = hi[j];
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const unsigned short ab = kbase + j < rk ? lds16(arow + j) : 0;
                                av[j] = to_f<Tin>(*reinterpret_cast<const Tin *>(&ab));
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[j] = fmaf(x, av[j], acc[j]);
                    }
                    // reduce-scatter over the warp: lane l ends with k = kbase + l/2
#pragma unroll
                    for (int half = 8; half >= 1; half >>= 1) {
                        const bool upper = (lane & (half * 2)) != 0;
#pragma unroll
                        for (int j = 0; j < half; ++j) {
                            const float keep = upper ? acc[half + j] : acc[j];
                            const float give = upper ? acc[j] : acc[half + j];
                            acc[j] = keep + __shfl_xor_sync(0xffffffffu, give, half * 2);
                        }
                    }
                    acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 1);
                    if ((lane & 1) == 0) {
                        float *dst = &s_red[(t * RMAX + kbase + (lane >> 1)) * WPG + wig];
                        *dst = i == 0 ? acc[0] : *dst + acc[0];
                    }
                }
            }
            __syncthreads();
            if (tid < 32 && i + ax_stages < nA) {
                if (lane == 0) issue_a(i + ax_stages);
                __syncwarp();
                issue_x(i + ax_stages, nvalid);
            }
        }
        // This CTA's partial of v[t][k]: the warps of the k-group summed in order.
        auto partial = [&](int t, int kk) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < WPG; ++w) s += s_red[(t * RMAX + kk) * WPG + w];
            return s;
        };
        if (clustered) {
            // Push the partial into slot `rank` of every CTA's receive buffer,
            // then sum the slots locally in rank order: the same bits in every
            // CTA, one cluster barrier, no remote loads.
            const int rank = (int)blockIdx.x;
            const int per = nrows * rk;
            cluster_wait();
            for (int e = tid; e < ncl * per; e += kThreads) {
                const int c = e / per, rem = e - (e / per) * per;
                const int t = rem / rk, kk = rem - (rem / rk) * rk;
                st_peer(peer_addr(&recv[(rank * kRowsMax + t) * RMAX + kk], (uint32_t)c),
                        partial(t, kk));
            }
            cluster_sync();
            for (int e = tid; e < per; e += kThreads) {
                const int t = e / rk, kk = e - (e / rk) * rk;
                float s = 0.f;
                for (int c = 0; c < ncl; ++c) s += ldsf(recv + (c * kRowsMax + t) * RMAX + kk);
                s_v[t * RMAX + kk] = s;
            }
        } else {
            for (int e = tid; e < nrows * rk; e += kThreads) {
                const int t = e / rk, kk = e - (e / rk) * rk;
                s_v[t * RMAX + kk] = partial(t, kk);
            }
        }
        if (MODE == kShrink) {
            if (blockIdx.x == 0 && !lost)
                for (int e = tid; e < nrows * rk; e += kThreads) {
                    const int t = e / rk, kk = e - (e / rk) * rk;
                    v_out[(size_t)(p0 + t) * rk + kk] = s_v[t * RMAX + kk];
                }
            return;
        }
    }
    __syncthreads();
    if (y_pref) cta_wait(&bars[4], 0);

    // ---- expand: y[row, j] += scale * v . B[a][:, j] for this CTA's slice ----
    // Each thread owns two adjacent columns and runs the whole r-sum, so a
    // warp reads 128 contiguous bytes of a B row per step (no bank conflicts)
    // and writes 128 contiguous bytes of y.
    for (int i = 0; i < nB; ++i) {
        const int st = i % b_stages;
        cta_wait(&bars[2 + st], (uint32_t)((i / b_stages) & 1));
        const int jlo = j0 + i * js;
        const int npair = min(js, j1 - jlo) >> 1;
        const Tin *Bs = b_buf(st);
        if (!lost) {
            for (int t = 0; t < nrows; ++t) {
                const int row = s_row[t];
                if (row < 0) continue;
                const float *vt = s_v + t * RMAX;
                for (int cp = tid; cp < npair; cp += kThreads) {
                    float a0 = 0.f, a1 = 0.f;
                    const Tin *bcol = Bs + 2 * cp;
#pragma unroll 4
                    for (int kk = 0; kk < rk; ++kk) {
                        const float vk = ldsf(vt + kk);
                        float b0, b1;
                        unpack2<Tin>(lds32(bcol + kk * js), b0, b1);
                        a0 = fmaf(vk, b0, a0);
                        a1 = fmaf(vk, b1, a1);
                    }
                    Ty *yp = gY + (size_t)row * H2 + jlo + 2 * cp;
                    float y0, y1;
                    if (y_pref)
                        lds2<Ty>(ybuf + t * jc + (jlo - j0) + 2 * cp, y0, y1);
                    else
                        ld2<Ty>(yp, y0, y1);
                    st2<Ty>(yp, fmaf(scale, a0, y0), fmaf(scale, a1, y1));
                }
            }
        }
        if (i + b_stages < nB) {  // the stage is refilled: everyone is done with it
            __syncthreads();
            if (tid < 32) issue_b(i + b_stages);
        }
    }
}

// ---- host-side launcher for one input type ----------------------------------
template <typename Tin, typename Ty, int RMAX>
static void *pick_mode(int mode) {
    switch (mode) {
        case kFused: return (void *)sgmv_cc_kernel<Tin, Ty, RMAX, kFused>;
        case kExpand: return (void *)sgmv_cc_kernel<Tin, Ty, RMAX, kExpand>;
        case kGrouped: return (void *)sgmv_cc_kernel<Tin, Ty, RMAX, kGrouped>;
        default: return (void *)sgmv_cc_kernel<Tin, float, RMAX, kShrink>;
    }
}

template <typename Tin, typename Ty>
static void *pick_rmax(int mode, int rmax) {
    switch (rmax) {
        case 16: return pick_mode<Tin, Ty, 16>(mode);
        case 32: return pick_mode<Tin, Ty, 32>(mode);
        case 64: return pick_mode<Tin, Ty, 64>(mode);
        default: return pick_mode<Tin, Ty, 128>(mode);
    }
}

template <typename Tin>
static int cc_launch_impl(const CCLaunch &l) {
    void *fn;
    switch (l.y_dtype) {
        case 0: fn = pick_rmax<Tin, __half>(l.mode, l.rmax); break;
        case 1: fn = pick_rmax<Tin, __nv_bfloat16>(l.mode, l.rmax); break;
        default: fn = pick_rmax<Tin, float>(l.mode, l.rmax); break;
    }
    const CCSmem lay = cc_smem_layout(l.p, (int)sizeof(Tin), l.mode);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lay.total);
    if (e != cudaSuccess) return (int)e;
    if (l.cluster > 8) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return (int)e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = l.grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = lay.total;
    cfg.stream = l.stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (l.cluster > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)l.cluster;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (l.pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = (unsigned)na;
    void *args[] = {(void *)&l.p};
    return (int)cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace sgmv
