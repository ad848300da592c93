// sgmv_fused.cu -- the LoRA layer in one pass over its weights: the base
// linear layer and every row's adapter update together,
//
//     y[t, :] = x[t, :] . W  +  scale * (x[t, :] . A[a_t]) . B[a_t]
//
// ("Punica: when LoRA fine-tuned models need multi-tenant serving",
// omica.com.cn article, §2.1: a LoRA layer computes y = xW + xAB; "How to
// deploy several LoRA adapters without reloading the base model (Punica,
// S-LoRA)?", aivaro.ru, §3.2 "Fused Kernel": the LoRA transform merged into
// the base model's linear layer so that memory is read fewer times).
//
// For decode batches (T <= 128 rows) the layer is a stream over W (H1 x H2)
// and the adapters' B slices with little arithmetic per byte.  After the
// shrink v = x . A[a] (a CUDA-core launch of its own, writing v to a small
// workspace), this kernel makes every output element of y once, on the
// tensor cores, in the transposed ("swap AB") form that suits few rows:
//
//   D[j, t] = sum_h W[h, j] x[t, h]  +  sum over segments s of
//             sum_k B[a_s][k, j] (scale v[t, k] if row t is in s, else 0)
//
// with M = 128 columns j of W per tile (W and B tiles are MN-major A
// operands, loaded by TMA with 128-byte swizzle), N = the batch's rows
// rounded up to 16 (x rows are the K-major B operand) and fp32 accumulation
// in tensor memory.  The LoRA terms are extra MMAs over blocks of up to 64
// rows: for every (segment, 64-row block) pair with a row in both, B[a]^T
// times a tile of scale * v that is zero outside the segment, as two 16-bit
// halves (hi = round(scale v), lo = round(scale v - hi)) so v keeps about 16
// significant bits.  The whole layer -- base and LoRA -- is one accumulation,
// rounded once to y's type.  Accumulator addresses stay at multiples of 64
// columns and accumulator reads at multiples of 32 (the placements the other
// tensor-core kernels here use).
//
// Decomposition: one tile of 128 columns per cluster of CL CTAs; CTA `rank`
// takes an even share of H1's 64-column k-blocks and every CL-th LoRA pair,
// so all CTAs stream about the same bytes.  The partial accumulators are
// exchanged through distributed shared memory (each CTA owns every CL-th
// group of 32 rows of the tile) and summed in rank order: deterministic.
//
// Warps: 0-3 read the accumulator (one TMEM lane, i.e. one column j, per
// thread) and write y; lane 0 of warp 0 also issues the MMAs; warp 4 fills
// the ring in order: TMA loads (W before griddepcontrol.wait, x after it)
// and the v tiles (v is written by the shrink launched just before).  Each
// barrier has one waiting role that takes its phases in order.  Every
// mbarrier wait is bounded.
#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "sgmv_device.cuh"
#include "sgmv_internal.h"
#include "sgmv_tcgen05.cuh"

namespace sgmv {
namespace {

constexpr int kFusedThreads = 160;
constexpr int kFusedCols = 128;               // columns of W per tile (M of every MMA)
constexpr int kFusedMaxStages = 8;
constexpr uint32_t kFusedStage = 32768;       // bytes of one ring stage
constexpr uint32_t kFusedXOff = 16384;        // x tile, or the v tiles, at this offset
constexpr uint32_t kFusedVloOff = kFusedXOff + 8192;  // v tiles hold up to 64 rows
constexpr uint32_t kFusedWBytes = 2u * 64u * 128u;  // two 64-column halves of a k-block of W

struct FusedParams {
    CUtensorMap tmap_w;  // W as [H1][H2], box {64, 64}, 128-byte swizzle
    CUtensorMap tmap_x;  // x as [T][H1], box {64, npad}
    CUtensorMap tmap_b;  // B as [L][r][H2], box {64, r16, 1}
    void *y;
    const float *v;      // [T][r] fp32 by sorted position
    const int32_t *perm, *seg_ptr, *idx;
    int *err;
    int32_t S, T, L, H1, H2, r;
    int32_t r16;   // r rounded up to 16 (K of the LoRA MMAs)
    int32_t npad;  // T rounded up to 16 (N of the base MMAs)
    int32_t cl;    // CTAs per cluster (split of H1)
    int32_t kbt;   // 64-column k-blocks of H1
    int32_t nst;   // ring stages
    uint32_t tmem_cols;
    float scale;
};

template <typename Tin, typename Ty>
__global__ void __launch_bounds__(kFusedThreads, 1)
    sgmv_fused_kernel(const __grid_constant__ FusedParams P) {
    const int T = P.T, S = P.S, L = P.L, H2 = P.H2, r = P.r, r16 = P.r16, npad = P.npad;
    const int C = P.cl, kbt = P.kbt, nst = P.nst;
    const float scale = P.scale;
    int *const err = P.err;
    const int32_t *const seg_ptr = P.seg_ptr;
    const int32_t *const idx = P.idx;
    const int32_t *const perm = P.perm;

    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[kFusedMaxStages], empty[kFusedMaxStages], done, red_full;
    __shared__ int s_rowseg[128];   // segment of physical row t (-1: no adapter)
    __shared__ int s_rowpos[128];   // its sorted position
    __shared__ int s_pseg[128];     // LoRA pairs: segment ...
    __shared__ int s_pblk[128];     // ... and 64-row block
    __shared__ int s_npairs, s_lost, s_wcnt[4];
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)blockIdx.x;
    const int j0 = (int)blockIdx.y * kFusedCols;
    const bool report = rank == 0 && blockIdx.y == 0;

    // The next kernel on the stream may start now: it reads nothing this one
    // writes before its own griddepcontrol.wait.
    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 2);   // base: W + x copies; LoRA: B copy + the v tiles
            mbar_init(&empty[s], 1);  // the MMAs that read the stage are done
        }
        mbar_init(&done, 1);
        mbar_init(&red_full, 1);
        mbar_init_fence();
        s_lost = 0;
    }
    if (tid < 128) {
        s_rowseg[tid] = -1;
        s_rowpos[tid] = 0;
    }
    __syncthreads();
    // Rows of every segment with an adapter (segment metadata may be read
    // before the wait).  Bad segments and ids are skipped and reported.
    for (int s = tid; s < S; s += kFusedThreads) {
        const int b = seg_ptr[s], e = seg_ptr[s + 1], a = idx[s];
        if (b < 0 || e < b || e > T) {
            if (report) set_error(err, kErrBadSegments);
            continue;
        }
        if (e == b || a == -1) continue;
        if (a < -1 || a >= L) {
            if (report) set_error(err, kErrBadIndex);
            continue;
        }
        for (int p = b; p < e; ++p) {
            const int row = perm ? perm[p] : p;
            if (row < 0 || row >= T) {
                if (report) set_error(err, kErrBadIndex);
                continue;
            }
            s_rowseg[row] = s;
            s_rowpos[row] = p;
        }
    }
    __syncthreads();
    if (warp == 0) tmem_alloc(&s_tmem, P.tmem_cols);  // a converged warp, as the instruction needs
    // LoRA pairs: (segment, 64-row block) with a row in both, one per row t
    // that is its segment's first row in its block, in order of t
    int first = 0;
    if (tid < T) {
        const int sg = s_rowseg[tid];
        if (sg >= 0) {
            first = 1;
            for (int u = tid & ~63; u < tid; ++u)
                if (s_rowseg[u] == sg) {
                    first = 0;
                    break;
                }
        }
    }
    const unsigned fb = warp < 4 ? __ballot_sync(0xffffffffu, first) : 0u;
    if (warp < 4 && lane == 0) s_wcnt[warp] = __popc(fb);
    __syncthreads();
    if (first) {
        int i = __popc(fb & ((1u << lane) - 1u));
        for (int w = 0; w < warp; ++w) i += s_wcnt[w];
        s_pseg[i] = s_rowseg[tid];
        s_pblk[i] = tid >> 6;
    }
    if (tid == 0) s_npairs = s_wcnt[0] + s_wcnt[1] + s_wcnt[2] + s_wcnt[3];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int npairs = s_npairs;
    const int kb0 = (int)((long long)rank * kbt / C), kb1 = (int)((long long)(rank + 1) * kbt / C);
    const int nbase = kb1 - kb0;  // >= 1: the host keeps CL <= kbt
    const int nmine = npairs > rank ? (npairs - rank + C - 1) / C : 0;
    const int total = nbase + nmine;
    uint8_t *const ring = align1024(dsm);
    auto stage = [&](int s) { return ring + (size_t)s * kFusedStage; };

    if (warp == 4) {
        // ---- producer warp: fills the ring in item order.  Lane 0 issues the
        // TMA copies -- W k-blocks (weights, before the wait), x tiles (after
        // it), the B tiles of this CTA's LoRA pairs -- and for a LoRA pair the
        // whole warp writes the v tiles: rows of the pair's block that belong
        // to its segment get scale * v, the others 0; K-major, 128-byte
        // swizzle, as hi and lo 16-bit halves.  A stage is waited for by this
        // warp alone and in order, so a parity wait never meets a barrier two
        // phases ahead.
        const uint32_t xbytes = (uint32_t)npad * 128u, bbytes = 2u * (uint32_t)r16 * 128u;
        auto issue_w = [&](int q) {
            const int s = q % nst;
            mbar_arrive_expect_tx(&full[s], kFusedWBytes);
            tma_load_2d(stage(s), &P.tmap_w, j0, (kb0 + q) * 64, &full[s]);
            tma_load_2d(stage(s) + 8192, &P.tmap_w, j0 + 64, (kb0 + q) * 64, &full[s]);
        };
        auto issue_x = [&](int q) {
            const int s = q % nst;
            mbar_arrive_expect_tx(&full[s], xbytes);
            tma_load_2d(stage(s) + kFusedXOff, &P.tmap_x, (kb0 + q) * 64, 0, &full[s]);
        };
        auto issue_b = [&](int q) {
            const int s = q % nst;
            const int a = idx[s_pseg[rank + (q - nbase) * C]];
            mbar_arrive_expect_tx(&full[s], bbytes);
            tma_load_3d(stage(s), &P.tmap_b, j0, 0, a, &full[s]);
            tma_load_3d(stage(s) + r16 * 128, &P.tmap_b, j0 + 64, 0, a, &full[s]);
        };
        const int pre = min(nst, nbase);  // base items only (pre <= nbase)
        if (lane == 0)
            for (int q = 0; q < pre; ++q) issue_w(q);
        pdl_wait();  // x may be written by an earlier kernel, v by the shrink
        if (lane == 0)
            for (int q = 0; q < pre; ++q) issue_x(q);
        const float *const v = P.v;
        const int cpr = r16 / 8;  // 16-byte chunks per v-tile row
        for (int q = pre; q < total; ++q) {
            const int s = q % nst;
            if (q >= nst) {
                // lane 0 waits for the MMAs of item q - nst; the warp follows
                int ok = 1;
                if (lane == 0) {
                    const uint32_t ph = (uint32_t)(((q / nst) - 1) & 1);
                    if (!mbar_wait(&empty[s], ph)) {
                        set_error(err, kErrTimeout);
                        ok = mbar_wait(&empty[s], ph) ? 1 : 0;
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            }
            if (q < nbase) {
                if (lane == 0) {
                    issue_w(q);
                    issue_x(q);
                }
                continue;
            }
            if (lane == 0) issue_b(q);
            const int pr = rank + (q - nbase) * C;
            const int sg = s_pseg[pr], blk = s_pblk[pr];
            const int nrow = min(64, npad - 64 * blk);  // rows of the block's tile
            uint8_t *hi = stage(s) + kFusedXOff, *lo = stage(s) + kFusedVloOff;
            fence_proxy_async();  // the tensor cores' reads of this stage come first
            for (int e = lane; e < nrow * cpr; e += 32) {
                const int m = e / cpr, c = e - (e / cpr) * cpr;
                const int t = 64 * blk + m;
                const bool mine = t < T && s_rowseg[t] == sg;
                const float *vr = v + (size_t)(mine ? s_rowpos[t] : 0) * r;
                __align__(16) Tin hv[8], lv[8];
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8) {
                    const int k = 8 * c + k8;
                    const float f = (mine && k < r) ? scale * vr[k] : 0.f;
                    hv[k8] = from_f<Tin>(f);
                    lv[k8] = from_f<Tin>(f - to_f<Tin>(hv[k8]));
                }
                sts128(hi + sw128_offset(m, c), *reinterpret_cast<const uint4 *>(hv));
                sts128(lo + sw128_offset(m, c), *reinterpret_cast<const uint4 *>(lv));
            }
            fence_proxy_async();  // generic-proxy writes -> the tensor cores
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[s]);
        }
    } else if (tid == 0) {
        // ---- MMA issuer
        const bool bf16 = std::is_same<Tin, __nv_bfloat16>::value;
        const uint32_t id_base = idesc_f16_amn(bf16, kFusedCols, npad);
        const uint32_t id_lora0 = idesc_f16_amn(bf16, kFusedCols, min(64, npad));
        const uint32_t id_lora1 = idesc_f16_amn(bf16, kFusedCols, max(16, npad - 64));
        bool lost = false;
        for (int q = 0; q < total; ++q) {
            const int s = q % nst;
            const uint32_t ph = (uint32_t)((q / nst) & 1);
            if (!mbar_wait(&full[s], ph)) {
                set_error(err, kErrTimeout);
                lost = true;
                if (!mbar_wait(&full[s], ph)) break;
            }
            fence_proxy_async();
            tc_fence_after();
            const uint32_t sa = smem_addr(stage(s));
            if (q < nbase) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16(tmem, sw128_desc(sa + kk * 2048, 8192, 1024),
                            sw128_desc(sa + kFusedXOff + kk * 32, 16, 1024), id_base,
                            (q | kk) != 0);
            } else {
                // rows 64 blk .. of the accumulator: columns at a multiple of 64
                const int blk = s_pblk[rank + (q - nbase) * C];
                const uint32_t d = tmem + (uint32_t)(64 * blk);
                const uint32_t id_lora = blk ? id_lora1 : id_lora0;
                for (int h = 0; h < 2; ++h)
                    for (int kk = 0; kk < r16 / 16; ++kk)
                        mma_f16(d, sw128_desc(sa + kk * 2048, (uint32_t)r16 * 128u, 1024),
                                sw128_desc(sa + (h ? kFusedVloOff : kFusedXOff) + kk * 32, 16, 1024),
                                id_lora, 1);
            }
            mma_commit(&empty[s]);
        }
        mma_commit(&done);
        if (lost) s_lost = 1;
    }

    // ---- epilogue: warps 0-3, thread tid = TMEM lane tid = column j0 + tid
    const int j = j0 + tid;
    Ty *const gY = static_cast<Ty *>(P.y);
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    bool lost = false;
    if (tid < 128) {
        if (!mbar_wait(&done, 0)) {
            set_error(err, kErrTimeout);
            lost = true;
            mbar_wait(&done, 0);
        }
        tc_fence_after();
        pdl_wait();  // y may be read by an earlier kernel
    }
    __syncwarp();  // the aligned TMEM loads below need the whole warp
    // The accumulator is read in groups of 32 columns (rows t), 32 columns
    // per tcgen05.ld at multiples of 32; columns past npad are allocated and
    // hold nothing used.
    const int ngrp = (npad + 31) / 32;
    const int nown = rank < ngrp ? (ngrp - rank + C - 1) / C : 0;
    const int nown_max = (ngrp + C - 1) / C;
    if (C == 1) {
        __syncthreads();  // s_lost
        lost = lost || s_lost != 0;
        if (tid < 128) {
            for (int g = 0; g < ngrp; ++g) {
                float f[32];
                tmem_ld32(lane_addr + (uint32_t)(g * 32), f);
                if (!lost && j < H2) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int t = g * 32 + i;
                        if (t < T) gY[(size_t)t * H2 + j] = from_f<Ty>(f[i]);
                    }
                }
            }
        }
    } else {
        // Partials of group g go to CTA g % C, slot (rank, g / C): eight
        // [128][4] float quads, so that 32 lanes store 512 contiguous bytes.
        float *const recv = reinterpret_cast<float *>(ring);
        auto slot = [&](int src, int lg, int q) {
            return recv + ((size_t)((src * nown_max + lg) * 8 + q) * 128 + tid) * 4;
        };
        if (tid == 0 && nown > 0) mbar_arrive_expect_tx(&red_full, (uint32_t)(C * nown) * 16384u);
        // every CTA's MMAs are done and its ring is idle: peers may write into it
        cluster_sync();
        lost = lost || s_lost != 0;
        if (tid < 128) {
            for (int g = 0; g < ngrp; ++g) {
                float f[32];
                tmem_ld32(lane_addr + (uint32_t)(g * 32), f);
                const uint32_t owner = (uint32_t)(g % C);
                const uint32_t rbar = peer_addr(&red_full, owner);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    st_async4(peer_addr(slot(rank, g / C, q), owner), f[4 * q], f[4 * q + 1],
                              f[4 * q + 2], f[4 * q + 3], rbar);
            }
            if (nown > 0) {
                if (!mbar_wait_cluster(&red_full, 0)) {
                    set_error(err, kErrTimeout);
                    lost = true;
                    mbar_wait_cluster(&red_full, 0);
                }
                for (int lg = 0; lg < nown; ++lg) {
                    const int g = rank + lg * C;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
                        for (int src = 0; src < C; ++src) {
                            const uint4 u = lds128(slot(src, lg, q));
                            acc[0] += __uint_as_float(u.x);
                            acc[1] += __uint_as_float(u.y);
                            acc[2] += __uint_as_float(u.z);
                            acc[3] += __uint_as_float(u.w);
                        }
                        if (!lost && j < H2) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int t = g * 32 + 4 * q + e;
                                if (t < T) gY[(size_t)t * H2 + j] = from_f<Ty>(acc[e]);
                            }
                        }
                    }
                }
            }
        }
        // No closing cluster barrier: each CTA has waited for every push
        // addressed to it before it gets here.
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, P.tmem_cols);
    }
}

template <typename Tin, typename Ty>
int fused_launch_t(const FusedArgs &g) {
    const bool bf16 = std::is_same<Tin, __nv_bfloat16>::value;
    FusedParams p;
    memset(&p, 0, sizeof p);
    p.y = g.y;
    p.v = g.v;
    p.perm = g.perm;
    p.seg_ptr = g.seg_ptr;
    p.idx = g.idx;
    p.err = g.err;
    p.S = g.S;
    p.T = g.T;
    p.L = g.L;
    p.H1 = g.H1;
    p.H2 = g.H2;
    p.r = g.r;
    p.r16 = (g.r + 15) / 16 * 16;
    p.npad = (g.T + 15) / 16 * 16;
    p.kbt = (g.H1 + 63) / 64;
    p.scale = g.scale;
    p.tmem_cols = p.npad <= 32 ? 32u : p.npad <= 64 ? 64u : 128u;
    const cuuint64_t es = 2;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)g.H2, (cuuint64_t)g.H1};
        const cuuint64_t strides[1] = {(cuuint64_t)g.H2 * es};
        const cuuint32_t box[2] = {64, 64};
        if (!tmap_encode(&p.tmap_w, bf16, 2, g.W, dims, strides, box, true))
            return (int)cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)g.H1, (cuuint64_t)g.T};
        const cuuint64_t strides[1] = {(cuuint64_t)g.H1 * es};
        const cuuint32_t box[2] = {64, (cuuint32_t)p.npad};
        if (!tmap_encode(&p.tmap_x, bf16, 2, g.x, dims, strides, box, true))
            return (int)cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)g.H2, (cuuint64_t)g.r, (cuuint64_t)g.L};
        const cuuint64_t strides[2] = {(cuuint64_t)g.H2 * es, (cuuint64_t)g.r * g.H2 * es};
        const cuuint32_t box[3] = {64, (cuuint32_t)p.r16, 1};
        if (!tmap_encode(&p.tmap_b, bf16, 3, g.B, dims, strides, box, true))
            return (int)cudaErrorInvalidValue;
    }
    // Cluster size: the split of H1 that keeps the most SMs busy over whole
    // waves of one CTA per SM (ties: the smaller split), each CTA with at
    // least one k-block.
    const int ntiles = (g.H2 + kFusedCols - 1) / kFusedCols;
    const int nsm = std::max(1, g.nsm);
    int best = 1;
    double best_eff = -1.0;
    for (int c = 1; c <= std::min(8, p.kbt); ++c) {
        const long long ctas = (long long)ntiles * c;
        const long long waves = (ctas + nsm - 1) / nsm;
        const double eff = (double)ctas / (double)(waves * nsm);
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = c;
        }
    }
    p.cl = best;
    auto kernel = sgmv_fused_kernel<Tin, Ty>;
    // ring stages: what the per-block limit leaves beside the kernel's static
    // shared memory and the 1024-byte alignment slack
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return (int)e;
    const size_t smem_max = 227u * 1024u;
    if (smem_max < fa.sharedSizeBytes + 1024u + kFusedStage) return (int)cudaErrorInvalidValue;
    p.nst = (int)std::min<size_t>(kFusedMaxStages,
                                  (smem_max - fa.sharedSizeBytes - 1024u) / kFusedStage);
    const size_t smem = (size_t)p.nst * kFusedStage + 1024u;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.cl, (unsigned)ntiles, 1);
    cfg.blockDim = dim3(kFusedThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = g.stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (p.cl > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)p.cl;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = (unsigned)na;
    return (int)cudaLaunchKernelEx(&cfg, kernel, p);
}

template <typename Tin>
int fused_launch_in(const FusedArgs &g) {
    switch (g.y_dtype) {
        case 0: return fused_launch_t<Tin, __half>(g);
        case 1: return fused_launch_t<Tin, __nv_bfloat16>(g);
        default: return fused_launch_t<Tin, float>(g);
    }
}

}  // namespace

int fused_launch(const FusedArgs &g) {
    return g.in_dtype == 0 ? fused_launch_in<__half>(g) : fused_launch_in<__nv_bfloat16>(g);
}

}  // namespace sgmv
