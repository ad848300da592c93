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
// and the adapters' B slices with little arithmetic per byte.  Three launches
// on the stream, chained by programmatic dependent launch:
//   1. the shrink v = x . A[a] (the CUDA-core kernel of sgmv_shrink), fp32
//      by sorted position into the workspace;
//   2. sgmv_fused_prep_kernel: the adapter terms' work list and operands
//      (below) into the workspace;
//   3. sgmv_fused_kernel: every output element of y, once, on the tensor
//      cores, in the transposed ("swap AB") form that suits few rows:
//
//   D[j, t] = sum_h W[h, j] x[t, h]  +  sum_k B[a_t][k, j] (scale v[t, k])
//
// with M = 128 columns j of W per tile (W and B tiles are MN-major A
// operands, loaded by TMA with 128-byte swizzle), N = the batch's rows
// rounded up to 16 (x rows are the K-major B operand) and fp32 accumulation
// in tensor memory, where accumulator column t is row t of the batch.
//
// Adapter terms.  The rows of the batch fall into 16-row chunks (accumulator
// columns 16c .. 16c + 15).  A "pair" is one segment with an adapter and one
// chunk holding at least one of its rows; there are at most T pairs.  For
// each pair the prep kernel writes a 16 x 64 tile of 16-bit values: row n is
// batch row 16c + n, holding scale * v of that row if the row is in the
// segment, else 0, as two halves (hi = round(scale v), lo = round(scale v -
// hi)) so that v keeps about 16 significant bits.  The pair's term is then a
// handful of N = 16 MMAs into accumulator columns 16c .., with the segment's
// B slice (r rows, padded to rp = 16, 32 or 64) as the A operand, once
// against the hi half and once against the lo half.  The whole layer -- base
// and adapter terms -- is one fp32 accumulation, rounded once to y's type.
//
// Decomposition of the fused kernel: one tile of 128 columns per cluster of
// CL CTAs; CTA `rank` takes an even share of H1's 64-column k-blocks and
// every CL-th group of pairs, so all CTAs stream about the same bytes.  The
// partial accumulators meet in an fp32 scratch area of the workspace (in L2:
// distributed shared memory moved them no faster); after a cluster barrier
// each CTA brings the slots of every CL-th group of 32 rows of the tile into
// its idle ring by bulk copies and sums them in rank order: deterministic.
//
// Warps of the fused kernel: 0-3 read the accumulator (one TMEM lane, i.e.
// one column j, per thread) and write y; before that, warp 3 issues the MMAs
// and warp 2 reads the pair table; warp 4 fills the ring in order (W before
// griddepcontrol.wait, and x too when the shrink was launched before it,
// since that kernel waits for x's producer first; the adapter operands after
// the wait).  The issuing warps wait as a whole and one lane issues: a warp
// whose other lanes sit in a suspended mbarrier wait holds up a lane that
// branched away from them.  Each barrier has one waiting role that takes its
// phases in order.  Every mbarrier wait is bounded.
#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "sgmv_device.cuh"
#include "sgmv_internal.h"
#include "sgmv_fused.h"
#include "sgmv_tcgen05.cuh"

namespace sgmv {
namespace {

constexpr int kFusedThreads = 160;
constexpr int kFusedCols = 128;               // columns of W per tile (M of every MMA)
constexpr int kFusedMaxStages = 16;
// Ring stages used: more bytes in flight per SM only lengthened the copies'
// latency (one, 32 and 128 rows at the Llama-2-7B q shape: four stages
// 15.8 / 21.0 / 36.0 us per call against 16.6 / 23.0 / 35.8 with as many as
// fit, and no better with three or five)
constexpr int kFusedRingStages = 4;
constexpr uint32_t kFusedXOff = 16384;        // x tile at this offset of a stage
constexpr uint32_t kFusedWBytes = 2u * 64u * 128u;  // two 64-column halves of a k-block of W
constexpr int kFusedMaxPairs = 128;           // at most T pairs, T <= 128
constexpr int kFusedMaxPPI = 8;               // pairs per ring stage
constexpr int kPrepThreads = 256;
constexpr int kPrepMaxCtas = 32;
constexpr int kFusedMaxCl = 8;                // CTAs per cluster (portable limit)
constexpr double kFusedCtaUs = 6.0;           // cluster-size model: fixed cost of a CTA
constexpr double kFusedStageUs = 0.45;        // ... and of one ring stage

// As tmem_ld32 without the wait: the registers are valid after tmem_wait_ld.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// The same for every state space (global memory written through the generic
// proxy, then read by a bulk copy).
__device__ __forceinline__ void fence_proxy_async_all() {
    asm volatile("fence.proxy.async;" ::: "memory");
}

__host__ __device__ inline int fused_rp(int r) { return r <= 16 ? 16 : r <= 32 ? 32 : 64; }
// 16 x 64 tiles of v per pair: hi and lo share one tile for rp <= 32
__host__ __device__ inline int fused_ntile(int rp) { return rp <= 32 ? 1 : 2; }
// bytes of a pair's B slice (both 64-column halves) and of its v tiles
__host__ __device__ inline uint32_t fused_abytes(int rp) { return 2u * (uint32_t)rp * 128u; }
__host__ __device__ inline uint32_t fused_vbytes(int rp) { return (uint32_t)fused_ntile(rp) * 2048u; }
// the pair table: [0] = pairs, then (adapter, chunk) per pair; 256-byte rounded
__host__ __device__ inline size_t fused_ptab_bytes(int T) {
    return ((size_t)(1 + 2 * T) * 4u + 255u) / 256u * 256u;
}

// ---- work list and v tiles -------------------------------------------------
struct PrepParams {
    const float *v;          // [T][r] fp32 by sorted position (the shrink's output)
    const int32_t *perm, *seg_ptr, *idx;
    int *err;
    int32_t *ptab;           // pair table
    void *vt;                // [pair][ntile][16][64] 16-bit
    int32_t S, T, L, r, rp;
    int32_t early;           // 1: the metadata may be read before griddepcontrol.wait
    float scale;
};

// Every CTA lists the slots (segments with an adapter and rows, in segment
// order), maps each position to its slot and each row to its position, and
// numbers the pairs: slot by slot, chunks in ascending order.  CTA 0 writes
// the pair table and reports bad metadata; all CTAs then write every
// gridDim.x-th 16-byte chunk of the pairs' v tiles.
template <typename Tin>
__global__ void __launch_bounds__(kPrepThreads) sgmv_fused_prep_kernel(const PrepParams P) {
    // the fused kernel may start its base k-blocks now: it reads what this
    // kernel writes only after its own griddepcontrol.wait
    pdl_trigger();
    if (!P.early) pdl_wait();  // the metadata may come from the kernel just before
    const int T = P.T, S = P.S, L = P.L, r = P.r, rp = P.rp;
    __shared__ int s_b[128], s_e[128], s_a[128];
    __shared__ unsigned s_mask[128];
    __shared__ int s_rowslot[128], s_rowpos[128];
    __shared__ int s_pslot[kFusedMaxPairs], s_pchunk[kFusedMaxPairs];
    __shared__ int s_wsum[kPrepThreads / 32];
    __shared__ int s_nslot, s_np;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool report = blockIdx.x == 0;
    if (tid < 128) {
        s_rowslot[tid] = -1;
        s_mask[tid] = 0u;
    }
    // the row at this thread's position, requested first: its load overlaps
    // the segments' below
    const int prow = tid < T ? (P.perm ? P.perm[tid] : tid) : 0;
    // slots: every thread reads one segment's bounds and id (all segments'
    // loads in flight together), then a block-wide scan numbers the valid ones
    int nbase = 0;
    for (int s0 = 0; s0 < S; s0 += kPrepThreads) {
        const int s = s0 + tid;
        int b = 0, e = 0, a = -1;
        bool ok = false;
        if (s < S) {
            b = P.seg_ptr[s];
            e = P.seg_ptr[s + 1];
            a = P.idx[s];
            const bool seg_good = b >= 0 && e >= b && e <= T;
            if (report && !seg_good) set_error(P.err, kErrBadSegments);
            if (report && seg_good && e > b && (a < -1 || a >= L)) set_error(P.err, kErrBadIndex);
            ok = seg_good && e > b && a >= 0 && a < L;
        }
        const unsigned m = __ballot_sync(0xffffffffu, ok);
        if (lane == 0) s_wsum[warp] = __popc(m);
        __syncthreads();
        int before = nbase;
        for (int w = 0; w < warp; ++w) before += s_wsum[w];
        const int i = before + __popc(m & ((1u << lane) - 1u));
        if (ok && i < 128) {
            s_b[i] = b;
            s_e[i] = e;
            s_a[i] = a;
        }
        for (int w = 0; w < kPrepThreads / 32; ++w) nbase += s_wsum[w];
        __syncthreads();  // s_wsum is reused
    }
    if (tid == 0) s_nslot = min(nbase, 128);  // slots hold disjoint rows: at most T
    __syncthreads();
    const int nslot = s_nslot;
    if (tid < T) {
        // position p: the last slot starting at or before it, if it ends after it
        const int p = tid;
        int lo = 0, hi = nslot - 1, i = -1;
        while (lo <= hi) {
            const int mid = (lo + hi) >> 1;
            if (s_b[mid] <= p) {
                i = mid;
                lo = mid + 1;
            } else {
                hi = mid - 1;
            }
        }
        if (i >= 0 && p < s_e[i]) {
            const int t = prow;
            if (t < 0 || t >= T) {
                if (report) set_error(P.err, kErrBadIndex);
            } else {
                s_rowslot[t] = i;
                s_rowpos[t] = p;
                atomicOr(&s_mask[i], 1u << (t >> 4));
            }
        }
    }
    __syncthreads();
    // pairs: exclusive prefix over slots of their chunk counts
    const int cnt = tid < nslot ? __popc(s_mask[tid]) : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int woff = 0;
    for (int w = 0; w < warp; ++w) woff += s_wsum[w];
    if (tid < nslot) {
        unsigned m = s_mask[tid];
        for (int k = woff + incl - cnt; m != 0u; ++k) {
            s_pslot[k] = tid;
            s_pchunk[k] = __ffs(m) - 1;
            m &= m - 1u;
        }
    }
    if (tid == kPrepThreads - 1) s_np = woff + incl;
    __syncthreads();
    const int np = min(s_np, kFusedMaxPairs);
    // Written only after the wait: the kernel before this one on the stream
    // (the last fused kernel) may still read the workspace until then.
    if (P.early) pdl_wait();  // also: v is written by the shrink
    if (report) {
        for (int k = tid; k < np; k += kPrepThreads) {
            P.ptab[1 + 2 * k] = s_a[s_pslot[k]];
            P.ptab[2 + 2 * k] = s_pchunk[k];
        }
        if (tid == 0) P.ptab[0] = np;
    }
    const int ntile = fused_ntile(rp);
    const int per_pair = ntile * 16 * 8;  // 16-byte chunks
    const float scale = P.scale;
    Tin *const out = static_cast<Tin *>(P.vt);
    for (int e = blockIdx.x * kPrepThreads + tid; e < np * per_pair; e += gridDim.x * kPrepThreads) {
        const int k = e / per_pair, rem = e - k * per_pair;
        const int tile = rem >> 7, n = (rem >> 3) & 15, c8 = rem & 7;
        const int t = 16 * s_pchunk[k] + n;
        __align__(16) Tin hv[8];
        if (t < T && s_rowslot[t] == s_pslot[k]) {
            const float *vr = P.v + (size_t)s_rowpos[t] * r;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int col = 8 * c8 + u;
                const int h = rp <= 32 ? col >> 5 : tile;
                const int kk = rp <= 32 ? col & 31 : col;
                const float f = kk < r ? scale * vr[kk] : 0.f;
                const Tin hi = from_f<Tin>(f);
                hv[u] = h ? from_f<Tin>(f - to_f<Tin>(hi)) : hi;
            }
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) hv[u] = from_f<Tin>(0.f);
        }
        *reinterpret_cast<uint4 *>(out + ((size_t)(k * ntile + tile) * 16 + n) * 64 + 8 * c8) =
            *reinterpret_cast<const uint4 *>(hv);
    }
}

// ---- the fused layer -------------------------------------------------------
struct FusedParams {
    CUtensorMap tmap_w;   // W as [H1][H2], box {64, 64}, 128-byte swizzle
    CUtensorMap tmap_x;   // x as [T][H1], box {64, npad}
    CUtensorMap tmap_b;   // B as [L][r][H2], box {64, rp, 1}
    CUtensorMap tmap_v;   // v tiles as [T * ntile * 16][64], box {64, ppi * ntile * 16}
    void *y;
    float *part;      // [tiles][CL][npad][128] fp32 partials (CL > 1)
    const int32_t *ptab;
    int *err;
    int32_t T, H1, H2;
    int32_t rp;       // r rounded up to 16, 32 or 64
    int32_t npad;     // T rounded up to 16 (N of the base MMAs)
    int32_t cl;       // CTAs per cluster (split of the tile's k-blocks)
    int32_t kbt;      // 64-column k-blocks of H1
    int32_t nst;      // ring stages
    int32_t ppi;      // pairs per ring stage
    int32_t x_early;  // 1: x may be read before griddepcontrol.wait
    int32_t lora;     // 1: the pair table and v tiles were written (segments given)
    uint32_t stage_bytes;  // >= 16 KB of W + the x tile, and >= ppi pairs' operands
    uint32_t tmem_cols;
};

constexpr int kItemLora = 1, kItemEnd = 2;

template <typename Tin, typename Ty>
__global__ void __launch_bounds__(kFusedThreads, 1)
    sgmv_fused_kernel(const __grid_constant__ FusedParams P) {
    const int T = P.T, H2 = P.H2, rp = P.rp, npad = P.npad;
    const int C = P.cl, kbt = P.kbt, nst = P.nst, ppi = P.ppi;
    int *const err = P.err;

    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[kFusedMaxStages], empty[kFusedMaxStages], done, tab_ready,
        red_full;
    __shared__ int s_pa[kFusedMaxPairs], s_pc[kFusedMaxPairs];  // pair table
    __shared__ int s_kind[kFusedMaxStages], s_cnt[kFusedMaxStages];
    __shared__ int s_chunk[kFusedMaxStages][kFusedMaxPPI];
    __shared__ int s_np, s_lost;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)blockIdx.x;
    const int j0 = (int)blockIdx.y * kFusedCols;

    // The next kernel on the stream may start now: it reads nothing this one
    // writes before its own griddepcontrol.wait.
    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 2);   // two arrivals: W + x, or B slices + v tiles, or the end
            mbar_init(&empty[s], 1);  // the MMAs that read the stage are done
        }
        mbar_init(&done, 1);
        mbar_init(&tab_ready, 1);
        mbar_init(&red_full, 1);  // the owner's slots of partial sums, by bulk copies
        mbar_init_fence();
        s_lost = 0;
    }
    __syncthreads();
    // This CTA's k-blocks of H1 depend on its rank only: the first stages of
    // W (and of x, when it may be read now) are requested before the rest of
    // the set-up, which then overlaps their latency.
    const int kb0 = (int)((long long)rank * kbt / C), kb1 = (int)((long long)(rank + 1) * kbt / C);
    const int nbase = kb1 - kb0;  // >= 1: the host keeps CL <= kbt
    const int pre = min(nst, nbase);
    const bool x_early = P.x_early != 0;
    uint8_t *const ring = align1024(dsm);
    const uint32_t stage_bytes = P.stage_bytes;
    auto stage = [&](int s) { return ring + (size_t)s * stage_bytes; };
    const uint32_t xbytes = (uint32_t)npad * 128u;
    const uint32_t abytes = fused_abytes(rp), vbytes = fused_vbytes(rp);
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
    if (warp == 4 && lane == 0)
        for (int q = 0; q < pre; ++q) {
            issue_w(q);
            if (x_early) issue_x(q);
        }
    if (warp == 0) tmem_alloc(&s_tmem, P.tmem_cols);  // a converged warp, as the instruction needs
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 2 && P.lora) {
        // ---- the pair table, read by a warp that is idle until the epilogue
        pdl_wait();  // the table is written by the kernel just before
        const int np = min(P.ptab[0], kFusedMaxPairs);
        for (int k = lane; k < np; k += 32) {
            s_pa[k] = P.ptab[1 + 2 * k];
            s_pc[k] = P.ptab[2 + 2 * k];
        }
        if (lane == 0) s_np = np;
        __syncwarp();
        if (lane == 0) mbar_arrive(&tab_ready);
    } else if (warp == 4) {
        // ---- producer: the whole warp takes the ring's phases in item order
        // (base k-blocks, then this CTA's groups of pairs, then an end marker)
        // and lane 0 issues the copies; the first stages were requested above.
        // (All lanes wait: a warp whose other lanes sit in a suspended wait
        // would hold up the issuing lane.)
        bool stop = false;
        auto wait_empty = [&](int q) {
            if (q < nst) return true;
            const int s = q % nst;
            const uint32_t ph = (uint32_t)(((q / nst) - 1) & 1);
            if (mbar_wait(&empty[s], ph)) return true;
            set_error(err, kErrTimeout);
            return mbar_wait(&empty[s], ph);
        };
        if (!x_early) {
            pdl_wait();  // x may be written by the kernel just before
            if (lane == 0)
                for (int q = 0; q < pre; ++q) issue_x(q);
        }
        int q = pre;
        for (; q < nbase; ++q) {
            if (!wait_empty(q)) {
                stop = true;
                break;
            }
            // the stage's expected bytes first, then three lanes issue a copy each
            const int s = q % nst;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], kFusedWBytes);
                mbar_arrive_expect_tx(&full[s], xbytes);
            }
            __syncwarp();
            if (lane < 2)
                tma_load_2d(stage(s) + lane * 8192, &P.tmap_w, j0 + lane * 64, (kb0 + q) * 64,
                            &full[s]);
            else if (lane == 2)
                tma_load_2d(stage(s) + kFusedXOff, &P.tmap_x, (kb0 + q) * 64, 0, &full[s]);
            __syncwarp();
        }
        if (!stop && P.lora) {
            pdl_wait();  // the v tiles: written by the kernel just before
            if (!mbar_wait(&tab_ready, 0)) {
                set_error(err, kErrTimeout);
                stop = !mbar_wait(&tab_ready, 0);
            }
            const int np = stop ? 0 : s_np;
            const int nitems = (np + ppi - 1) / ppi;
            for (int it = rank; it < nitems; it += C, ++q) {
                if (!wait_empty(q)) {
                    stop = true;
                    break;
                }
                // the stage's expected bytes first, then one lane per copy: lanes
                // 2i and 2i + 1 the two halves of pair i's B slice, lane 31 the
                // v tiles of all ppi pairs in one box (past the last pair: unused)
                const int s = q % nst, k0 = it * ppi, n = min(ppi, np - k0);
                uint8_t *const st = stage(s);
                if (lane == 0) {
                    s_kind[s] = kItemLora;
                    s_cnt[s] = n;
                    for (int i = 0; i < n; ++i) s_chunk[s][i] = s_pc[k0 + i];
                    mbar_arrive_expect_tx(&full[s], (uint32_t)n * abytes);
                    mbar_arrive_expect_tx(&full[s], (uint32_t)ppi * vbytes);
                }
                __syncwarp();
                if (lane < 2 * n) {
                    const int i = lane >> 1, h = lane & 1;
                    tma_load_3d(st + i * abytes + h * rp * 128, &P.tmap_b, j0 + h * 64, 0,
                                s_pa[k0 + i], &full[s]);
                } else if (lane == 31) {
                    tma_load_2d(st + ppi * abytes, &P.tmap_v, 0, k0 * (int)(vbytes / 128u),
                                &full[s]);
                }
                __syncwarp();
            }
        }
        if (!stop && wait_empty(q) && lane == 0) {
            const int s = q % nst;
            s_kind[s] = kItemEnd;
            mbar_arrive(&full[s]);
            mbar_arrive(&full[s]);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ---- MMA issuer: the whole warp waits, lane 0 issues
        // one accumulator [128 columns of W][npad rows]
        const bool bf16 = std::is_same<Tin, __nv_bfloat16>::value;
        const uint32_t idesc = idesc_f16_amn(bf16, kFusedCols, npad);
        const uint32_t idesc16 = idesc_f16_amn(bf16, kFusedCols, 16);
        const uint32_t lo_off = rp <= 32 ? 64u : 2048u;  // the lo half of a pair's v
        bool lost = false;
        for (int q = 0;; ++q) {
            const int s = q % nst;
            const uint32_t ph = (uint32_t)((q / nst) & 1);
            if (!mbar_wait(&full[s], ph)) {
                set_error(err, kErrTimeout);
                lost = true;
                if (!mbar_wait(&full[s], ph)) break;
            }
            tc_fence_after();
            const uint32_t sa = smem_addr(stage(s));
            const int kind = q < nbase ? 0 : s_kind[s];
            if (kind == kItemEnd) break;
            if (lane == 0) {
                if (kind == 0) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16(tmem, sw128_desc(sa + kk * 2048, 8192, 1024),
                                sw128_desc(sa + kFusedXOff + kk * 32, 16, 1024), idesc,
                                (q | kk) != 0);
                } else {
                    const int n = s_cnt[s];
                    for (int i = 0; i < n; ++i) {
                        const uint32_t d = tmem + 16u * (uint32_t)s_chunk[s][i];
                        const uint32_t a = sa + i * abytes, v = sa + ppi * abytes + i * vbytes;
                        for (int kk = 0; kk < rp / 16; ++kk) {
                            const uint64_t ad = sw128_desc(a + kk * 2048, rp * 128, 1024);
                            mma_f16(d, ad, sw128_desc(v + kk * 32, 16, 1024), idesc16, 1);
                            mma_f16(d, ad, sw128_desc(v + lo_off + kk * 32, 16, 1024), idesc16,
                                    1);
                        }
                    }
                }
                mma_commit(&empty[s]);
            }
            __syncwarp();
        }
        if (lane == 0) {
            mma_commit(&done);
            if (lost) s_lost = 1;
        }
        __syncwarp();
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
    // hold nothing used.  Every group holds at least one row t < T.
    const int ngrp = (npad + 31) / 32;
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
        // This CTA's partials into the tile's scratch slot `rank`, as [group]
        // [8 quads of rows][128 columns][4 rows] so that a warp moves 512
        // contiguous bytes per access (quads holding rows t < T only); a
        // cluster barrier; then groups g = rank, rank + CL, ... summed over
        // the CL slots in rank order.
        float4 *const part = reinterpret_cast<float4 *>(P.part) + (size_t)blockIdx.y * C * ngrp * 1024;
        auto nq_of = [&](int g) { return min(8, (T - g * 32 + 3) >> 2); };
        if (tid < 128) {
            // every group's accumulator columns requested before one wait
            // (ngrp <= 4: the accumulator has at most 128 columns)
            uint32_t f[4][32];
#pragma unroll
            for (int g = 0; g < 4; ++g)
                if (g < ngrp) tmem_ld32_async(lane_addr + (uint32_t)(g * 32), f[g]);
            tmem_wait_ld();
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                if (g >= ngrp) break;
                const int nq = nq_of(g);
                float4 *const dst = part + ((size_t)rank * ngrp + g) * 1024 + tid;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q < nq)
                        dst[q * 128] = make_float4(
                            __uint_as_float(f[g][4 * q]), __uint_as_float(f[g][4 * q + 1]),
                            __uint_as_float(f[g][4 * q + 2]), __uint_as_float(f[g][4 * q + 3]));
            }
            fence_proxy_async_all();  // the owners read these by bulk copies
        }
        // release / acquire at cluster scope: the partials are visible after it
        cluster_sync();
        lost = lost || s_lost != 0;
        // The owner's slots come into the (idle) ring by one bulk copy per
        // (group, source), compactly, when they fit: one copy engine keeps
        // them all in flight (register loads of the same bytes took ~3 us).
        uint32_t rbytes = 0;
        for (int g = rank; g < ngrp; g += C) rbytes += (uint32_t)(C * nq_of(g)) * 2048u;
        const bool by_copy = rbytes <= (uint32_t)nst * stage_bytes;
        float *const recv = reinterpret_cast<float *>(ring);
        if (by_copy && rbytes > 0) {
            if (tid == 0) {
                fence_proxy_async_all();  // generic writes of the peers -> the copy unit
                mbar_arrive_expect_tx(&red_full, rbytes);
                uint32_t off = 0;
                for (int g = rank; g < ngrp; g += C) {
                    const uint32_t nb = (uint32_t)nq_of(g) * 2048u;
                    for (int src = 0; src < C; ++src, off += nb)
                        bulk_g2s(reinterpret_cast<uint8_t *>(recv) + off,
                                 part + ((size_t)src * ngrp + g) * 1024, nb, &red_full);
                }
            }
            if (tid < 128 && !mbar_wait(&red_full, 0)) {
                set_error(err, kErrTimeout);
                lost = true;
                mbar_wait(&red_full, 0);
            }
        }
        if (tid < 128) {
            uint32_t off = 0;  // floats
            for (int g = rank; g < ngrp; g += C) {
                const int nq = nq_of(g);
                float4 acc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (by_copy) {
                    for (int src = 0; src < C; ++src, off += (uint32_t)nq * 512u) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            if (q < nq) {
                                const uint4 u = lds128(recv + off + (q * 128 + tid) * 4);
                                acc[q].x += __uint_as_float(u.x);
                                acc[q].y += __uint_as_float(u.y);
                                acc[q].z += __uint_as_float(u.z);
                                acc[q].w += __uint_as_float(u.w);
                            }
                    }
                } else {
                    for (int s0 = 0; s0 < C; s0 += 4) {
                        float4 u[4][8];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                if (s0 + i < C && q < nq)
                                    u[i][q] = __ldcg(part + ((size_t)(s0 + i) * ngrp + g) * 1024 + q * 128 + tid);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                if (s0 + i < C && q < nq) {
                                    acc[q].x += u[i][q].x;
                                    acc[q].y += u[i][q].y;
                                    acc[q].z += u[i][q].z;
                                    acc[q].w += u[i][q].w;
                                }
                    }
                }
                if (!lost && j < H2) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float a4[4] = {acc[q].x, acc[q].y, acc[q].z, acc[q].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int t = g * 32 + 4 * q + e;
                            if (t < T) gY[(size_t)t * H2 + j] = from_f<Ty>(a4[e]);
                        }
                    }
                }
            }
        }
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
    p.err = g.err;
    p.T = g.T;
    p.H1 = g.H1;
    p.H2 = g.H2;
    p.rp = fused_rp(g.r);
    p.npad = (g.T + 15) / 16 * 16;
    // x may be read before the wait when the shrink was launched before this
    // kernel: the shrink waits for the kernel before it (which may write x)
    // before it lets the next kernels start
    p.x_early = g.x_early ? 1 : 0;
    p.lora = g.prep ? 1 : 0;
    p.kbt = (g.H1 + 63) / 64;
    p.tmem_cols = p.npad <= 32 ? 32u : p.npad <= 64 ? 64u : 128u;
    const uint32_t abytes = fused_abytes(p.rp), vbytes = fused_vbytes(p.rp);
    p.stage_bytes = std::max(kFusedXOff + (uint32_t)p.npad * 128u, abytes + vbytes);  // 1024 | both
    p.ppi = (int)std::min<uint32_t>((uint32_t)std::min(kFusedMaxPPI, (int)g.T),
                                    p.stage_bytes / (abytes + vbytes));
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
        const cuuint32_t box[3] = {64, (cuuint32_t)p.rp, 1};  // rows r .. rp-1 read as 0
        if (!tmap_encode(&p.tmap_b, bf16, 3, g.B, dims, strides, box, true))
            return (int)cudaErrorInvalidValue;
    }
    const int ntile = fused_ntile(p.rp);
    uint8_t *const vt = g.prep ? static_cast<uint8_t *>(g.prep) + fused_ptab_bytes(g.T) : nullptr;
    if (g.prep) {
        // rows past the T pairs' tiles read as 0 (a box may run past the last pair)
        const cuuint64_t dims[2] = {64, (cuuint64_t)g.T * ntile * 16};
        const cuuint64_t strides[1] = {128};
        const cuuint32_t box[2] = {64, (cuuint32_t)(p.ppi * ntile * 16)};
        if (!tmap_encode(&p.tmap_v, bf16, 2, vt, dims, strides, box, true))
            return (int)cudaErrorInvalidValue;
        p.ptab = static_cast<const int32_t *>(g.prep);
    }
    // Cluster size: the split of H1 with the least modelled time, waves of
    // one CTA per SM times a CTA's fixed cost plus its items (k-blocks of W
    // and groups of pairs) at a stage each.  Constants measured on the
    // Llama-2-7B shapes at 128 rows (about 6 us of set-up and reduction per
    // CTA, 0.45 us per stage); the model picks the measured best split of
    // the three (4096 -> 4096: 4; 4096 -> 11008: 3, 63 us against 92 with
    // the most SMs busy; 11008 -> 4096: 4).
    const int ntiles = (g.H2 + kFusedCols - 1) / kFusedCols;
    const int nsm = std::max(1, g.nsm);
    const int nl = g.prep ? (g.T + p.ppi - 1) / p.ppi : 0;  // groups of pairs, at most
    int best = 1;
    double best_t = 1e30;
    for (int c = 1; c <= std::min(kFusedMaxCl, p.kbt); ++c) {
        const long long waves = ((long long)ntiles * c + nsm - 1) / nsm;
        const double items = (double)((p.kbt + c - 1) / c) + (double)((nl + c - 1) / c);
        const double t = (double)waves * (kFusedCtaUs + items * kFusedStageUs);
        if (t < best_t - 1e-9) {
            best_t = t;
            best = c;
        }
    }
    p.cl = best;
    p.part = g.part;
    auto kernel = sgmv_fused_kernel<Tin, Ty>;
    // ring stages: what the per-block limit leaves beside the kernel's static
    // shared memory and the 1024-byte alignment slack
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return (int)e;
    const size_t smem_max = 227u * 1024u;
    p.nst = (int)std::min<size_t>(kFusedRingStages,
                                  (smem_max - fa.sharedSizeBytes - 1024u) / p.stage_bytes);
    if (p.nst < 2) return (int)cudaErrorInvalidValue;
    const size_t smem = (size_t)p.nst * p.stage_bytes + 1024u;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchAttribute attrs[2];
    // the work list and v tiles first (after the shrink)
    if (g.prep) {
        PrepParams vp;
        vp.v = g.v;
        vp.perm = g.perm;
        vp.seg_ptr = g.seg_ptr;
        vp.idx = g.idx;
        vp.err = g.err;
        vp.ptab = static_cast<int32_t *>(g.prep);
        vp.vt = vt;
        vp.S = g.S;
        vp.T = g.T;
        vp.L = g.L;
        vp.r = g.r;
        vp.rp = p.rp;
        vp.early = g.x_early ? 1 : 0;
        vp.scale = g.scale;
        cudaLaunchConfig_t vc = {};
        vc.gridDim = dim3((unsigned)std::min(kPrepMaxCtas, (int)g.T), 1, 1);
        vc.blockDim = dim3(kPrepThreads, 1, 1);
        vc.stream = g.stream;
        attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[0].val.programmaticStreamSerializationAllowed = 1;
        vc.attrs = attrs;
        vc.numAttrs = 1;
        e = cudaLaunchKernelEx(&vc, sgmv_fused_prep_kernel<Tin>, vp);
        if (e != cudaSuccess) return (int)e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.cl, (unsigned)ntiles, 1);
    cfg.blockDim = dim3(kFusedThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = g.stream;
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

size_t fused_prep_bytes(int32_t T, int32_t r) {
    if (T <= 0 || r <= 0) return 0;
    return fused_ptab_bytes(T) + (size_t)T * fused_vbytes(fused_rp(r));
}

size_t fused_part_bytes(int32_t T, int32_t H2) {
    if (T <= 0 || H2 <= 0) return 0;
    const size_t tiles = ((size_t)H2 + kFusedCols - 1) / kFusedCols;
    return tiles * kFusedMaxCl * (size_t)((T + 31) / 32 * 32) * kFusedCols * 4u;
}

int fused_launch(const FusedArgs &g) {
    return g.in_dtype == 0 ? fused_launch_in<__half>(g) : fused_launch_in<__nv_bfloat16>(g);
}

}  // namespace sgmv
