// sgmv_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) SGMV for long segments.
//
// A prefill segment of hundreds of rows turns each SGMV step into a real
// dense contraction ("Punica: when LoRA fine-tuned models need multi-tenant
// serving", omica.com.cn article, §2.2: shrink x.A, then expand v.B, per
// adapter): X[rows, H1] . A[a] is [rows, r], and v[rows, r] . B[a] is
// [rows, H2].  These kernels run both on the 5th-generation tensor cores.
//
// Shrink (sgmv_tc_shrink_kernel): one 128-row tile of a segment per cluster;
//   the cluster's CL CTAs split H1.  Each CTA streams 64-column k-blocks
//   through a 4-stage ring: X rows are gathered through perm with 16-byte
//   cp.async writes (a warp reads four whole 128-byte row pieces per
//   instruction) into the 128-byte-swizzled K-major layout, A[a] k-blocks
//   come by TMA (N-major, same swizzle).  One thread issues
//   tcgen05.mma (M=128, N=r, K=16) into a TMEM accumulator; commits free the
//   stages.  The partial v is read out of TMEM, pushed to the CTA that owns
//   its rows through distributed shared memory (into the ring's memory, once
//   every CTA of the cluster has made its products), summed in rank order and
//   written as two 16-bit halves, hi = round(v) and lo = round(v - hi), so
//   the expand can run on 16-bit tensor cores and still see v to about
//   16 significant bits.
// Expand (sgmv_tc_expand_kernel): one CTA per SM.  The (128-row tile,
//   column block of N = 64 (fp32 y) or 128 columns) pairs lie end to end,
//   each weighing its tile's rows plus a fixed cost per block; each CTA takes
//   an equal share of the first part of that line (a run that may cross into
//   the next tile) and, with fp32 y, then claims blocks of the rest four at a
//   time from a counter the shrink kernel zeroed.  v hi/lo of a block's tile
//   is loaded by TMA (K-major) whenever the tile changes.  A B warp streams
//   B[a][:, j:j+N] (N-major) through a ring and hands claimed blocks (column,
//   tile, rows) to the other warps through a ring of descriptors; the
//   MMA warp makes 2 x r/16 MMAs per block, v_hi.B + v_lo.B, into one of
//   four (fp32 y) or two TMEM buffers, so it runs up to that many blocks
//   ahead of the epilogue.  Two epilogue groups take alternate blocks; each
//   thread owns one row and reads 32 accumulator columns per tcgen05.ld.
//   fp32 y: the row's scale * acc goes to shared memory and one bulk
//   reduction per row adds it to y in L2 (y never passes through the SM).
//   16-bit y: y comes in by coalesced 16-byte cp.async copies through a
//   2-stage ring, y += scale * acc in fp32 is rounded once, and coalesced
//   16-byte stores write the block back.
// Every mbarrier wait is bounded; TMEM is freed on every path.
#include <mutex>

#include <cuda.h>  // CUtensorMap and the encoder's signature (no libcuda link)

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "sgmv_device.cuh"
#include "sgmv_internal.h"
#include "sgmv_tcgen05.cuh"
#include "sgmv_tiles.cuh"

namespace sgmv {

constexpr int kTcThreads = 128;  // 4 warps: one TMEM lane (tile row) per thread
constexpr int kTcRows = 128;     // M of one tile
constexpr int kKB = 64;          // k-block: 64 16-bit elements = one 128-byte swizzle row
constexpr int kStages = 4;       // shrink ring depth
constexpr int kShrinkProducers = 96;  // warps 1-3 of the shrink load its ring
constexpr int kExpandThreads = 2 * kTcRows + 64;  // two epilogue groups, an MMA warp, a B warp
constexpr int kExpandYStages = 2;  // most y stages per epilogue group
constexpr int kExpandBStages = 8;  // most B stages
// Fixed cost of one column block of the expand (its MMAs, barriers and
// epilogue steps), in the y rows that take as long: part of a tile's weight
// when the expand's CTAs are dealt to tiles.
constexpr int kExpandBlockRows = 128;
constexpr size_t kExpandSmemMax = 226u * 1024u;

struct TCShrinkParams {
    CUtensorMap tmap_a;  // A as [L][H1][r], box {64, 64, 1}
    const void *x;
    const int32_t *perm, *seg_ptr, *idx;
    int *err;
    void *vhi, *vlo;     // [T][r] each, input type
    int *claim;          // the expand's claim counter: zeroed here
    int32_t S, T, L, H1, r, hk, cl, min_len, max_len;
};

struct TCExpandParams {
    CUtensorMap tmap_b;    // B as [L][r][H2], box {64, r, 1}
    CUtensorMap tmap_vhi;  // v hi as [T][r], box {64, 128}
    CUtensorMap tmap_vlo;
    void *y;
    const int32_t *perm, *seg_ptr, *idx;
    int *err;
    int32_t S, T, L, H2, r, min_len, max_len;
    int32_t kw;   // weight of a tile = its rows + kw (B bytes of a column block in y rows)
    int32_t red;  // fp32 y updated by bulk reductions in L2 (H2 % 4 == 0)
    int32_t ny;   // y stages per epilogue group (1 or 2)
    int32_t nbs;  // B stages (2 .. kExpandBStages)
    int *claim;      // counter of claimed chunks (zeroed by the shrink kernel)
    int32_t sfrac;   // static part of the work line in 64ths (64: no claiming)
    int32_t chunk;   // column blocks per claim
    float scale;
};

// Claimed blocks of the expand: descriptors handed from the B warp (which
// claims) to the MMA warp and the epilogue group of the block.
constexpr int kDynSlots = 4;  // descriptors in flight
constexpr int kDynAhead = 3;  // block k is claimed once block k - 3 has left its accumulator
struct DynSlot {
    int col, p0, end, pad;
    int row[kTcRows];
};

// ---------------------------------------------------------------- shrink
template <typename Tin>
__global__ void __launch_bounds__(kTcThreads)
    sgmv_tc_shrink_kernel(const __grid_constant__ TCShrinkParams P) {
    // Parameters read once into registers (see the CUDA-core kernel); the
    // tensor map stays in the parameter buffer, where TMA reads it.
    const int32_t *const seg_ptr = P.seg_ptr;
    const int32_t *const idx = P.idx;
    const int32_t *const perm = P.perm;
    int *const err = P.err;
    const int nseg = P.S, nrows_all = P.T, nadapters = P.L, min_len = P.min_len,
              max_len = P.max_len, ncl = P.cl, rk = P.r, hk = P.hk, H1 = P.H1;
    const void *const xptr = P.x;
    void *const vhi_ptr = P.vhi;
    void *const vlo_ptr = P.vlo;
    const CUtensorMap *const tmap_a = &P.tmap_a;

    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], done;
    __shared__ int s_info[4];
    __shared__ int s_xrow[kTcRows];  // physical row of each tile row, -1 past the tile
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool report = blockIdx.x == 0 && blockIdx.y == 0;

    if (warp == 0) {
        find_tile(seg_ptr, idx, nseg, nrows_all, nadapters, kTcRows, min_len, max_len, err,
                  blockIdx.y, false, report, s_info);
        if (lane == 0) {
            for (int s = 0; s < kStages; ++s) {
                mbar_init(&full[s], kShrinkProducers + 1);  // cp.async arrivals + the TMA one
                mbar_init(&empty[s], 1);
            }
            mbar_init(&done, 1);
            mbar_init_fence();
        }
    }
    __syncthreads();
    if (s_info[0] < 0) return;  // same decision in every CTA of the cluster
    const int p0 = s_info[1], nrows = s_info[2], a = s_info[3];
    const bool clustered = ncl > 1;
    if (warp == 0) tmem_alloc(&s_tmem, (uint32_t)rk);

    uint8_t *base = align1024(dsm);
    const uint32_t x_bytes = kTcRows * kKB * sizeof(Tin);  // 16 KB
    const uint32_t a_bytes = kKB * rk * sizeof(Tin);       // 8 or 16 KB
    auto stage_x = [&](int st) { return base + st * (x_bytes + a_bytes); };
    auto stage_a = [&](int st) { return base + st * (x_bytes + a_bytes) + x_bytes; };
    // partials of v from the cluster: in the ring's memory, once every CTA's
    // products are made
    float *recv = reinterpret_cast<float *>(base);
    const Tin *gX = static_cast<const Tin *>(xptr);

    const int k0 = (int)blockIdx.x * hk;
    const int k1 = min(H1, k0 + hk);
    const int nkb = k1 > k0 ? (k1 - k0 + kKB - 1) / kKB : 0;

    auto issue_a = [&](int kb) {  // thread kTcThreads - kShrinkProducers (first producer)
        const int st = kb % kStages;
        mbar_arrive_expect_tx(&full[st], a_bytes);
        for (int c = 0; c < rk; c += 64)
            tma_load_3d(stage_a(st) + c * kKB * sizeof(Tin), tmap_a, c, k0 + kb * kKB, a,
                        &full[st]);
    };
    // Warp 0 issues the MMAs (lane 0); warps 1-3 are the producers: the
    // first of them loads A by TMA, all of them gather the tile's X rows.
    const int prod = tid - (kTcThreads - kShrinkProducers);  // producer index, < 0 in warp 0
    if (prod == 0)
        for (int kb = 0; kb < min(nkb, kStages); ++kb) issue_a(kb);

    // Physical rows of this producer's tile rows prod and prod + kShrinkProducers
    // (metadata is complete before launch).
    auto phys = [&](int m) {
        if (m >= nrows) return -1;
        int row = perm ? perm[p0 + m] : p0 + m;
        if (row < 0 || row >= nrows_all) {
            set_error(err, kErrBadIndex);
            row = -1;
        }
        return row;
    };
    if (tid < kTcRows) s_xrow[tid] = phys(tid);
    __syncthreads();
    // Every producer: (row, 16-byte chunk) pairs e = prod, prod + 96, ... of
    // the 128 x 8 in a k-block, so that a warp reads 4 whole 128-byte row
    // pieces per instruction.
    auto issue_x = [&](int kb) {
        const int st = kb % kStages;
        uint8_t *xs = stage_x(st);
        const int kk0 = k0 + kb * kKB;
        for (int e = prod; e < kTcRows * 8; e += kShrinkProducers) {
            const int m = e >> 3, c = e & 7;
            const int row = s_xrow[m];
            const int k = kk0 + c * 8;
            const bool ok = row >= 0 && k < k1;
            cp_async16(xs + sw128_offset(m, c), ok ? gX + (size_t)row * H1 + k : gX, ok ? 16u : 0u);
        }
        cp_async_arrive(&full[st]);
    };
    pdl_wait();
    // the expand that follows claims blocks from this counter (the previous
    // kernel, which may have used it, is complete)
    if (P.claim && report && tid == 0) *P.claim = 0;
    if (prod >= 0)
        for (int kb = 0; kb < min(nkb, kStages); ++kb) issue_x(kb);
    pdl_trigger();

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t idesc = idesc_f16(std::is_same<Tin, __nv_bfloat16>::value, kTcRows, rk);
    bool lost = false;
    if (tid == 0) {
        // MMA issuer: each k-block once its stage is full, then the stage back
        for (int kb = 0; kb < nkb; ++kb) {
            const int st = kb % kStages;
            const uint32_t ph = (uint32_t)((kb / kStages) & 1);
            if (!mbar_wait(&full[st], ph)) {
                lost = true;
                set_error(err, kErrTimeout);
                mbar_wait(&full[st], ph);
            }
            fence_proxy_async();  // cp.async (generic proxy) data -> tensor core (async proxy)
            tc_fence_after();
            const uint32_t xa = smem_addr(stage_x(st)), aa = smem_addr(stage_a(st));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_f16(tmem, sw128_desc(xa + kk * 32, 16, 1024),
                        sw128_desc(aa + kk * 2048, kKB * 128, 1024), idesc, (kb | kk) != 0);
            mma_commit(&empty[st]);
        }
    } else if (prod >= 0) {
        // producers: refill a stage once the MMAs that read it are done; one
        // producer waits, a producer-only barrier releases the others
        for (int kb = kStages; kb < nkb; ++kb) {
            const int st = kb % kStages;
            const uint32_t ph = (uint32_t)(((kb / kStages) - 1) & 1);
            if (prod == 0 && !mbar_wait(&empty[st], ph)) {
                set_error(err, kErrTimeout);
                mbar_wait(&empty[st], ph);
                lost = true;
            }
            named_sync<1, kShrinkProducers>();
            if (prod == 0) issue_a(kb);
            issue_x(kb);
        }
    }
    {
        int bad = 0;
        if (tid == 0) {
            mma_commit(&done);
            if (!mbar_wait(&done, 0)) {
                set_error(err, kErrTimeout);
                mbar_wait(&done, 0);
                bad = 1;
            }
        }
        if (__syncthreads_or(bad)) lost = true;
    }
    tc_fence_after();

    // Partial v of this CTA's H1 slice -> the CTA that owns the row.
    const int rpc = kTcRows / ncl;  // rows summed by each CTA of the cluster
    const int rank = (int)blockIdx.x;
    // every CTA of the cluster is done with its ring (and has started, so
    // its shared memory can be written)
    if (clustered) cluster_sync();
    for (int c0 = 0; c0 < rk; c0 += 32) {
        float v[32];
        if (nkb > 0) {
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        if (tid < nrows) {
            const int owner = tid / rpc, mr = tid - (tid / rpc) * rpc;
            float *dst = recv + (size_t)(rank * rpc + mr) * rk + c0;
            if (clustered) {
                const uint32_t pa = peer_addr(dst, (uint32_t)owner);
#pragma unroll
                for (int j = 0; j < 32; j += 4) st_peer4(pa + j * 4, v[j], v[j + 1], v[j + 2], v[j + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) stsf(dst + j, v[j]);
            }
        }
    }
    if (clustered)
        cluster_sync();
    else
        __syncthreads();
    Tin *vhi = static_cast<Tin *>(vhi_ptr);
    Tin *vlo = static_cast<Tin *>(vlo_ptr);
    // four consecutive columns per thread, partials summed in rank order
    const int rq = rk / 4;
    for (int e = tid; e < rpc * rq; e += kTcThreads) {
        const int mr = e / rq, col = 4 * (e - mr * rq);
        const int m = rank * rpc + mr;
        if (m >= nrows || lost) continue;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int c = 0; c < ncl; ++c) {
            const uint4 u = lds128(recv + (size_t)(c * rpc + mr) * rk + col);
            s[0] += __uint_as_float(u.x);
            s[1] += __uint_as_float(u.y);
            s[2] += __uint_as_float(u.z);
            s[3] += __uint_as_float(u.w);
        }
        __align__(8) Tin hv[4], lv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            hv[q] = from_f<Tin>(s[q]);
            lv[q] = from_f<Tin>(s[q] - to_f<Tin>(hv[q]));
        }
        const size_t o = (size_t)(p0 + m) * rk + col;
        *reinterpret_cast<uint2 *>(vhi + o) = *reinterpret_cast<const uint2 *>(hv);
        *reinterpret_cast<uint2 *>(vlo + o) = *reinterpret_cast<const uint2 *>(lv);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, (uint32_t)rk);
}

// ---------------------------------------------------------------- expand
// Columns of H2 per expand CTA: 128 for 16-bit y, 64 for fp32 y (the y tile
// staged in shared memory then stays at 32 KB and two or more CTAs fit per SM).
// Barrier of one 128-thread epilogue group (named barriers 1 and 2).
__device__ __forceinline__ void group_sync(int g) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "n"(kTcRows) : "memory");
}
template <typename Ty> constexpr int tc_cols() { return sizeof(Ty) == 4 ? 64 : 128; }
// Bytes of one staged y row: the tile's columns plus 16 bytes, so that the
// 16-byte accesses of 8 consecutive rows fall in different banks.
template <typename Ty> constexpr int tc_ypitch() { return tc_cols<Ty>() * (int)sizeof(Ty) + 16; }

template <typename Tin, typename Ty>
__global__ void __launch_bounds__(kExpandThreads, 1)
    sgmv_tc_expand_kernel(const __grid_constant__ TCExpandParams P) {
    constexpr int N = tc_cols<Ty>();   // columns of one block
    constexpr int YP = tc_ypitch<Ty>();
    constexpr int CH = N * (int)sizeof(Ty) / 16;  // 16-byte chunks of a row's block (16)
    constexpr int RPI = kTcRows / CH;              // rows covered by one pass of a group (8)
    constexpr int E16 = 16 / (int)sizeof(Ty);      // elements per chunk
    constexpr int NACC = 256 / N;                  // TMEM accumulator buffers (4 or 2)
    const int32_t *const seg_ptr = P.seg_ptr;
    const int32_t *const idx = P.idx;
    const int32_t *const perm = P.perm;
    int *const err = P.err;
    const int nseg = P.S, nrows_all = P.T, nadapters = P.L, min_len = P.min_len,
              max_len = P.max_len, rk = P.r, H2 = P.H2, ny = P.ny, nbs = P.nbs;
    const float scale = P.scale;
    Ty *const gY = static_cast<Ty *>(P.y);
    const CUtensorMap *const tmap_b = &P.tmap_b;
    const CUtensorMap *const tmap_vhi = &P.tmap_vhi;
    const CUtensorMap *const tmap_vlo = &P.tmap_vlo;

    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ __align__(8) uint64_t bar_v, b_full[kExpandBStages], b_empty[kExpandBStages];
    __shared__ __align__(8) uint64_t acc_full[4], acc_empty[4], y_full[2][kExpandYStages];
    __shared__ __align__(8) uint64_t d_full[kDynSlots], d_empty[kDynSlots];
    __shared__ Run s_run;
    __shared__ DynTable s_dyn;
    __shared__ int s_row[kMaxPieces][kTcRows];
    __shared__ __align__(16) DynSlot s_slot[kDynSlots];
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool report = blockIdx.x == 0 && blockIdx.y == 0;

    const int nblk = (H2 + N - 1) / N;

    if (warp == 0) {
        find_run(seg_ptr, idx, nseg, nrows_all, nadapters, kTcRows, P.kw, nblk, min_len, max_len,
                 err, (int)blockIdx.x, (int)gridDim.x, report, P.sfrac, &s_run, &s_dyn);
        if (lane == 0) {
            mbar_init(&bar_v, 1);
            for (int i = 0; i < kDynSlots; ++i) {
                mbar_init(&d_full[i], 1);                // the B warp, once it is written
                mbar_init(&d_empty[i], 1 + kTcRows);     // the MMA warp + the epilogue group's threads
            }
            for (int i = 0; i < nbs; ++i) {
                mbar_init(&b_full[i], 1);
                mbar_init(&b_empty[i], 1);
            }
            for (int b = 0; b < NACC; ++b) {
                mbar_init(&acc_full[b], 1);
                mbar_init(&acc_empty[b], kTcRows / 32);  // one arrival per warp of its group
            }
            for (int g = 0; g < 2; ++g)
                for (int i = 0; i < ny; ++i) mbar_init(&y_full[g][i], kTcRows);  // cp.async, per thread
            mbar_init_fence();
        }
    }
    __syncthreads();
    // this CTA's static run: blocks 0 .. nb-1 of its sequence, piece q
    // holding blocks k0[q] .. k0[q+1]-1 = column blocks b0[q], ... of one
    // tile; then, when the work line has a claimed part, blocks nb, nb+1, ...
    // claimed at run time (P.chunk at a time) until none is left
    const int npc = s_run.n;
    const int nb = npc > 0 ? s_run.k0[npc] : 0;
    const bool dyn = s_dyn.n > 0;
    const int nd = dyn ? s_dyn.d0[s_dyn.n] : 0;
    if (nb <= 0 && !dyn) return;
    auto piece_of = [&](int k) {
        int q = 0;
        while (q + 1 < npc && k >= s_run.k0[q + 1]) ++q;
        return q;
    };
    auto col_of = [&](int k, int q) { return (s_run.b0[q] + k - s_run.k0[q]) * N; };
    if (warp == 0) tmem_alloc(&s_tmem, (uint32_t)(NACC * N));

    uint8_t *base = align1024(dsm);
    const uint32_t v_bytes = (uint32_t)rk * 256u;   // [128 rows][r] 16-bit, as r/64 K-blocks
    const uint32_t b_bytes = (uint32_t)rk * N * 2u;  // N/64 N-atoms of [r rows][64 columns]
    uint8_t *vhi_tile = base;
    uint8_t *vlo_tile = base + v_bytes;
    uint8_t *b_stage0 = base + 2 * v_bytes;
    uint8_t *y_stage0 = b_stage0 + (size_t)nbs * b_bytes;  // [2 groups][ny][128 rows][YP]
    const uint32_t ystage_bytes = (uint32_t)kTcRows * YP;

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    pdl_trigger();

    if (warp == 2 * kTcRows / 32 + 1) {
        // ---- B warp: B[a][:, block k] through the ring, a stage refilled as
        // soon as the products that read it are made; it also claims the
        // blocks after the static run and hands them on in s_slot
        auto load_b_at = [&](int k, int j, int a) {
            const int st = k % nbs;
            mbar_arrive_expect_tx(&b_full[st], b_bytes);
            for (int c = 0; c < N; c += 64)
                tma_load_3d(b_stage0 + (size_t)st * b_bytes + c * rk * 2, tmap_b, j + c, 0, a,
                            &b_full[st]);
        };
        bool ok = true;
        if (lane == 0) {
            auto load_b = [&](int k) {
                const int q = piece_of(k);
                load_b_at(k, col_of(k, q), s_run.a[q]);
            };
            for (int k = 0; k < min(nbs, nb); ++k) load_b(k);  // weights: before the wait
            for (int k = nbs; k < nb; ++k) {
                if (!mbar_wait(&b_empty[k % nbs], (uint32_t)(((k / nbs) - 1) & 1))) {
                    set_error(err, kErrTimeout);
                    ok = false;
                    break;
                }
                load_b(k);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (dyn && ok) {
            pdl_wait();  // the counter is zeroed by the shrink kernel
            int pj = 0, pend = 0;  // claimed blocks not handed on yet: pj .. pj + pend - 1
            for (int k = nb, kd = 0;; ++k, ++kd) {
                const int sl = kd % kDynSlots;
                // claim late: once block k - kDynAhead has left its accumulator
                // (with NACC >= kDynAhead that phase cannot have been passed)
                if (k >= kDynAhead)
                    ok = mbar_wait(&acc_empty[(k - kDynAhead) % NACC],
                                   (uint32_t)(((k - kDynAhead) / NACC) & 1));
                if (ok && kd >= kDynSlots)
                    ok = mbar_wait(&d_empty[sl], (uint32_t)(((kd / kDynSlots) - 1) & 1));
                ok = __all_sync(0xffffffffu, ok);  // one decision for the whole warp
                if (!ok) {
                    if (lane == 0) set_error(err, kErrTimeout);
                    break;
                }
                if (pend == 0) {
                    int c0 = 0;
                    if (lane == 0) c0 = atomicAdd(P.claim, 1);
                    c0 = __shfl_sync(0xffffffffu, c0, 0);
                    pj = c0 * P.chunk;
                    pend = max(0, min(P.chunk, nd - pj));
                }
                DynSlot *ds = &s_slot[sl];
                if (pend == 0) {
                    // nothing left: an end mark here and in the next slot (the
                    // next block of the other epilogue group)
                    if (lane == 0) {
                        ds->end = 1;
                        mbar_arrive(&d_full[sl]);
                    }
                    const int kd2 = kd + 1, sl2 = kd2 % kDynSlots;
                    if (kd2 >= kDynSlots)
                        ok = mbar_wait(&d_empty[sl2], (uint32_t)(((kd2 / kDynSlots) - 1) & 1));
                    if (!__all_sync(0xffffffffu, ok)) {
                        if (lane == 0) set_error(err, kErrTimeout);
                        break;
                    }
                    if (lane == 0) {
                        s_slot[sl2].end = 1;
                        mbar_arrive(&d_full[sl2]);
                    }
                    break;
                }
                const int j = pj++;
                --pend;
                int t = 0;  // the tile of claimed block j
                while (t + 1 < s_dyn.n && j >= s_dyn.d0[t + 1]) ++t;
                const int col = (s_dyn.b0[t] + j - s_dyn.d0[t]) * N, p0 = s_dyn.p0[t];
                const int nr = s_dyn.rows[t];
                for (int r = lane; r < kTcRows; r += 32) {
                    int row = -1;
                    if (r < nr) {
                        row = perm ? perm[p0 + r] : p0 + r;
                        if (row < 0 || row >= nrows_all) {
                            set_error(err, kErrBadIndex);
                            row = -1;
                        }
                    }
                    ds->row[r] = row;
                }
                if (lane == 0) {
                    ds->col = col;
                    ds->p0 = p0;
                    ds->end = 0;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&d_full[sl]);
                // its B, once the stage is free (the whole warp waits)
                if (k >= nbs) ok = mbar_wait(&b_empty[k % nbs], (uint32_t)(((k / nbs) - 1) & 1));
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    if (lane == 0) set_error(err, kErrTimeout);
                    break;
                }
                if (lane == 0) load_b_at(k, col, s_dyn.a[t]);
                __syncwarp();
            }
        }
    } else if (warp == 2 * kTcRows / 32) {
        // ---- MMA warp: each piece's v (its tile's rows), then the products of
        // block k into accumulator buffer k % NACC (read by epilogue group k & 1)
        if (lane == 0) {
            pdl_wait();  // v: written by the shrink kernel
            bool ok = true;
            // after a wait runs out, later ones are skipped: the error is set
            // and every wait of the compute warps is bounded as well
            auto pwait = [&](uint64_t *bar, uint32_t par) {
                if (ok) ok = mbar_wait(bar, par);
            };
            const uint32_t idesc = idesc_f16(std::is_same<Tin, __nv_bfloat16>::value, kTcRows, N);
            int vp0 = -1, nv = 0;  // tile (first position) of the v in shared memory; v loads
            for (int k = 0;; ++k) {
                const int st = k % nbs, ab = k % NACC;
                int p0;
                if (k < nb) {
                    p0 = s_run.p0[piece_of(k)];
                } else {
                    if (!dyn) break;
                    const int kd = k - nb, sl = kd % kDynSlots;
                    pwait(&d_full[sl], (uint32_t)((kd / kDynSlots) & 1));
                    if (!ok || s_slot[sl].end) break;
                    p0 = s_slot[sl].p0;
                    mbar_arrive(&d_empty[sl]);
                }
                if (p0 != vp0) {
                    // v of another tile: once the products of the previous
                    // block (the last to read the old v) are made.  The
                    // epilogue is still draining up to NACC accumulators.
                    if (k > 0) pwait(&acc_full[(k - 1) % NACC], (uint32_t)(((k - 1) / NACC) & 1));
                    mbar_arrive_expect_tx(&bar_v, 2 * v_bytes);
                    for (int kb = 0; kb < rk / kKB; ++kb) {
                        tma_load_2d(vhi_tile + kb * 16384, tmap_vhi, kb * kKB, p0, &bar_v);
                        tma_load_2d(vlo_tile + kb * 16384, tmap_vlo, kb * kKB, p0, &bar_v);
                    }
                    pwait(&bar_v, (uint32_t)(nv & 1));
                    ++nv;
                    vp0 = p0;
                }
                pwait(&b_full[st], (uint32_t)((k / nbs) & 1));
                if (k >= NACC) pwait(&acc_empty[ab], (uint32_t)(((k / NACC) - 1) & 1));
                tc_fence_after();
                const uint32_t ba = smem_addr(b_stage0 + (size_t)st * b_bytes);
                const uint32_t d = tmem + (uint32_t)(ab * N);
                uint32_t acc = 0;
                for (int h = 0; h < 2; ++h) {
                    const uint32_t va = smem_addr(h ? vlo_tile : vhi_tile);
                    for (int kb = 0; kb < rk / kKB; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            mma_f16(d, sw128_desc(va + kb * 16384 + kk * 32, 16, 1024),
                                    sw128_desc(ba + (kb * 4 + kk) * 2048, (uint32_t)rk * 128, 1024),
                                    idesc, acc);
                            acc = 1;
                        }
                }
                mma_commit(&acc_full[ab]);
                mma_commit(&b_empty[st]);
            }
            if (!ok) set_error(err, kErrTimeout);
        }
    } else {
        // ---- epilogue groups: group g (warps 4g .. 4g+3, one tile row per
        // thread, TMEM lanes of warp % 4) takes blocks g, g + 2, ...
        const int g = warp >> 2, lt = tid & (kTcRows - 1);
        const int nmine = (nb - g + 1) >> 1;  // blocks of this group
        // physical rows of the pieces' tiles (group g looks up pieces g, g + 2;
        // the loads are independent, so they are in flight together)
        {
            int row[(kMaxPieces + 1) / 2];
            bool in[(kMaxPieces + 1) / 2];
#pragma unroll
            for (int h = 0; h < (kMaxPieces + 1) / 2; ++h) {
                const int q = g + 2 * h;
                in[h] = q < npc && lt < s_run.rows[q];
                row[h] = -1;
                if (in[h]) row[h] = perm ? perm[s_run.p0[q] + lt] : s_run.p0[q] + lt;
            }
#pragma unroll
            for (int h = 0; h < (kMaxPieces + 1) / 2; ++h) {
                const int q = g + 2 * h;
                if (q >= npc) continue;
                if (in[h] && (row[h] < 0 || row[h] >= nrows_all)) {
                    set_error(err, kErrBadIndex);
                    row[h] = -1;
                }
                s_row[q][lt] = row[h];
            }
            // both groups' rows are in (the two epilogue groups only)
            asm volatile("bar.sync 3, %0;" ::"n"(2 * kTcRows) : "memory");
        }
        uint8_t *my_y = y_stage0 + (size_t)g * ny * ystage_bytes;
        // y of the group's i-th block into stage i % ny: thread lt copies chunk
        // lt % CH of rows lt / CH + RPI * j (two 256-byte row pieces per warp
        // instruction)
        auto load_y = [&](int i) {
            uint8_t *st = my_y + (size_t)(i % ny) * ystage_bytes;
            const int k = g + 2 * i, q = piece_of(k);
            const int j = col_of(k, q);
            const int c = lt % CH;
            const bool col_ok = j + c * E16 < H2;
#pragma unroll 4
            for (int r = lt / CH; r < kTcRows; r += RPI) {
                const int row = s_row[q][r];
                if (row >= 0 && col_ok)
                    cp_async16(st + r * YP + c * 16, gY + (size_t)row * H2 + j + c * E16, 16);
            }
            cp_async_arrive(&y_full[g][i % ny]);
        };
        bool lost = false;
        auto wait = [&](uint64_t *bar, uint32_t par) {
            if (!mbar_wait(bar, par)) {
                set_error(err, kErrTimeout);
                mbar_wait(bar, par);
                lost = true;
            }
        };
        pdl_wait();  // y may be written by the previous kernel
        if (P.red) {
            // fp32 y: y += scale * acc by one bulk reduction per row and block,
            // added in L2, so y never passes through the SM.  Stage i % ny
            // holds scale * acc of the group's i-th block, one row per thread.
            for (int i = 0;; ++i) {
                const int k = g + 2 * i, ab = k % NACC;
                int my_row, j;
                if (k < nb) {
                    const int q = piece_of(k);
                    my_row = s_row[q][lt];
                    j = col_of(k, q);
                } else {
                    // a claimed block: its descriptor, then the slot back
                    if (!dyn) break;
                    const int kd = k - nb, sl = kd % kDynSlots;
                    wait(&d_full[sl], (uint32_t)((kd / kDynSlots) & 1));
                    if (lost || s_slot[sl].end) break;
                    my_row = s_slot[sl].row[lt];
                    j = s_slot[sl].col;
                    mbar_arrive(&d_empty[sl]);
                }
                wait(&acc_full[ab], (uint32_t)((k / NACC) & 1));
                tc_fence_after();
                if (i >= ny) {  // the reduction that last read this stage is done with it
                    if (ny == 2) bulk_wait_read1();
                    else bulk_wait_read();
                }
                uint8_t *yr = my_y + (size_t)(i % ny) * ystage_bytes + (size_t)lt * YP;
                for (int c0 = 0; c0 < N; c0 += 32) {
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(ab * N + c0), v);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        sts128(yr + (c0 + 4 * q) * 4,
                               make_uint4(__float_as_uint(scale * v[4 * q]),
                                          __float_as_uint(scale * v[4 * q + 1]),
                                          __float_as_uint(scale * v[4 * q + 2]),
                                          __float_as_uint(scale * v[4 * q + 3])));
                }
                // the accumulator buffer is free for block k + NACC
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[ab]);
                fence_proxy_async();  // this thread's row -> the bulk copy unit
                if (!lost && my_row >= 0)
                    bulk_s2g_add_f32(reinterpret_cast<float *>(gY) + (size_t)my_row * H2 + j, yr,
                                     (uint32_t)min(N, H2 - j) * 4u);
                bulk_commit();
            }
            bulk_wait_all();
        } else {
        // (16-bit y: static runs only, the host asks for no claiming)
        for (int i = 0; i < min(ny, nmine); ++i) load_y(i);
        for (int i = 0; i < nmine; ++i) {
            const int k = g + 2 * i, ab = k % NACC, q = piece_of(k);
            const int my_row = s_row[q][lt];
            wait(&acc_full[ab], (uint32_t)((k / NACC) & 1));
            tc_fence_after();
            wait(&y_full[g][i % ny], (uint32_t)((i / ny) & 1));
            // y row in shared memory += scale * accumulator row, 32 columns at a time
            uint8_t *st = my_y + (size_t)(i % ny) * ystage_bytes;
            uint8_t *yr = st + (size_t)lt * YP;
            for (int c0 = 0; c0 < N; c0 += 32) {
                float v[32];
                tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(ab * N + c0), v);
                if (my_row >= 0) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        Ty *p = reinterpret_cast<Ty *>(yr) + c0 + q * 8;
                        float y[8];
                        lds8<Ty>(p, y);
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = fmaf(scale, v[q * 8 + e], y[e]);
                        sts8<Ty>(p, y);
                    }
                }
            }
            // the accumulator buffer is free for block k + NACC
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ab]);
            group_sync(g);
            // write the block back: 16-byte stores, two row pieces per warp instruction
            {
                const int j = col_of(k, q);
                const int c = lt % CH;
                if (!lost && j + c * E16 < H2) {
#pragma unroll 4
                    for (int r = lt / CH; r < kTcRows; r += RPI) {
                        const int row = s_row[q][r];
                        if (row >= 0)
                            *reinterpret_cast<uint4 *>(gY + (size_t)row * H2 + j + c * E16) =
                                lds128(st + r * YP + c * 16);
                    }
                }
            }
            group_sync(g);  // stage i % ny has been read: refill it
            if (i + ny < nmine) load_y(i + ny);
        }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)(NACC * N));
    }
}

// ---------------------------------------------------------------- host side
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library does not link libcuda), looked up once.
EncodeTiledFn tiled_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

bool tmap_encode(CUtensorMap *m, bool bf16, int rank, const void *ptr, const cuuint64_t *dims,
                 const cuuint64_t *strides, const cuuint32_t *box, bool swizzle128) {
    EncodeTiledFn fn = tiled_encoder();
    if (!fn) return false;
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
              (cuuint32_t)rank, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

bool encode(CUtensorMap *m, bool bf16, int rank, const void *ptr, const cuuint64_t *dims,
            const cuuint64_t *strides, const cuuint32_t *box) {
    return sgmv::tmap_encode(m, bf16, rank, ptr, dims, strides, box, true);
}

template <typename K, typename P>
int launch(K kernel, const P &params, dim3 grid, int cluster, size_t smem, cudaStream_t stream,
           int threads = kTcThreads) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (cluster > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)cluster;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = (unsigned)na;
    return (int)cudaLaunchKernelEx(&cfg, kernel, params);
}

template <typename Tin, typename Ty>
int tc_launch_t(const TCArgs &g) {
    const bool bf16 = std::is_same<Tin, __nv_bfloat16>::value;
    const size_t es = sizeof(Tin);
    // -- shrink: CL CTAs split H1 in multiples of 64 columns, each with >= 1 k-block
    int cl = 8;
    while (cl > 1 && (g.H1 + kKB - 1) / kKB < cl) cl >>= 1;
    int hk = (int)(((g.H1 + cl - 1) / cl + kKB - 1) / kKB * kKB);
    while (cl > 1 && (cl - 1) * hk >= g.H1) {
        cl >>= 1;
        hk = (int)(((g.H1 + cl - 1) / cl + kKB - 1) / kKB * kKB);
    }
    TCShrinkParams sp;
    memset(&sp, 0, sizeof sp);
    {
        const cuuint64_t dims[3] = {(cuuint64_t)g.r, (cuuint64_t)g.H1, (cuuint64_t)g.L};
        const cuuint64_t strides[2] = {(cuuint64_t)g.r * es, (cuuint64_t)g.H1 * g.r * es};
        const cuuint32_t box[3] = {64, 64, 1};
        if (!encode(&sp.tmap_a, bf16, 3, g.A, dims, strides, box)) return (int)cudaErrorInvalidValue;
    }
    sp.x = g.x;
    sp.perm = g.perm;
    sp.seg_ptr = g.seg_ptr;
    sp.idx = g.idx;
    sp.err = g.err;
    sp.vhi = g.vhi;
    sp.vlo = g.vlo;
    // the claim counter: the workspace's 256 bytes after v's two halves
    int *const claim = reinterpret_cast<int *>(static_cast<uint8_t *>(g.vlo) +
                                               ((size_t)g.T * g.r * es + 255u) / 256u * 256u);
    sp.claim = claim;
    sp.S = g.S;
    sp.T = g.T;
    sp.L = g.L;
    sp.H1 = g.H1;
    sp.r = g.r;
    sp.hk = hk;
    sp.cl = cl;
    sp.min_len = g.min_len;
    sp.max_len = g.max_len;
    const size_t shrink_smem =
        1024 + std::max((size_t)kStages * (kTcRows * kKB + kKB * g.r) * es, (size_t)kTcRows * g.r * 4);
    int rc = launch(sgmv_tc_shrink_kernel<Tin>, sp, dim3((unsigned)cl, (unsigned)g.slots, 1), cl,
                    shrink_smem, g.stream);
    if (rc != 0) return rc;

    // -- expand
    TCExpandParams ep;
    memset(&ep, 0, sizeof ep);
    {
        const cuuint64_t dims[3] = {(cuuint64_t)g.H2, (cuuint64_t)g.r, (cuuint64_t)g.L};
        const cuuint64_t strides[2] = {(cuuint64_t)g.H2 * es, (cuuint64_t)g.r * g.H2 * es};
        const cuuint32_t box[3] = {64, (cuuint32_t)g.r, 1};
        if (!encode(&ep.tmap_b, bf16, 3, g.B, dims, strides, box)) return (int)cudaErrorInvalidValue;
        const cuuint64_t vd[2] = {(cuuint64_t)g.r, (cuuint64_t)g.T};
        const cuuint64_t vs[1] = {(cuuint64_t)g.r * es};
        const cuuint32_t vb[2] = {64, (cuuint32_t)kTcRows};
        if (!encode(&ep.tmap_vhi, bf16, 2, g.vhi, vd, vs, vb)) return (int)cudaErrorInvalidValue;
        if (!encode(&ep.tmap_vlo, bf16, 2, g.vlo, vd, vs, vb)) return (int)cudaErrorInvalidValue;
    }
    ep.y = g.y;
    ep.perm = g.perm;
    ep.seg_ptr = g.seg_ptr;
    ep.idx = g.idx;
    ep.err = g.err;
    ep.S = g.S;
    ep.T = g.T;
    ep.L = g.L;
    ep.H2 = g.H2;
    ep.r = g.r;
    ep.min_len = g.min_len;
    ep.max_len = g.max_len;
    ep.scale = g.scale;
    constexpr int N = tc_cols<Ty>();
    // One CTA per SM (a multiple of the SM count when there are more tiles),
    // dealt to the tiles in proportion to the bytes they move: y rows read
    // and written, plus B once per column block (r / sizeof(y) rows' worth).
    const int64_t nsm = std::max<int64_t>(1, g.nsm);
    const int64_t nct = (((int64_t)g.slots + nsm - 1) / nsm) * nsm;
    if (nct > 0x7fffffff) return (int)cudaErrorInvalidValue;
    ep.kw = (int32_t)std::max<int64_t>(1, g.r / (int64_t)sizeof(Ty)) + kExpandBlockRows;
    // fp32 rows of whole 16-byte pieces: y += delta by bulk reductions
    ep.red = std::is_same<Ty, float>::value && g.H2 % 4 == 0 ? 1 : 0;
    // With bulk reductions, the last quarter of the work line is claimed at
    // run time, four column blocks at a time: CTAs on SMs that stream faster
    // take more of it (CTAs with equal static shares end up to 1.7x apart).
    // Measured on the prefill batch (µs per call back to back): 57.8-58.0
    // against 59.2 with no claiming; a claimed 3/8 took 59.5-61.5, claims of
    // two or six blocks 59.2-59.8.
    // (claiming relies on NACC >= kDynAhead accumulators, true for fp32 y)
    static_assert(256 / tc_cols<float>() >= kDynAhead, "claims run too far ahead");
    ep.claim = claim;
    ep.sfrac = ep.red ? 48 : 64;
    ep.chunk = 4;
    // v once, B ring, two y stages per epilogue group: as deep as fits
    const size_t vb = (size_t)2 * g.r * 256, bstage = (size_t)g.r * N * 2;
    const size_t ystage = (size_t)kTcRows * tc_ypitch<Ty>();
    ep.nbs = kExpandBStages;
    ep.ny = kExpandYStages;
    auto total = [&]() { return 1024 + vb + ep.nbs * bstage + (size_t)2 * ep.ny * ystage; };
    // dynamic shared memory: what the block may have, less the kernel's static part
    size_t cap = kExpandSmemMax;
    {
        int dev = 0, optin = 0;
        cudaFuncAttributes fa;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
            cudaFuncGetAttributes(&fa, sgmv_tc_expand_kernel<Tin, Ty>) == cudaSuccess &&
            (size_t)optin > fa.sharedSizeBytes)
            cap = std::min(cap, (size_t)optin - fa.sharedSizeBytes);
    }
    while (total() > cap && ep.nbs > 2) --ep.nbs;
    if (total() > cap) ep.ny = 1;
    while (total() > cap && ep.nbs > 2) --ep.nbs;
    const size_t expand_smem = total();
    return launch(sgmv_tc_expand_kernel<Tin, Ty>, ep, dim3((unsigned)nct, 1, 1), 1, expand_smem,
                  g.stream, kExpandThreads);
}

template <typename Tin>
int tc_launch_in(const TCArgs &g) {
    switch (g.y_dtype) {
        case 0: return tc_launch_t<Tin, __half>(g);
        case 1: return tc_launch_t<Tin, __nv_bfloat16>(g);
        default: return tc_launch_t<Tin, float>(g);
    }
}

}  // namespace

int tc_launch(const TCArgs &g) {
    return g.in_dtype == 0 ? tc_launch_in<__half>(g) : tc_launch_in<__nv_bfloat16>(g);
}

}  // namespace sgmv
