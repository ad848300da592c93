// sgmv_device.cuh -- device helpers shared by the SGMV kernels: inline PTX for
// mbarriers, 1-D bulk (TMA) copies, thread-block clusters and distributed
// shared memory, and programmatic dependent launch; plus f16/bf16/f32 loads,
// stores and conversions.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sgmv {

// Status codes written into the device error word (same values as sgmv.h).
constexpr int kErrBadIndex = 4;
constexpr int kErrTimeout = 7;
constexpr int kErrBadSegments = 8;

// Bounds of every mbarrier wait: about one second of %globaltimer, and at most
// kMaxPolls polls.  Each poll may suspend the thread for up to kSuspendNs
// (it resumes as soon as the phase completes).
constexpr uint32_t kMaxPolls = 1u << 22;
constexpr uint32_t kSuspendNs = 20000;
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ void set_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ---- programmatic dependent launch -------------------------------------
// Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
// Makes barrier initialisation visible to the async (TMA) proxy and the cluster.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Arrive (count 1) and add `bytes` to the expected transaction count.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait for phase `parity` to complete.  Returns false if it did not.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < kMaxPolls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) break;
    }
    return false;
}

// Plain arrive (count 1) on a barrier of this CTA.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Arrive, with release semantics at cluster scope, on the barrier at the
// shared::cluster address `remote` (from peer_addr: another CTA's, or this one's).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
                 : "memory");
}
// Test for phase completion with acquire semantics at cluster scope: what the
// arriving CTAs wrote before their release-arrive is visible afterwards.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
// Bounded wait, as mbar_wait, with cluster-scope acquire.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < kMaxPolls; ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) break;
    }
    return false;
}
__device__ __forceinline__ void fence_acq_rel_cluster() {
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
}
// Barrier over the first `count` threads of the CTA (count a multiple of 32).
template <int ID, int COUNT> __device__ __forceinline__ void named_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(COUNT) : "memory");
}

// ---- 1-D bulk copy global -> shared, completes on an mbarrier --------------
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// ---- tiled tensor (TMA) load of a 3-D box, completes on an mbarrier ---------
// The innermost coordinate times the element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const void *map, int c0, int c1, int c2,
                                            int c3, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3)
        : "memory");
}

// ---- 1-D bulk copy shared -> global (bulk-group completion) ---------------
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until this thread's committed bulk copies have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Bulk reduction shared -> global, in L2: dst[i] += src[i] for `bytes` / 4
// floats (both addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_s2g_add_f32(float *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src)), "r"(bytes)
                 : "memory");
}
// ... until at most one committed group is still reading shared memory.
__device__ __forceinline__ void bulk_wait_read1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// ... until every committed bulk operation of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---- clusters / distributed shared memory ---------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// Full cluster barrier: every thread of every CTA in the cluster arrives;
// release/acquire orders shared-memory writes before it with reads after it.
// The non-.aligned forms are used so that warps need not be converged here.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// Split barrier: arrive without ordering (kernel start), wait before the first
// access to a peer's shared memory (every CTA of the cluster has started).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait;" ::: "memory");
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void *local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(local)), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_peer(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_peer(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Store 16 bytes into another CTA's shared memory (addresses from peer_addr)
// and count them on that CTA's mbarrier `remote_bar` as transaction bytes.
__device__ __forceinline__ void st_async4(uint32_t remote, float a, float b, float c, float d,
                                          uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
            remote),
        "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
        : "memory");
}

// ---- explicit shared-memory access ----------------------------------------
// Pointers into dynamic shared memory that pass through lambdas or offset
// arithmetic can lose their address space, and the generic loads the compiler
// then emits are several times slower than ld.shared here.  Hot paths use
// these instead.
__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p))
                 : "memory");
    return v;
}
__device__ __forceinline__ unsigned short lds16(const void *p) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}
__device__ __forceinline__ float ldsf(const void *p) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}
__device__ __forceinline__ void stsf(void *p, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(smem_addr(p)), "f"(v) : "memory");
}
__device__ __forceinline__ void sts128(void *p, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_addr(p)), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t lds32(const void *p) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}
__device__ __forceinline__ uint2 lds64(const void *p) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_addr(p))
                 : "memory");
    return v;
}

// ---- fused multiply-adds --------------------------------------------------
// c + a * b with 16-bit a, b and an fp32 accumulator, rounded once: the
// product of two 16-bit floats is exact in fp32, so this equals
// fmaf(float(a), float(b), c) bit for bit, without the two conversions.
template <typename T> __device__ __forceinline__ float fma16(unsigned short a, unsigned short b, float c);
template <> __device__ __forceinline__ float fma16<__half>(unsigned short a, unsigned short b, float c) {
    float d;
    asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
    return d;
}
template <> __device__ __forceinline__ float fma16<__nv_bfloat16>(unsigned short a, unsigned short b,
                                                                 float c) {
    float d;
    asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
    return d;
}
// (c0, c1) += a * (b0, b1) as one packed fp32 instruction (each lane one fmaf).
__device__ __forceinline__ void fma2(float a, float b0, float b1, float &c0, float &c1) {
    uint64_t av, bv, cv;
    asm("mov.b64 %0, {%1, %1};" : "=l"(av) : "f"(a));
    asm("mov.b64 %0, {%1, %2};" : "=l"(bv) : "f"(b0), "f"(b1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(cv) : "f"(c0), "f"(c1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(cv) : "l"(av), "l"(bv));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(c0), "=f"(c1) : "l"(cv));
}

// ---- element conversions ---------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }

// Eight consecutive 16-bit values (one 16-byte vector) widened to fp32.
template <typename T> __device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    const T *h = reinterpret_cast<const T *>(&u);
#pragma unroll
    for (int q = 0; q < 8; ++q) f[q] = to_f<T>(h[q]);
}

// Read 8 consecutive output elements at p (16 B for 16-bit types, 32 B for f32).
template <typename Ty> __device__ __forceinline__ void load8(const Ty *p, float (&f)[8]) {
    uint4 u = *reinterpret_cast<const uint4 *>(p);
    unpack8<Ty>(u, f);
}
template <> __device__ __forceinline__ void load8<float>(const float *p, float (&f)[8]) {
    float4 a = reinterpret_cast<const float4 *>(p)[0];
    float4 b = reinterpret_cast<const float4 *>(p)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
template <typename Ty> __device__ __forceinline__ void store8(Ty *p, const float (&f)[8]) {
    uint4 u;
    Ty *h = reinterpret_cast<Ty *>(&u);
#pragma unroll
    for (int q = 0; q < 8; ++q) h[q] = from_f<Ty>(f[q]);
    *reinterpret_cast<uint4 *>(p) = u;
}
template <> __device__ __forceinline__ void store8<float>(float *p, const float (&f)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
// Write 8 elements to shared memory (16 bytes, or 32 for fp32).
template <typename Ty> __device__ __forceinline__ void sts8(Ty *p, const float (&f)[8]) {
    uint4 u;
    Ty *h = reinterpret_cast<Ty *>(&u);
#pragma unroll
    for (int q = 0; q < 8; ++q) h[q] = from_f<Ty>(f[q]);
    sts128(p, u);
}
template <> __device__ __forceinline__ void sts8<float>(float *p, const float (&f)[8]) {
    sts128(p, make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                         __float_as_uint(f[3])));
    sts128(p + 4, make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                             __float_as_uint(f[7])));
}

// Two consecutive elements widened to fp32: from 32 bits of a 16-bit pair, or
// from 64 bits of an fp32 pair.
template <typename T> __device__ __forceinline__ void unpack2(uint32_t u, float &a, float &b) {
    const T *h = reinterpret_cast<const T *>(&u);
    a = to_f<T>(h[0]);
    b = to_f<T>(h[1]);
}
// y pairs: read / write two consecutive outputs (4 bytes, or 8 for fp32).
template <typename Ty> __device__ __forceinline__ void ld2(const Ty *p, float &a, float &b) {
    unpack2<Ty>(*reinterpret_cast<const uint32_t *>(p), a, b);
}
template <> __device__ __forceinline__ void ld2<float>(const float *p, float &a, float &b) {
    const float2 v = *reinterpret_cast<const float2 *>(p);
    a = v.x;
    b = v.y;
}
template <typename Ty> __device__ __forceinline__ void lds2(const Ty *p, float &a, float &b) {
    unpack2<Ty>(lds32(p), a, b);
}
template <> __device__ __forceinline__ void lds2<float>(const float *p, float &a, float &b) {
    const uint2 v = lds64(p);
    a = __uint_as_float(v.x);
    b = __uint_as_float(v.y);
}
template <typename Ty> __device__ __forceinline__ void st2(Ty *p, float a, float b) {
    uint32_t u;
    Ty *h = reinterpret_cast<Ty *>(&u);
    h[0] = from_f<Ty>(a);
    h[1] = from_f<Ty>(b);
    *reinterpret_cast<uint32_t *>(p) = u;
}
template <> __device__ __forceinline__ void st2<float>(float *p, float a, float b) {
    *reinterpret_cast<float2 *>(p) = make_float2(a, b);
}

// The same 8-element read from shared memory.
template <typename Ty> __device__ __forceinline__ void lds8(const Ty *p, float (&f)[8]) {
    unpack8<Ty>(lds128(p), f);
}
template <> __device__ __forceinline__ void lds8<float>(const float *p, float (&f)[8]) {
    const uint4 a = lds128(p), b = lds128(p + 4);
    f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
    f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
    f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
    f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
}

}  // namespace sgmv
