// sgmv_gather.cu -- many copies in one kernel: the pieces of an adapter
// loaded on demand ("Punica: Multi-Tenant LoRA Serving", nubint.ai review,
// "Proposed method" and findings: LoRA weights are loaded on demand, in
// milliseconds).
//
// One Llama-2-7B adapter is 448 pieces of 32-352 KB, one per projection and
// matrix.  As 448 copy-engine transfers each piece pays a fixed cost of a few
// microseconds; here one launch moves them all: the pieces are cut into
// 512-byte chunks, one per warp instruction (16 bytes per lane), and every
// warp keeps several chunks' loads in flight before it stores them.  The
// sources are read directly by the SMs, so they must be device-accessible:
// device memory, or page-locked host memory, which on this system the GPU
// reads over its coherent link to the CPU.  The host side checks that before
// the launch (and copies through the copy engine otherwise).
#include <algorithm>

#include "sgmv_device.cuh"
#include "sgmv_gather.h"

namespace sgmv {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 4;     // chunks in flight per warp
constexpr uint32_t kChunk = 512;     // bytes per warp instruction

struct GatherParams {
    int32_t n;
    uint64_t total;                  // chunks over all copies
    uint64_t first[kGatherMaxCopies + 1];  // first chunk of every copy (prefix sums)
    const uint8_t *src[kGatherMaxCopies];
    uint8_t *dst[kGatherMaxCopies];
    uint64_t bytes[kGatherMaxCopies];
};

// copy holding chunk k: the last i with first[i] <= k
__device__ __forceinline__ int copy_of(const GatherParams &P, uint64_t k) {
    int lo = 0, hi = P.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.first[mid] <= k) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const __grid_constant__ GatherParams P) {
    const int lane = threadIdx.x & 31;
    const uint64_t nwarps = (uint64_t)gridDim.x * (kGatherThreads / 32);
    const uint64_t w = (uint64_t)blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5);
    // the previous kernel on the stream may still read the destinations
    pdl_wait();
    for (uint64_t k0 = w; k0 < P.total; k0 += nwarps * kGatherUnroll) {
        uint4 v[kGatherUnroll];
        uint8_t *d[kGatherUnroll];
#pragma unroll
        for (int u = 0; u < kGatherUnroll; ++u) {
            const uint64_t k = k0 + (uint64_t)u * nwarps;
            d[u] = nullptr;
            if (k < P.total) {
                const int c = copy_of(P, k);
                const uint64_t off = (k - P.first[c]) * kChunk + (uint64_t)lane * 16u;
                if (off < P.bytes[c]) {
                    v[u] = __ldg(reinterpret_cast<const uint4 *>(P.src[c] + off));
                    d[u] = P.dst[c] + off;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kGatherUnroll; ++u)
            if (d[u]) *reinterpret_cast<uint4 *>(d[u]) = v[u];
    }
}

}  // namespace

int gather_launch(int32_t n, void *const *dst, const void *const *src, const uint64_t *bytes,
                  int max_ctas, cudaStream_t stream) {
    if (n < 1 || n > kGatherMaxCopies) return (int)cudaErrorInvalidValue;
    GatherParams p;
    p.n = n;
    uint64_t total = 0;
    for (int i = 0; i < n; ++i) {
        p.first[i] = total;
        p.src[i] = static_cast<const uint8_t *>(src[i]);
        p.dst[i] = static_cast<uint8_t *>(dst[i]);
        p.bytes[i] = bytes[i];
        total += (bytes[i] + kChunk - 1) / kChunk;
    }
    p.first[n] = total;
    p.total = total;
    if (total == 0) return (int)cudaSuccess;
    // no more CTAs than the chunks need, nor than the caller's cap
    const uint64_t want = (total + kGatherUnroll * (kGatherThreads / 32) - 1) /
                          (kGatherUnroll * (kGatherThreads / 32));
    const int grid = (int)std::max<uint64_t>(1, std::min<uint64_t>(want, (uint64_t)std::max(1, max_ctas)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kGatherThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, gather_kernel, p);
}

}  // namespace sgmv
