// sgmv_floor.cu -- the streaming floor of a decode-sized SGMV launch.
//
// A decode batch moves only a few MB per call ("Punica: when LoRA fine-tuned
// models need multi-tenant serving", omica.com.cn article, §2.2: the gathered
// A and B slices of each request's adapter dominate), so the call time is set
// as much by launch, ramp-up and the last CTA's tail as by bandwidth.  This
// kernel does nothing but read: the same bytes, spread evenly over the same
// grid, cluster shape, ring depth and copy size as the streaming SGMV kernel
// gets for the batch, each CTA pulling its share on chip through 1-D bulk
// copies completing on mbarriers.  Its time is the floor the SGMV launch can
// approach on this GPU; the difference is what grouping, the cluster exchange
// of v and the arithmetic add.
//
// One warp issues the copies (one lane), one warp waits for each stage and
// frees it.  Every copy is awaited before the CTA exits; every wait is bounded
// and reports a timeout in the device error word.
#include "sgmv_device.cuh"
#include "sgmv_internal.h"

namespace sgmv {
namespace {

constexpr int kFloorThreads = 64;

__global__ void __launch_bounds__(kFloorThreads)
    read_floor_kernel(const uint8_t *__restrict__ src, uint64_t bytes, uint32_t chunk, int nst,
                      int *err) {
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ __align__(8) uint64_t full[kStreamMaxStages], empty[kStreamMaxStages];
    const uint64_t ctas = (uint64_t)gridDim.x * gridDim.y;
    const uint64_t id = (uint64_t)blockIdx.y * gridDim.x + blockIdx.x;
    // this CTA's share: consecutive bytes, starting on a 16-byte boundary
    const uint64_t per = ((bytes + ctas - 1) / ctas + 15) & ~15ull;
    const uint64_t lo = min(bytes, id * per), hi = min(bytes, lo + per);
    const int n = (int)((hi - lo + chunk - 1) / chunk);
    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init_fence();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        if (lane == 0) {
            for (int q = 0; q < n; ++q) {
                const int s = q % nst;
                if (q >= nst && !mbar_wait(&empty[s], (uint32_t)((q / nst - 1) & 1)))
                    set_error(err, kErrTimeout);
                const uint64_t off = lo + (uint64_t)q * chunk;
                const uint32_t nb = (uint32_t)min((uint64_t)chunk, hi - off);
                mbar_arrive_expect_tx(&full[s], nb);
                bulk_g2s(sm + (size_t)s * chunk, src + off, nb, &full[s]);
            }
        }
    } else {
        for (int q = 0; q < n; ++q) {
            const int s = q % nst;
            const uint32_t parity = (uint32_t)((q / nst) & 1);
            if (!mbar_wait(&full[s], parity)) {
                set_error(err, kErrTimeout);
                mbar_wait(&full[s], parity);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
    // The kernel after this one on the stream may read what precedes it.
    pdl_wait();
}

}  // namespace

int read_floor_launch(const void *src, uint64_t bytes, int cl, int G, int nst, uint32_t chunk,
                      int *err, cudaStream_t stream) {
    if (nst < 1 || nst > kStreamMaxStages || chunk < 16 || chunk % 16 != 0 || bytes % 16 != 0)
        return (int)cudaErrorInvalidValue;
    const size_t smem = (size_t)nst * chunk;
    cudaError_t e = cudaFuncSetAttribute(read_floor_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cl, (unsigned)G, 1);
    cfg.blockDim = dim3(kFloorThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (cl > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)cl;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = (unsigned)na;
    const uint8_t *s8 = static_cast<const uint8_t *>(src);
    return (int)cudaLaunchKernelEx(&cfg, read_floor_kernel, s8, bytes, chunk, nst, err);
}

}  // namespace sgmv
