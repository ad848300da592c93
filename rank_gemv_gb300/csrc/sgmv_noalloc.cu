// sgmv_noalloc.cu -- sgmv_apply for callers that cannot allocate device memory.
//
// sgmv_apply needs a scratch workspace for its tensor-core path (v of the long
// segments, kept between the shrink and the expand kernels), and the caller
// normally allocates it.  Some callers cannot: an inference engine that hands
// a plugin only the buffers it planned at start-up, a real-time serving loop
// that forbids allocation after warm-up, or code that runs while a CUDA graph
// is being captured, where cudaMalloc is not allowed.  sgmv_apply_noalloc
// serves them with a fixed scratch array that lives in this library's device
// image instead.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes
// (4 MiB): every GPU that loads the library holds it until the process exits.
// In host code its name is only a host-side stand-in, not a device address,
// so the device address is looked up once per device, with that device
// current, through cudaGetSymbolAddress, and passed to the kernels.  Problems
// that cannot reach the tensor-core path need no scratch and are passed on
// without it, whatever their size.
#include <climits>
#include <cstdio>
#include <mutex>

#include "sgmv.h"
#include "sgmv_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device (looked up on the
// first call per device), or nullptr with the failing CUDA call recorded for
// sgmv_last_error_string.
void *scratch_address() {
    static std::mutex mu;
    static void *cache[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        sgmv::note_cuda_error("cudaGetDevice", e);
        return nullptr;
    }
    if (dev < 0 || dev >= 256) {
        sgmv::note_cuda_error("device ordinal above 255", cudaErrorInvalidDevice);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            sgmv::note_cuda_error("cudaGetSymbolAddress(noalloc scratch)",
                                  e != cudaSuccess ? e : cudaErrorInvalidSymbol);
            return nullptr;
        }
        cache[dev] = p;
    }
    return cache[dev];
}

}  // namespace

extern "C" int sgmv_apply_noalloc(void *y, int y_dtype, const void *x, const void *A,
                                  const void *B, int in_dtype, float scale, const int32_t *perm,
                                  const int32_t *seg_ptr, const int32_t *idx, int32_t S,
                                  const int32_t *seg_ptr_host, int32_t T, int32_t L, int32_t H1,
                                  int32_t H2, int32_t r, void *stream) {
    // sgmv_apply sends segments to the tensor cores only for r = 64 or 128 and
    // batches of at least kTcMinLen rows; every other problem runs on the
    // CUDA cores without scratch, whatever its size.
    const bool tc_possible = (r == 64 || r == 128) && T >= sgmv::kTcMinLen;
    if (!tc_possible)
        return sgmv_apply(y, y_dtype, x, A, B, in_dtype, scale, perm, seg_ptr, idx, S,
                          seg_ptr_host, T, L, H1, H2, r, nullptr, 0, stream);
    // A problem whose v does not fit the fixed array is refused before
    // anything touches the GPU.
    const size_t need = sgmv_workspace_bytes(T, H1, H2, r);
    if (need > kNoAllocScratchBytes) return SGMV_ERR_WORKSPACE;
    void *scratch = scratch_address();
    if (!scratch) return SGMV_ERR_CUDA;
    return sgmv_apply(y, y_dtype, x, A, B, in_dtype, scale, perm, seg_ptr, idx, S, seg_ptr_host,
                      T, L, H1, H2, r, scratch, need, stream);
}
