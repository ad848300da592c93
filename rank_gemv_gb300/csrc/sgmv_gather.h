// sgmv_gather.h -- the gather-copy kernel's launcher (sgmv_gather.cu), used by
// sgmv_copy_gather in sgmv_api.cu.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace sgmv {

// Most copies of one sgmv_copy_gather call (they travel in the kernel's
// parameters: 32 bytes each).
constexpr int kGatherMaxCopies = 512;

// One launch of the gather kernel: every source and destination readable or
// writable by the current device, every pointer 16-byte aligned, every size a
// multiple of 16; at most max_ctas CTAs.  Returns a cudaError_t value.
int gather_launch(int32_t n, void *const *dst, const void *const *src, const uint64_t *bytes,
                  int max_ctas, cudaStream_t stream);

}  // namespace sgmv
