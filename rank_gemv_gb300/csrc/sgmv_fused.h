// sgmv_fused.h -- host-side interface of the fused base linear + LoRA
// kernels (sgmv_fused.cu), kept apart from the other kernels' parameters.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sgmv {

// One launch of the fused base linear + LoRA kernel (sgmv_fused.cu), after
// the shrink has written v [T][r] fp32 by sorted position.
struct FusedArgs {
    void *y;
    const void *x;
    const void *W;
    const void *B;
    const float *v;      // the shrink's output [T][r] fp32, or nullptr (no segments)
    void *prep;          // workspace for the pair table and v tiles (fused_prep_bytes), or nullptr
    float *part;         // workspace for the split partials (fused_part_bytes)
    const int32_t *perm;
    const int32_t *seg_ptr;
    const int32_t *idx;
    int *err;
    int32_t S, T, L, H1, H2, r;
    float scale;
    int in_dtype, y_dtype;
    int32_t nsm;
    bool x_early;        // a kernel that waits for x's producer was launched just before
    cudaStream_t stream;
};

// Bytes of the fused layer's pair table and v tiles (a bound over any
// segmentation of T rows).
size_t fused_prep_bytes(int32_t T, int32_t r);
// Bytes of the fused layer's fp32 scratch for the partial sums of split tiles.
size_t fused_part_bytes(int32_t T, int32_t H2);

// Rows the fused kernel takes (the N of its base MMAs) and the largest rank.
constexpr int kFusedMaxT = 128;
constexpr int kFusedMaxR = 64;

// Launch the fused kernel; returns a cudaError_t value.
int fused_launch(const FusedArgs &g);

}  // namespace sgmv
