// CUDA-core SGMV kernels, bf16 inputs (all output types and rank bounds).
#include "sgmv_cc.cuh"

namespace sgmv {
int cc_launch_bf16(const CCLaunch &l) { return cc_launch_impl<__nv_bfloat16>(l); }
}  // namespace sgmv
