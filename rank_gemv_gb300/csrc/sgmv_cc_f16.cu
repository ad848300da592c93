// CUDA-core SGMV kernels, f16 inputs (all output types and rank bounds).
#include "sgmv_cc.cuh"

namespace sgmv {
int cc_launch_f16(const CCLaunch &l) { return cc_launch_impl<__half>(l); }
}  // namespace sgmv
