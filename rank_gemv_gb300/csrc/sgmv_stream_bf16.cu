// Streaming CUDA-core SGMV kernel, bf16 inputs (all output types, rank bounds 16 / 32 / 64).
#include "sgmv_stream.cuh"

namespace sgmv {
int stream_launch_bf16(const StreamLaunch &l) { return stream_launch_impl<__nv_bfloat16>(l); }
}  // namespace sgmv
