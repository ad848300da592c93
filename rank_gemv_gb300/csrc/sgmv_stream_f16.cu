// Streaming CUDA-core SGMV kernel, f16 inputs (all output types, rank bounds 16 / 32 / 64).
#include "sgmv_stream.cuh"

namespace sgmv {
int stream_launch_f16(const StreamLaunch &l) { return stream_launch_impl<__half>(l); }
}  // namespace sgmv
