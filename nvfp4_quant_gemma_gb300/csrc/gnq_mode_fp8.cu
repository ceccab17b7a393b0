// Instances of the kernels for quantization mode FP8.
#include "gnq_launch.cuh"

namespace gnq {
template cudaError_t launch_mode<MODE_FP8>(const Params &, int, bool, const LaunchShape &,
                                           cudaStream_t);
template int stream_blocks_per_sm<MODE_FP8>(int, bool, int, bool, bool, int, size_t);
}  // namespace gnq
