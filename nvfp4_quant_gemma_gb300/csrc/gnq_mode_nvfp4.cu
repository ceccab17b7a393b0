// Instances of the kernels for quantization mode NVFP4.
#include "gnq_launch.cuh"

namespace gnq {
template cudaError_t launch_mode<MODE_NVFP4>(const Params &, int, bool, const LaunchShape &,
                                           cudaStream_t);
template int stream_blocks_per_sm<MODE_NVFP4>(int, bool, int, bool, bool, int, size_t);
}  // namespace gnq
