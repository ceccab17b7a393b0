// Instances of the kernels for quantization mode MXFP8.
#include "gnq_launch.cuh"

namespace gnq {
template cudaError_t launch_mode<MODE_MXFP8>(const Params &, int, bool, const LaunchShape &,
                                           cudaStream_t);
template int stream_blocks_per_sm<MODE_MXFP8>(int, bool, int, bool, bool, int, size_t);
}  // namespace gnq
