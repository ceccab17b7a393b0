// Instances of the row kernel for quantization mode MXFP8.
#include "gnq_launch.cuh"

namespace gnq {
template cudaError_t launch_mode<MODE_MXFP8>(const Params &, int, bool, const LaunchShape &,
                                            cudaStream_t);
}  // namespace gnq
