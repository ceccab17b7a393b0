// Instances of the row kernel for quantization mode NVFP4.
#include "gnq_launch.cuh"

namespace gnq {
template cudaError_t launch_mode<MODE_NVFP4>(const Params &, int, bool, const LaunchShape &,
                                            cudaStream_t);
}  // namespace gnq
