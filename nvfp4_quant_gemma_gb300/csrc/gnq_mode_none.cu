// Instances of the row kernel for quantization mode NONE.
#include "gnq_launch.cuh"

namespace gnq {
template cudaError_t launch_mode<MODE_NONE>(const Params &, int, bool, const LaunchShape &,
                                            cudaStream_t);
}  // namespace gnq
