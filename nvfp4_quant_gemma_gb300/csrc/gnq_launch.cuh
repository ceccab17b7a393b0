// Launch of the row kernel for one quantization mode: picks the template
// instance (activation type, partials or not, chunks per thread) and applies
// the cluster size as a launch attribute.  One translation unit per mode
// instantiates it, so the library builds in parallel.
#pragma once

#include "gnq_kernels.cuh"

namespace gnq {

struct LaunchShape {
    int cluster;  // CTAs per row (1, 2, 4, 8)
    int vpt;      // 16-byte chunks per thread (1, 2, 4)
    int threads;  // threads per CTA, a multiple of 32
};

template <int MODE>
cudaError_t launch_mode(const Params &p, int dtype, bool parts, const LaunchShape &ls,
                        cudaStream_t stream);

#define GNQ_PICK(T, VPT)                                                          \
    (parts ? (void (*)(const Params))row_kernel<T, MODE, true, VPT>               \
           : (void (*)(const Params))row_kernel<T, MODE, false, VPT>)

template <int MODE>
cudaError_t launch_mode(const Params &p, int dtype, bool parts, const LaunchShape &ls,
                        cudaStream_t stream) {
    void (*fn)(const Params) = nullptr;
    if (dtype == 0) {
        fn = ls.vpt == 1 ? GNQ_PICK(__nv_bfloat16, 1)
           : ls.vpt == 2 ? GNQ_PICK(__nv_bfloat16, 2)
                         : GNQ_PICK(__nv_bfloat16, 4);
    } else {
        fn = ls.vpt == 1 ? GNQ_PICK(__half, 1)
           : ls.vpt == 2 ? GNQ_PICK(__half, 2)
                         : GNQ_PICK(__half, 4);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.M * ls.cluster), 1, 1);
    cfg.blockDim = dim3((unsigned)ls.threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = 0;
    if (ls.cluster > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)ls.cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.numAttrs = 1;
    }
    cfg.attrs = attr;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

#undef GNQ_PICK

}  // namespace gnq
