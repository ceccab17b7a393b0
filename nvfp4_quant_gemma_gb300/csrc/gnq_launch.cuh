// Launch of the kernels for one quantization mode: picks the template
// instance (kernel kind, activation type, partials or not, chunks per thread)
// and applies the cluster size or the dynamic shared memory size.  One
// translation unit per mode instantiates it, so the library builds in
// parallel.
#pragma once

#include "gnq_kernels.cuh"

namespace gnq {

struct LaunchShape {
    bool stream;     // persistent streaming kernel (else one CTA/cluster per row)
    int cluster;     // row kernel: CTAs per row (1, 2, 4, 8)
    int vpt;         // 16-byte chunks per thread (1, 2, 4)
    int threads;     // threads per CTA, a multiple of 32
    int64_t grid;    // CTAs
    int stages;      // streaming kernel: rows in flight per CTA
    size_t smem;     // streaming kernel: dynamic shared memory bytes
    bool pdl;        // launch as a programmatic dependent of the preceding grid
    bool lean;       // packed h / w form (fewest registers) instead of fp32 (fewest instructions)
    bool full;       // every unit of a CTA's segment in range (VPT x threads units)
};

template <int MODE>
cudaError_t launch_mode(const Params &p, int dtype, bool parts, const LaunchShape &ls,
                        cudaStream_t stream);

// Opts a kernel instance in to the largest dynamic shared memory one of its
// CTAs may have on the current device (the device's opt-in limit less the
// instance's static shared memory), once per device and instance.  The value
// never changes, so calls from several host threads agree; each launch states
// its own size in cudaLaunchConfig_t::dynamicSmemBytes.  (Defined in
// gnq_api.cu.)
cudaError_t opt_in_dynamic_smem(const void *fn);

// Resident CTAs per SM of the streaming kernel instance for this shape (0 on
// error); opts the instance in to `smem` bytes of dynamic shared memory.
template <int MODE>
int stream_blocks_per_sm(int dtype, bool parts, int vpt, bool lean, bool full, int threads,
                         size_t smem);

#define GNQ_PICK_L(K, T, VPT, L, F)                                                   \
    (parts ? (void (*)(const Params))K<T, MODE, true, VPT, L, F>                        \
           : (void (*)(const Params))K<T, MODE, false, VPT, L, F>)
#define GNQ_PICK(K, T, VPT, F) (lean ? GNQ_PICK_L(K, T, VPT, true, F) : GNQ_PICK_L(K, T, VPT, false, F))

#define GNQ_PICK_VPT(K, T, F)                                                         \
    (vpt == 1 ? GNQ_PICK(K, T, 1, F) : vpt == 2 ? GNQ_PICK(K, T, 2, F) : GNQ_PICK(K, T, 4, F))
#define GNQ_PICK_T(K, F) (dtype == 0 ? GNQ_PICK_VPT(K, __nv_bfloat16, F) : GNQ_PICK_VPT(K, __half, F))

// The kernel instance of a launch shape.  `full`: every unit of a CTA's
// segment is in range; FP8 streaming, and NVFP4 streaming of one
// activation, then run instances without per-unit checks (2.7 % and 3.0 %
// faster on the fp16 16384 x 8192 no-residual batches; the same for the FP8
// row kernel measured 4 % slower on the decode batch, for NVFP4 partials
// 0.6 % slower).
template <int MODE>
void (*pick_kernel(int dtype, bool parts, int vpt, bool lean, bool stream, bool full))(const Params) {
    if constexpr (MODE == MODE_NVFP4) {
        // one activation only: with k partials the check-free instance was slower
        if (stream)
            return full && !parts ? GNQ_PICK_T(stream_kernel_nvfp4, true)
                                  : GNQ_PICK_T(stream_kernel_nvfp4, false);
        return GNQ_PICK_T(row_kernel_nvfp4, false);
    } else if constexpr (MODE == MODE_FP8) {
        if (stream) return full ? GNQ_PICK_T(stream_kernel, true) : GNQ_PICK_T(stream_kernel, false);
        return GNQ_PICK_T(row_kernel, false);
    } else {
        return stream ? GNQ_PICK_T(stream_kernel, false) : GNQ_PICK_T(row_kernel, false);
    }
}

template <int MODE>
int stream_blocks_per_sm(int dtype, bool parts, int vpt, bool lean, bool full, int threads,
                         size_t smem) {
    void (*fn)(const Params) = pick_kernel<MODE>(dtype, parts, vpt, lean, true, full);
    if (opt_in_dynamic_smem(reinterpret_cast<const void *>(fn)) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess)
        return 0;
    return n;
}

template <int MODE>
cudaError_t launch_mode(const Params &p, int dtype, bool parts, const LaunchShape &ls,
                        cudaStream_t stream) {
    void (*fn)(const Params) = pick_kernel<MODE>(dtype, parts, ls.vpt, ls.lean, ls.stream, ls.full);
    if (ls.stream) {
        const cudaError_t e = opt_in_dynamic_smem(reinterpret_cast<const void *>(fn));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ls.grid, 1, 1);
    cfg.blockDim = dim3((unsigned)ls.threads, 1, 1);
    cfg.dynamicSmemBytes = ls.stream ? ls.smem : 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (!ls.stream && ls.cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)ls.cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (ls.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.numAttrs = n;
    cfg.attrs = attr;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

#undef GNQ_PICK_T
#undef GNQ_PICK_VPT
#undef GNQ_PICK
#undef GNQ_PICK_L

}  // namespace gnq
