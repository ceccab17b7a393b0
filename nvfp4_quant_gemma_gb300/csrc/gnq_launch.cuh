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
    int opt;         // OPT_* options of the instance
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

// CTAs of this instance that one wave holds on the current device (resident
// CTAs per SM x SMs; 0 on error), cached per device, instance and block size.
// (Defined in gnq_api.cu.)
int one_wave_ctas(const void *fn, int threads);

// Resident CTAs per SM of the streaming kernel instance for this shape (0 on
// error); opts the instance in to its largest dynamic shared memory.
template <int MODE>
int stream_blocks_per_sm(int dtype, bool parts, int vpt, bool lean, bool full, int threads,
                         size_t smem);

using KernelFn = void (*)(const Params);

// The kernel instance of one launch.  Which instances exist:
//   * `full` (every unit of a CTA's segment in range): FP8 streaming, and
//     NVFP4 streaming of one activation, run instances without per-unit
//     checks (2.7 % and 3.0 % faster on the fp16 16384 x 8192 no-residual
//     batches; the same for the FP8 row kernel measured 4 % slower on the
//     decode batch, for NVFP4 partials 0.6 % slower);
//   * OPT_A32: NVFP4 instances that move a unit's 32-byte block in one
//     256-bit access: row instances (which also exist without it, for
//     tensors that are only 16-byte aligned), and the streaming instances
//     of k partials, which store a residual and y (the host keeps such calls
//     without 32-byte alignment on the row kernel).  The streaming
//     instances of one activation -- under the automatic policy, batches
//     that store neither -- keep the plain stores: the option changed their
//     code and cost 2 % on the fp16 16384 x 8192 no-residual batch;
//   * OPT_EARLYW: row instances of one unit per thread for one activation
//     (the small batches, where reading the constants before the wait
//     shortens the call).
template <typename T, int MODE, bool PARTS, int VPT, bool LEAN>
KernelFn pick_instance(bool stream, bool full, int opt) {
    if constexpr (MODE == MODE_NVFP4) {
        if (stream) {
            if constexpr (!PARTS) {
                if (full) return stream_kernel_nvfp4<T, MODE, PARTS, VPT, LEAN, true, 0>;
                return stream_kernel_nvfp4<T, MODE, PARTS, VPT, LEAN, false, 0>;
            } else {
                return stream_kernel_nvfp4<T, MODE, PARTS, VPT, LEAN, false, OPT_A32>;
            }
        }
        if (opt & OPT_A32) {
            if constexpr (VPT == 1 && !PARTS) {
                if (opt & OPT_EARLYW)
                    return row_kernel_nvfp4<T, MODE, PARTS, VPT, LEAN, false, OPT_A32 | OPT_EARLYW>;
            }
            return row_kernel_nvfp4<T, MODE, PARTS, VPT, LEAN, false, OPT_A32>;
        }
        return row_kernel_nvfp4<T, MODE, PARTS, VPT, LEAN, false, 0>;
    } else {
        if (stream) {
            if constexpr (MODE == MODE_FP8) {
                if (full) return stream_kernel<T, MODE, PARTS, VPT, LEAN, true, 0>;
            }
            return stream_kernel<T, MODE, PARTS, VPT, LEAN, false, 0>;
        }
        if constexpr (VPT == 1 && !PARTS) {
            if (opt & OPT_EARLYW) return row_kernel<T, MODE, PARTS, VPT, LEAN, false, OPT_EARLYW>;
        }
        return row_kernel<T, MODE, PARTS, VPT, LEAN, false, 0>;
    }
}

template <int MODE, typename T>
KernelFn pick_typed(bool parts, int vpt, bool lean, bool stream, bool full, int opt) {
#define GNQ_PICK(P, V, L) \
    if (parts == P && vpt == V && lean == L) return pick_instance<T, MODE, P, V, L>(stream, full, opt);
    GNQ_PICK(false, 1, false) GNQ_PICK(false, 1, true) GNQ_PICK(false, 2, false)
    GNQ_PICK(false, 2, true) GNQ_PICK(false, 4, false) GNQ_PICK(false, 4, true)
    GNQ_PICK(true, 1, false) GNQ_PICK(true, 1, true) GNQ_PICK(true, 2, false)
    GNQ_PICK(true, 2, true) GNQ_PICK(true, 4, false) GNQ_PICK(true, 4, true)
#undef GNQ_PICK
    return nullptr;
}

template <int MODE>
KernelFn pick_kernel(int dtype, bool parts, int vpt, bool lean, bool stream, bool full, int opt) {
    return dtype == 0 ? pick_typed<MODE, __nv_bfloat16>(parts, vpt, lean, stream, full, opt)
                      : pick_typed<MODE, __half>(parts, vpt, lean, stream, full, opt);
}

template <int MODE>
int stream_blocks_per_sm(int dtype, bool parts, int vpt, bool lean, bool full, int threads,
                         size_t smem) {
    KernelFn fn = pick_kernel<MODE>(dtype, parts, vpt, lean, true, full, 0);
    if (!fn || opt_in_dynamic_smem(reinterpret_cast<const void *>(fn)) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess)
        return 0;
    return n;
}

template <int MODE>
cudaError_t launch_mode(const Params &p, int dtype, bool parts, const LaunchShape &ls,
                        cudaStream_t stream) {
    KernelFn fn = pick_kernel<MODE>(dtype, parts, ls.vpt, ls.lean, ls.stream, ls.full, ls.opt);
    if (!fn) return cudaErrorInvalidConfiguration;
    if (ls.stream) {
        const cudaError_t e = opt_in_dynamic_smem(reinterpret_cast<const void *>(fn));
        if (e != cudaSuccess) return e;
    }
    Params q = p;
    q.pf_ctas = ls.stream ? 0 : one_wave_ctas(reinterpret_cast<const void *>(fn), ls.threads);
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
    return cudaLaunchKernelEx(&cfg, fn, q);
}

}  // namespace gnq
