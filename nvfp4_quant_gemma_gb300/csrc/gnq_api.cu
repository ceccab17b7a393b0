// C ABI of the fused add + Gemma RMSNorm + quant library: argument checks,
// launch-shape policy and dispatch.  The contract of every entry point is in
// include/gemma_nq.h.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "gemma_nq.h"
#include "gnq_launch.cuh"

namespace gnq {
extern template cudaError_t launch_mode<MODE_NONE>(const Params &, int, bool,
                                                   const LaunchShape &, cudaStream_t);
extern template cudaError_t launch_mode<MODE_FP8>(const Params &, int, bool,
                                                  const LaunchShape &, cudaStream_t);
extern template cudaError_t launch_mode<MODE_NVFP4>(const Params &, int, bool,
                                                    const LaunchShape &, cudaStream_t);
extern template cudaError_t launch_mode<MODE_MXFP8>(const Params &, int, bool,
                                                    const LaunchShape &, cudaStream_t);
extern template int stream_blocks_per_sm<MODE_NONE>(int, bool, int, bool, bool, int, size_t);
extern template int stream_blocks_per_sm<MODE_FP8>(int, bool, int, bool, bool, int, size_t);
extern template int stream_blocks_per_sm<MODE_NVFP4>(int, bool, int, bool, bool, int, size_t);
extern template int stream_blocks_per_sm<MODE_MXFP8>(int, bool, int, bool, bool, int, size_t);

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxH = 65536;
constexpr int kMaxParts = 8;

struct DevInfo {
    int sms;
    int smem_optin;     // largest dynamic shared memory a CTA may opt in to
    unsigned int *err;  // device address of the error word
};

// Error word written by kernels whose bounded waits gave up (bit
// DEVERR_WAIT_TIMEOUT); one per device, read and cleared by
// gnq_read_device_error.
__device__ unsigned int g_device_error;

std::atomic<int> g_ready[kMaxDevices];
DevInfo g_info[kMaxDevices];
std::atomic<int> g_force_kernel{0};  // 0 auto, 1 row kernel, 2 streaming kernel
std::atomic<int> g_force_cluster{0};
std::atomic<int> g_force_vpt{0};
std::atomic<int> g_force_form{0};  // 0 auto, 1 fp32 form, 2 packed (lean) form
std::atomic<int> g_pdl{1};  // 1: launch as programmatic dependents, 0: plain launches
std::atomic<int> g_const_w{0};  // 1: small batches read w and scale before the PDL wait
std::atomic<int> g_inject_timeout{0};  // test hook: streaming waits give up (see the header)

constexpr long long kWaitLimit = 1LL << 31;      // cycles: about a second
constexpr long long kTestWaitLimit = 1LL << 20;  // cycles: under a millisecond

// Device properties and the error word's address, queried once per device
// with that device current.
const DevInfo *dev_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (g_ready[dev].load(std::memory_order_acquire) == 0) {
        DevInfo d{};
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                   dev) != cudaSuccess ||
            cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err), g_device_error) !=
                cudaSuccess)
            return nullptr;
        g_info[dev] = d;  // identical values if two threads race here
        g_ready[dev].store(1, std::memory_order_release);
    }
    return &g_info[dev];
}

}  // namespace

cudaError_t opt_in_dynamic_smem(const void *fn) {
    struct Done {
        int dev;
        const void *fn;
    };
    static std::mutex mu;
    static Done done[512];
    static int n_done = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].dev == dev && done[i].fn == fn) return cudaSuccess;
    cudaFuncAttributes a;
    int optin = 0;
    if ((e = cudaFuncGetAttributes(&a, fn)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess)
        return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)a.sharedSizeBytes);
    if (e == cudaSuccess && n_done < 512) done[n_done++] = Done{dev, fn};
    return e;
}

int one_wave_ctas(const void *fn, int threads) {
    struct Entry {
        int dev;
        const void *fn;
        int threads, ctas;
    };
    static std::mutex mu;
    static Entry cache[512];
    static int n_cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < n_cached; ++i)
            if (cache[i].dev == dev && cache[i].fn == fn && cache[i].threads == threads)
                return cache[i].ctas;
    }
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, 0) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const int ctas = per_sm * sms;
    std::lock_guard<std::mutex> lock(mu);
    if (n_cached < 512) cache[n_cached++] = Entry{dev, fn, threads, ctas};
    return ctas;
}

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Elements per NVFP4 scale group (4 blocks), MXFP8 block, or vector chunk: a
// cluster may only split a row at multiples of this.
int granule(int mode) { return mode == MODE_NVFP4 ? 64 : mode == MODE_MXFP8 ? 32 : 8; }

int max_threads(bool stream, int vpt) { return stream ? (vpt == 1 ? 1024 : 512) : 1024 / vpt; }

// Elements one thread handles per unit (a whole NVFP4 block, else a chunk).
int unit_elems(int mode) { return mode == MODE_NVFP4 ? 16 : 8; }

bool row_shape_fits(int64_t H, int mode, int cluster, int vpt) {
    if (cluster < 1 || cluster > 8 || (cluster & (cluster - 1))) return false;
    if (vpt != 1 && vpt != 2 && vpt != 4) return false;
    if (H % ((int64_t)cluster * granule(mode)) != 0) return false;
    const int64_t threads = (H / cluster / unit_elems(mode) + vpt - 1) / vpt;
    return threads <= max_threads(false, vpt);
}

int stream_occupancy_query(int mode, int dtype, bool parts, int vpt, bool lean, bool full,
                           int threads, size_t smem) {
    switch (mode) {
        case MODE_NONE:
            return stream_blocks_per_sm<MODE_NONE>(dtype, parts, vpt, lean, full, threads, smem);
        case MODE_FP8:
            return stream_blocks_per_sm<MODE_FP8>(dtype, parts, vpt, lean, full, threads, smem);
        case MODE_NVFP4:
            return stream_blocks_per_sm<MODE_NVFP4>(dtype, parts, vpt, lean, full, threads, smem);
        default:
            return stream_blocks_per_sm<MODE_MXFP8>(dtype, parts, vpt, lean, full, threads, smem);
    }
}

// Occupancy answers are cached per (device, instance, threads, smem): the
// query is a driver call, and the answer never changes for a device.
int stream_occupancy(int mode, int dtype, bool parts, int vpt, bool lean, bool full, int threads,
                     size_t smem) {
    struct Entry {
        int dev, mode, dtype, parts, vpt, lean, full, threads;
        size_t smem;
        int blocks;
    };
    static std::mutex mu;
    static Entry cache[256];
    static int n_cached = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < n_cached; ++i) {
            const Entry &e = cache[i];
            if (e.dev == dev && e.mode == mode && e.dtype == dtype && e.parts == (int)parts &&
                e.vpt == vpt && e.lean == (int)lean && e.full == (int)full && e.threads == threads &&
                e.smem == smem)
                return e.blocks;
        }
    }
    const int blocks = stream_occupancy_query(mode, dtype, parts, vpt, lean, full, threads, smem);
    std::lock_guard<std::mutex> lock(mu);
    if (n_cached < 256)
        cache[n_cached++] =
            Entry{dev, mode, dtype, (int)parts, vpt, (int)lean, (int)full, threads, smem, blocks};
    return blocks;
}

// True if `ptr` is plain device memory: the only memory the streaming
// kernel's bulk copies are given.  Pinned host memory, managed memory and
// anything the runtime does not know (or fails to classify) give false.
bool in_device_memory(const void *ptr) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();  // clear the error, so it is not reported by the launch
        return false;
    }
    return a.type == cudaMemoryTypeDevice;
}

// Streaming kernel shape.  For each ring depth S (rows in flight per CTA,
// 2..4) the occupancy calculator gives the resident CTAs per SM of this
// instance; the shape with the most resident threads wins (ties: deeper
// ring).  The grid is one wave of resident CTAs.  False if nothing fits.
bool stream_shape(const DevInfo &d, int64_t M, int64_t H, int mode, int dtype, int k, int nops,
                  int vpt, bool lean, LaunchShape &ls) {
    if (vpt != 1 && vpt != 2 && vpt != 4) return false;
    const int64_t threads = (H / unit_elems(mode) + vpt - 1) / vpt;
    if (threads > max_threads(true, vpt)) return false;
    const int64_t thr = (threads + 31) / 32 * 32;
    const bool full = H == (int64_t)vpt * unit_elems(mode) * thr;
    const int64_t stage = (int64_t)nops * 2 * H;
    if (stage >= (1 << 20)) return false;  // mbarrier transaction count limit
    // fp32 bias + w table of the register-light form (see stream_kernel)
    const int64_t wtab = (!lean && vpt >= 2 && mode == MODE_NVFP4) ? 4 * H : 0;
    auto smem_for = [&](int S) { return (stage * S + 8 * S + 15) / 16 * 16 + wtab; };
    int best_blocks = 0, best_S = 0;
    for (int S = 4; S >= 2; --S) {
        const int64_t smem = smem_for(S);
        if (smem > d.smem_optin) continue;
        const int blocks =
            stream_occupancy(mode, dtype, k > 1, vpt, lean, full, (int)thr, (size_t)smem);
        if (blocks > best_blocks) {
            best_blocks = blocks;
            best_S = S;
        }
    }
    if (best_blocks == 0) return false;
    ls.stream = true;
    ls.cluster = 1;
    ls.vpt = vpt;
    ls.threads = (int)thr;
    ls.stages = best_S;
    ls.smem = (size_t)smem_for(best_S);
    const int64_t wave = (int64_t)d.sms * best_blocks;
    ls.grid = M < wave ? M : wave;
    ls.pdl = g_pdl.load() != 0;
    ls.lean = lean;
    ls.full = full;
    return true;
}

// Automatic launch shape, from sweeps of both kernels x units per thread x
// register form x M = 16 .. 16384 on the decode, prefill, no-residual and
// partial-sum workload classes (GB300, 152 SMs):
//   * one activation with a residual: one CTA per row at every M -- one
//     unit per thread below ~SMs rows, else ~256 threads per CTA (NVFP4 at
//     H = 5120: 160; the fp16 16384 x 8192 NVFP4 batch ran 125.1 us at 256
//     threads against 126.1 us at 128 with 256-bit accesses);
//   * no residual: one CTA per row up to 16 x SMs rows, then -- unless y
//     is written (norm only, or write_y), where the row kernel stays ahead --
//     rows stream through persistent CTAs of four units per thread (~256
//     threads for FP8 at H = 8192, ~128 for NVFP4), in the packed form;
//   * k partials: streaming from 4 x SMs rows (~256 threads; FP8 / MXFP8 /
//     no quant ~512 from 16 x SMs rows), one CTA per row below.
// A row is split over a cluster only when it has more than 1024 units: on
// these shapes the cluster barrier always cost more than the extra SMs
// gave back.
// `forced`: apply the shape forced by gnq_set_launch_policy (else the
// automatic choice alone).
LaunchShape choose_shape(const DevInfo &d, int64_t M, int64_t H, int mode, int dtype, int k,
                         bool res, bool write_y, float weight_bias, bool forced = true,
                         bool allow_stream = true) {
    const int fk = forced ? g_force_kernel.load() : 0, fc = forced ? g_force_cluster.load() : 0;
    const int fv = forced ? g_force_vpt.load() : 0, ff = forced ? g_force_form.load() : 0;
    const int nops = k + (res ? 1 : 0);
    LaunchShape ls{false, 1, 1, 32, M, 0, 0, g_pdl.load() != 0, false, false, 0};
    // The packed (lean) form is chosen where four units per thread would
    // otherwise cost occupancy; it needs the Gemma or plain weight bias.
    const bool lean_ok = weight_bias == 1.f || weight_bias == 0.f;
    auto lean_for = [&](int v) { return lean_ok && (ff ? ff == 2 : v == 4); };
    const int64_t units = H / unit_elems(mode);
    auto vpt_for = [&](int64_t target) {
        int v = 1;
        while (v < 4 && (units + v - 1) / v > target) v *= 2;
        return v;
    };
    const int64_t sms = d.sms;
    bool stream = false;
    int vpt = 1;
    if (k > 1) {
        stream = M >= 4 * sms;
        vpt = stream ? vpt_for(M >= 16 * sms && mode != MODE_NVFP4 ? 512 : 256) : 1;
    } else if (res) {
        vpt = M < sms ? 1 : vpt_for(256);
    } else {
        stream = M >= 16 * sms && !write_y;
        vpt = M < sms ? 1 : vpt_for(stream && mode == MODE_NVFP4 ? 128 : 256);
    }
    if (fk) stream = fk == 2;
    if (!allow_stream) stream = false;
    if (fv) vpt = fv;
    if (stream && (stream_shape(d, M, H, mode, dtype, k, nops, vpt, lean_for(vpt), ls) ||
                   stream_shape(d, M, H, mode, dtype, k, nops, vpt_for(256), lean_for(vpt_for(256)),
                                ls))) {
        // a forced streaming launch may ask for at least `fc` rows per CTA
        if (fk == 2 && fc > 1) ls.grid = std::min<int64_t>(ls.grid, (M + fc - 1) / fc);
        return ls;
    }

    ls.vpt = fv ? fv : (stream ? 1 : vpt);
    const int64_t gran2 = 2LL * granule(mode);
    // rows wider than 1024 units: a CTA handles at most 1024 units
    while (ls.cluster < 8 && units / ls.cluster > 1024 && H % (gran2 * ls.cluster) == 0)
        ls.cluster *= 2;
    const int64_t nunits = H / ls.cluster / unit_elems(mode);
    while (ls.vpt < 4 && (nunits + ls.vpt - 1) / ls.vpt > max_threads(false, ls.vpt)) ls.vpt *= 2;
    if (fc || fv) {
        const int c = fc ? fc : ls.cluster, v = fv ? fv : ls.vpt;
        if (row_shape_fits(H, mode, c, v)) {
            ls.cluster = c;
            ls.vpt = v;
        }
    }
    const int64_t threads = (H / ls.cluster / unit_elems(mode) + ls.vpt - 1) / ls.vpt;
    ls.threads = (int)((threads + 31) / 32 * 32);
    ls.full = H / ls.cluster == (int64_t)ls.vpt * unit_elems(mode) * ls.threads;
    ls.grid = M * ls.cluster;
    ls.lean = lean_for(ls.vpt);
    return ls;
}

int run(const void *x, int k, int64_t part_stride, void *residual, const void *w, float eps,
        float weight_bias, const float *scale, int mode, int write_y, void *q, void *block_scale,
        void *y, int64_t M, int64_t H, int dtype, void *stream) {
    if (dtype != GNQ_BF16 && dtype != GNQ_FP16) return GNQ_ERR_DTYPE;
    if (mode < MODE_NONE || mode > MODE_MXFP8) return GNQ_ERR_MODE;
    if (k < 1 || k > kMaxParts) return GNQ_ERR_MODE;
    if (M < 0 || H <= 0 || H > kMaxH || H % 8 != 0) return GNQ_ERR_SHAPE;
    if (mode == MODE_NVFP4 && H % 64 != 0) return GNQ_ERR_SHAPE;
    if (mode == MODE_MXFP8 && H % 32 != 0) return GNQ_ERR_SHAPE;
    if (M > (int64_t)0x7FFFFFFF / 8) return GNQ_ERR_SHAPE;
    if (k > 1 && (part_stride < M * H || part_stride % 8 != 0)) return GNQ_ERR_ALIGN;
    if (mode == MODE_NONE) write_y = 1;
    if (M == 0) return GNQ_OK;  // nothing to do (and empty tensors may be NULL)

    if (!x || !w) return GNQ_ERR_NULL;
    if (write_y && !y) return GNQ_ERR_NULL;
    if (mode != MODE_NONE && !q) return GNQ_ERR_NULL;
    if ((mode == MODE_FP8 || mode == MODE_NVFP4) && !scale) return GNQ_ERR_NULL;
    if ((mode == MODE_NVFP4 || mode == MODE_MXFP8) && !block_scale) return GNQ_ERR_NULL;

    if (residual && residual == x) return GNQ_ERR_ALIAS;
    if (write_y && (y == x || (residual && y == residual))) return GNQ_ERR_ALIAS;

    if (!aligned(x, 16) || !aligned(w, 16) || (residual && !aligned(residual, 16)) ||
        (write_y && !aligned(y, 16)) || (q && mode != MODE_NONE && !aligned(q, 16)) ||
        (scale && !aligned(scale, 4)) || (block_scale && mode != MODE_FP8 && !aligned(block_scale, 4)))
        return GNQ_ERR_ALIGN;

    Params p;
    p.x = static_cast<const uint16_t *>(x);
    p.part_stride = part_stride;
    p.k = k;
    p.residual = static_cast<uint16_t *>(residual);
    p.w = static_cast<const uint16_t *>(w);
    p.eps = eps;
    p.inv_h = 1.0f / (float)H;
    p.weight_bias = weight_bias;
    p.scale = scale;
    p.q = static_cast<uint8_t *>(q);
    p.block_scale = static_cast<uint8_t *>(block_scale);
    p.y = write_y ? static_cast<uint16_t *>(y) : nullptr;
    p.M = M;
    p.H = (int)H;
    p.Kp4 = (int)(((H / 16) + 3) / 4);
    p.write_y = write_y ? 1 : 0;

    const DevInfo *d = dev_info();
    if (!d) return GNQ_ERR_CUDA;
    // NVFP4 instances move a unit's 32-byte block in one 256-bit access when
    // every 16-bit tensor is 32-byte aligned (the streaming ones of k
    // partials always do).
    const bool a32 = mode == MODE_NVFP4 && aligned(x, 32) && aligned(w, 32) &&
                     (!residual || aligned(residual, 32)) && (!write_y || aligned(y, 32)) &&
                     (k == 1 || (part_stride * 2) % 32 == 0);
    LaunchShape ls =
        choose_shape(*d, M, H, mode, dtype, k, residual != nullptr, write_y != 0, weight_bias);
    // The streaming kernel's bulk copies read device memory; activations
    // anywhere else (mapped pinned host memory, read over the host link) run
    // on the row kernel, whose plain loads and stores reach any address the
    // device can access.  So do NVFP4 calls without 32-byte alignment.
    if (ls.stream && ((mode == MODE_NVFP4 && k > 1 && !a32) || !in_device_memory(x) ||
                      (residual && !in_device_memory(residual))))
        ls = choose_shape(*d, M, H, mode, dtype, k, residual != nullptr, write_y != 0, weight_bias,
                          true, false);
    ls.opt = (a32 ? OPT_A32 : 0) |
             (g_const_w.load() && !ls.stream && ls.vpt == 1 && k == 1 ? OPT_EARLYW : 0);
    p.seg = (int)(H / ls.cluster);
    p.stages = ls.stages;
    p.err = d->err;
    const bool inject = g_inject_timeout.load() != 0;
    p.wait_limit = inject ? kTestWaitLimit : kWaitLimit;
    p.tx_extra = inject ? 16u : 0u;
    p.pf_ctas = 0;  // set per launch

    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool parts = k > 1;
    cudaError_t e;
    switch (mode) {
        case MODE_NONE: e = launch_mode<MODE_NONE>(p, dtype, parts, ls, s); break;
        case MODE_FP8: e = launch_mode<MODE_FP8>(p, dtype, parts, ls, s); break;
        case MODE_NVFP4: e = launch_mode<MODE_NVFP4>(p, dtype, parts, ls, s); break;
        default: e = launch_mode<MODE_MXFP8>(p, dtype, parts, ls, s); break;
    }
    if (e == cudaSuccess) return GNQ_OK;
    cudaGetLastError();  // reported here; do not leave it for the caller's next check
    return GNQ_ERR_CUDA;
}

// Groups of 8 values through the kernels' FP8 encoder: the paired path
// with the magnitude clamp the kernels apply to bf16 y (a no-op for
// bf16/fp16 values that cannot overflow), or IEEE division for extreme
// scales.  The ragged tail is padded to a group.
__global__ void fp8_values_kernel(const float *y, int64_t n, const float *scale, uint8_t *q) {
    const Fp8Div fd = make_fp8_div(*scale);
    const int64_t groups = (n + 7) / 8;
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < groups;
         g += (int64_t)gridDim.x * blockDim.x) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t j = 8 * g + i;
            v[i] = j < n ? y[j] : 0.f;
            if (fd.fast) v[i] = copysignf(min_nan(fabsf(v[i]), fd.ylim), v[i]);
        }
        uint32_t lo, hi;
        if (fd.fast) fp8_codes8<FP8_PAIR>(v, fd, lo, hi);
        else fp8_codes8<FP8_IEEE>(v, fd, lo, hi);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t j = 8 * g + i;
            if (j < n) q[j] = (uint8_t)((i < 4 ? lo : hi) >> (8 * (i & 3)));
        }
    }
}

__global__ void encode_kernel(const float *v, int64_t n, uint8_t *e4m3, uint8_t *e2m1) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float x = v[i];
        if (e4m3) e4m3[i] = (uint8_t)(e4m3x2(x, 0.f) & 0xFF);
        if (e2m1) e2m1[i] = (uint8_t)(e2m1x4(x, 0.f, 0.f, 0.f) & 0xF);
    }
}

// Stand-in for the first kernel of the next linear layer: each CTA reads
// its share of an independent buffer (the layer's weight) before it waits on
// the preceding grid, then its share of that grid's codes, and stores one
// checksum word per thread.  Launched as a programmatic dependent.
__global__ void consumer_kernel(const uint4 *q, int64_t nq, const uint4 *wt, int64_t nw,
                                uint32_t *out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (int64_t i = i0; i < nw; i += stride) {
        const uint4 v = ld_stream(wt + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    pdl_wait();
    for (int64_t i = i0; i < nq; i += stride) {
        const uint4 v = ld_stream(q + i);
        acc += v.x ^ v.y ^ v.z ^ v.w;
    }
    out[i0] = acc;
}

}  // namespace
}  // namespace gnq

extern "C" {

int gemma_add_rms_norm(const void *x, void *residual, const void *w, float eps, void *y,
                       int64_t M, int64_t H, int dtype, void *stream) {
    return gnq::run(x, 1, 0, residual, w, eps, 1.0f, nullptr, gnq::MODE_NONE, 1, nullptr,
                    nullptr, y, M, H, dtype, stream);
}

int gemma_add_rms_norm_quant(const void *x, void *residual, const void *w, float eps,
                             const float *scale, int mode, int write_y, void *q,
                             void *block_scale, void *y, int64_t M, int64_t H, int dtype,
                             void *stream) {
    if (mode < GNQ_FP8 || mode > GNQ_MXFP8) return GNQ_ERR_MODE;
    return gnq::run(x, 1, 0, residual, w, eps, 1.0f, scale, mode, write_y, q, block_scale, y,
                    M, H, dtype, stream);
}

int gemma_add_rms_norm_quant_parts(const void *x_parts, int k, int64_t part_stride,
                                   void *residual, const void *w, float eps,
                                   const float *scale, int mode, int write_y, void *q,
                                   void *block_scale, void *y, int64_t M, int64_t H, int dtype,
                                   void *stream) {
    return gnq::run(x_parts, k, part_stride, residual, w, eps, 1.0f, scale, mode, write_y, q,
                    block_scale, y, M, H, dtype, stream);
}

int add_rms_norm_quant(const void *x_parts, int k, int64_t part_stride, void *residual,
                       const void *w, float eps, const float *scale, int mode, int write_y,
                       void *q, void *block_scale, void *y, int64_t M, int64_t H, int dtype,
                       void *stream) {
    return gnq::run(x_parts, k, part_stride, residual, w, eps, 0.0f, scale, mode, write_y, q,
                    block_scale, y, M, H, dtype, stream);
}

const char *gnq_status_string(int status) {
    switch (status) {
        case GNQ_OK: return "ok";
        case GNQ_ERR_NULL: return "a required pointer is NULL";
        case GNQ_ERR_SHAPE: return "unsupported shape (M < 0, or H out of range / not a supported multiple)";
        case GNQ_ERR_DTYPE: return "dtype must be GNQ_BF16 or GNQ_FP16";
        case GNQ_ERR_MODE: return "unknown quantization mode or partial count";
        case GNQ_ERR_ALIAS: return "x, residual and y must be distinct buffers";
        case GNQ_ERR_ALIGN: return "misaligned pointer or partial stride";
        case GNQ_ERR_CUDA: return "CUDA launch error";
        default: return "unknown status";
    }
}

int gnq_set_launch_policy(int kernel, int cluster, int vpt, int form) {
    if (kernel < 0 || kernel > 2) return GNQ_ERR_SHAPE;
    if (cluster < 0 || cluster > 8 || (cluster & (cluster - 1))) return GNQ_ERR_SHAPE;
    if (vpt != 0 && vpt != 1 && vpt != 2 && vpt != 4) return GNQ_ERR_SHAPE;
    if (form < 0 || form > 2) return GNQ_ERR_SHAPE;
    gnq::g_force_kernel.store(kernel);
    gnq::g_force_cluster.store(cluster);
    gnq::g_force_vpt.store(vpt);
    gnq::g_force_form.store(form);
    return GNQ_OK;
}

int gnq_query_launch(int64_t M, int64_t H, int k, int has_residual, int write_y, int mode,
                     int dtype, float weight_bias, int *kernel, int *cluster, int *vpt,
                     int *form) {
    if (!kernel || !cluster || !vpt || !form) return GNQ_ERR_NULL;
    if (dtype != GNQ_BF16 && dtype != GNQ_FP16) return GNQ_ERR_DTYPE;
    if (mode < gnq::MODE_NONE || mode > gnq::MODE_MXFP8) return GNQ_ERR_MODE;
    if (k < 1 || k > gnq::kMaxParts) return GNQ_ERR_MODE;
    if (M < 1 || H <= 0 || H > gnq::kMaxH || H % 8 != 0) return GNQ_ERR_SHAPE;
    if (mode == gnq::MODE_NVFP4 && H % 64 != 0) return GNQ_ERR_SHAPE;
    if (mode == gnq::MODE_MXFP8 && H % 32 != 0) return GNQ_ERR_SHAPE;
    if (M > (int64_t)0x7FFFFFFF / 8) return GNQ_ERR_SHAPE;
    const gnq::DevInfo *d = gnq::dev_info();
    if (!d) return GNQ_ERR_CUDA;
    const gnq::LaunchShape ls =
        gnq::choose_shape(*d, M, H, mode, dtype, k, has_residual != 0,
                          write_y != 0 || mode == gnq::MODE_NONE, weight_bias, false);
    *kernel = ls.stream ? 2 : 1;
    *cluster = ls.stream ? 0 : ls.cluster;
    *vpt = ls.vpt;
    *form = ls.lean ? 2 : 1;
    return GNQ_OK;
}

int gnq_set_pdl(int enable) {
    if (enable != 0 && enable != 1) return GNQ_ERR_SHAPE;
    gnq::g_pdl.store(enable);
    return GNQ_OK;
}

int gnq_set_constant_weights(int enable) {
    if (enable != 0 && enable != 1) return GNQ_ERR_SHAPE;
    gnq::g_const_w.store(enable);
    return GNQ_OK;
}

int gnq_inject_wait_timeout(int enable) {
    if (enable != 0 && enable != 1) return GNQ_ERR_SHAPE;
    gnq::g_inject_timeout.store(enable);
    return GNQ_OK;
}

int gnq_read_device_error(unsigned int *flags, int clear) {
    if (!flags) return GNQ_ERR_NULL;
    const gnq::DevInfo *d = gnq::dev_info();
    if (!d) return GNQ_ERR_CUDA;
    if (cudaMemcpy(flags, d->err, sizeof(unsigned int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GNQ_ERR_CUDA;
    if (clear && cudaMemset(d->err, 0, sizeof(unsigned int)) != cudaSuccess) return GNQ_ERR_CUDA;
    return GNQ_OK;
}

int gnq_encode_e4m3_e2m1(const float *v, int64_t n, uint8_t *e4m3, uint8_t *e2m1,
                         void *stream) {
    if (n < 0) return GNQ_ERR_SHAPE;
    if (n == 0) return GNQ_OK;
    if (!v) return GNQ_ERR_NULL;
    const int64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    gnq::encode_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        v, n, e4m3, e2m1);
    return cudaGetLastError() == cudaSuccess ? GNQ_OK : GNQ_ERR_CUDA;
}

int gnq_pdl_consumer(const void *q, int64_t q_bytes, const void *wt, int64_t wt_bytes,
                     unsigned int *out, int ctas, void *stream) {
    if (q_bytes < 0 || wt_bytes < 0 || q_bytes % 16 || wt_bytes % 16 || ctas < 1 || ctas > 65535)
        return GNQ_ERR_SHAPE;
    if (!out || (q_bytes && !q) || (wt_bytes && !wt)) return GNQ_ERR_NULL;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
    cfg.attrs = &attr;
    if (cudaLaunchKernelEx(&cfg, gnq::consumer_kernel, static_cast<const uint4 *>(q),
                           q_bytes / 16, static_cast<const uint4 *>(wt), wt_bytes / 16,
                           static_cast<uint32_t *>(out)) == cudaSuccess)
        return GNQ_OK;
    cudaGetLastError();
    return GNQ_ERR_CUDA;
}

int gnq_quantize_fp8_values(const float *y, int64_t n, const float *scale, uint8_t *q,
                            void *stream) {
    if (n < 0) return GNQ_ERR_SHAPE;
    if (n == 0) return GNQ_OK;
    if (!y || !scale || !q) return GNQ_ERR_NULL;
    const int64_t groups = (n + 7) / 8;
    const int64_t blocks = (groups + 255) / 256 < 4096 ? (groups + 255) / 256 : 4096;
    gnq::fp8_values_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        y, n, scale, q);
    return cudaGetLastError() == cudaSuccess ? GNQ_OK : GNQ_ERR_CUDA;
}

}  // extern "C"
