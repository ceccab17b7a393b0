// C ABI of the fused add + Gemma RMSNorm + quant library: argument checks,
// launch-shape policy and dispatch.  The contract of every entry point is in
// include/gemma_nq.h.
#include <atomic>

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

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxH = 65536;
constexpr int kMaxParts = 8;

std::atomic<int> g_sm_count[kMaxDevices];  // 0 = not yet queried
std::atomic<int> g_force_cluster{0};
std::atomic<int> g_force_vpt{0};

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Elements per NVFP4 scale group (4 blocks), MXFP8 block, or vector chunk: a
// cluster may only split a row at multiples of this.
int granule(int mode) { return mode == MODE_NVFP4 ? 64 : mode == MODE_MXFP8 ? 32 : 8; }

bool shape_fits(int64_t H, int mode, int cluster, int vpt) {
    if (cluster < 1 || cluster > 8 || (cluster & (cluster - 1))) return false;
    if (vpt != 1 && vpt != 2 && vpt != 4) return false;
    if (H % ((int64_t)cluster * granule(mode)) != 0) return false;
    const int64_t nch = H / cluster / 8;
    const int64_t threads = (nch + vpt - 1) / vpt;
    return threads <= 1024 / vpt;
}

// Launch shape: rows are split over a cluster while the grid would otherwise
// give fewer than ~4 CTAs per SM (small decode batches), then each CTA gets
// enough chunks per thread to stay within 512 threads.
LaunchShape choose_shape(int64_t M, int64_t H, int mode) {
    const int sms = sm_count();
    LaunchShape ls{1, 1, 32};
    while (ls.cluster < 8 && M * ls.cluster < 4LL * sms &&
           H % (2LL * ls.cluster * granule(mode)) == 0 && H / (2 * ls.cluster) >= 256)
        ls.cluster *= 2;
    const int64_t nch = H / ls.cluster / 8;
    while (ls.vpt < 4 && (nch + ls.vpt - 1) / ls.vpt > 512) ls.vpt *= 2;
    const int fc = g_force_cluster.load(), fv = g_force_vpt.load();
    if (fc || fv) {
        const int c = fc ? fc : ls.cluster, v = fv ? fv : ls.vpt;
        if (shape_fits(H, mode, c, v)) {
            ls.cluster = c;
            ls.vpt = v;
        }
    }
    const int64_t n = H / ls.cluster / 8;
    const int64_t threads = (n + ls.vpt - 1) / ls.vpt;
    ls.threads = (int)((threads + 31) / 32 * 32);
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
    p.weight_bias = weight_bias;
    p.scale = scale;
    p.q = static_cast<uint8_t *>(q);
    p.block_scale = static_cast<uint8_t *>(block_scale);
    p.y = write_y ? static_cast<uint16_t *>(y) : nullptr;
    p.M = M;
    p.H = (int)H;
    p.Kp4 = (int)(((H / 16) + 3) / 4);
    p.write_y = write_y ? 1 : 0;

    const LaunchShape ls = choose_shape(M, H, mode);
    p.seg = (int)(H / ls.cluster);

    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool parts = k > 1;
    cudaError_t e;
    switch (mode) {
        case MODE_NONE: e = launch_mode<MODE_NONE>(p, dtype, parts, ls, s); break;
        case MODE_FP8: e = launch_mode<MODE_FP8>(p, dtype, parts, ls, s); break;
        case MODE_NVFP4: e = launch_mode<MODE_NVFP4>(p, dtype, parts, ls, s); break;
        default: e = launch_mode<MODE_MXFP8>(p, dtype, parts, ls, s); break;
    }
    return e == cudaSuccess ? GNQ_OK : GNQ_ERR_CUDA;
}

__global__ void encode_kernel(const float *v, int64_t n, uint8_t *e4m3, uint8_t *e2m1) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float x = v[i];
        if (e4m3) e4m3[i] = (uint8_t)(e4m3x2(x, 0.f) & 0xFF);
        if (e2m1) e2m1[i] = (uint8_t)(e2m1x4(x, 0.f, 0.f, 0.f) & 0xF);
    }
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

int gnq_set_launch_policy(int cluster, int vpt) {
    if (cluster < 0 || cluster > 8 || (cluster & (cluster - 1))) return GNQ_ERR_SHAPE;
    if (vpt != 0 && vpt != 1 && vpt != 2 && vpt != 4) return GNQ_ERR_SHAPE;
    gnq::g_force_cluster.store(cluster);
    gnq::g_force_vpt.store(vpt);
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

}  // extern "C"
