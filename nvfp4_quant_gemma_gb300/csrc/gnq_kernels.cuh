// Fused residual add + Gemma RMSNorm + FP8 / NVFP4 / MXFP8 quantization
// kernels for sm_103a.
//
// Semantics: "vllm.models.qwen3_5.nvidia.ops.fused_norm_quant",
// gemma_add_rms_norm_quant (residual updated in place, norm scaled by
// (1 + w), quantized from the activation-dtype-rounded normed output, NVFP4
// block scales in the 128x4 swizzled layout); k-partial input per
// "vllm.models.qwen3_5.nvidia.ops.fused_allreduce_norm_quant" (partials summed
// with fp32 accumulation); MXFP8 per "vllm.model_executor.layers.
// fused_allreduce_gemma_rms_norm", allreduce_gemma_rms_norm_mxfp8.
//
// Design (GB300, HBM-bound, no tensor cores -- this is not a contraction):
//   * One CTA owns a row segment of `seg` elements: the whole row, or 1/C of
//     it when the row is split over a thread-block cluster of C CTAs (small
//     M, so that more SMs pull on HBM at once).  The partial sums of squares
//     of a cluster meet through distributed shared memory.
//   * Each thread owns VPT 16-byte chunks (8 elements) of the segment,
//     chunk c = v * blockDim.x + threadIdx.x, so each warp-wide access is one
//     contiguous 512-byte line.  Everything stays in registers: the row is
//     read from HBM exactly once and every output is written exactly once.
//   * Sum of squares: fp32, warp shuffle tree, then one shared-memory stage
//     whose partials every thread adds in the same fixed order.
//   * NVFP4: a 16-element block is two adjacent lanes; its amax takes one
//     xor-shuffle.  Four consecutive blocks (8 lanes) have their scale bytes
//     contiguous in the swizzled layout, so lane 8i gathers and stores them
//     as one 32-bit word.
//   * Every rounding step that decides a code uses IEEE round-to-nearest
//     intrinsics (__fdiv_rn, __fmul_rn, __fadd_rn), so no fused multiply-add
//     or approximate reciprocal can change a code.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gnq {

enum { MODE_NONE = -1, MODE_FP8 = 0, MODE_NVFP4 = 1, MODE_MXFP8 = 2 };

struct Params {
    const uint16_t *x;    // the activation, or partial 0 of k
    int64_t part_stride;  // elements from one partial to the next
    int k;                // number of partials (1 = plain activation)
    uint16_t *residual;   // (M, H) or nullptr; updated in place
    const uint16_t *w;    // (H,)
    float eps;
    float weight_bias;    // 1 for the Gemma norm, 0 for a plain RMSNorm
    const float *scale;   // device fp32: FP8 scale or NVFP4 global scale
    uint8_t *q;
    uint8_t *block_scale;
    uint16_t *y;          // (M, H) or nullptr
    int64_t M;
    int H;
    int Kp4;              // NVFP4: round_up(H/16, 4) / 4 scale tiles per 128 rows
    int seg;              // elements owned by one CTA (H / cluster size)
    int write_y;
};

// ---------------------------------------------------------------------------
// memory access (16-byte vectors; cache hints chosen for a one-pass stream)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    // read-only input touched once: no L1 allocation
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_inout(const void *p) {
    // the residual: read, then overwritten by the same thread
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_weight(const void *p) {
    // the norm weight is re-read by every row: keep it in L1
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void *p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void st_u32(void *p, uint32_t a) {
    asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}

__device__ __forceinline__ void st_u8(void *p, uint32_t a) {
    asm volatile("st.global.u8 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}

// ---------------------------------------------------------------------------
// 16-bit activation types: 8 values <-> one uint4
// ---------------------------------------------------------------------------
template <typename T> struct Act;

template <> struct Act<__nv_bfloat16> {
    static __device__ __forceinline__ void unpack(uint4 v, float f[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // round to nearest even
        return *reinterpret_cast<uint32_t *>(&b);
    }
};

template <> struct Act<__half> {
    static __device__ __forceinline__ void unpack(uint4 v, float f[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 p = __half22float2(h);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
    static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);  // round to nearest even
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

template <typename T> __device__ __forceinline__ uint4 pack8(const float f[8]) {
    uint4 r;
    r.x = Act<T>::pack2(f[0], f[1]);
    r.y = Act<T>::pack2(f[2], f[3]);
    r.z = Act<T>::pack2(f[4], f[5]);
    r.w = Act<T>::pack2(f[6], f[7]);
    return r;
}

// ---------------------------------------------------------------------------
// element encoders (hardware conversions, round to nearest even, saturating)
// ---------------------------------------------------------------------------
// Two E4M3 codes in 16 bits, `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// Four E2M1 codes in 16 bits: element 0 in bits 0-3, element 1 in 4-7, ...
__device__ __forceinline__ uint32_t e2m1x4(float v0, float v1, float v2, float v3) {
    uint16_t d;
    asm("{\n\t.reg .b8 lo8, hi8;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 lo8, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 hi8, %4, %3;\n\t"
        "mov.b16 %0, {lo8, hi8};\n\t}"
        : "=h"(d)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
    return d;
}

// Value of a finite E4M3 code (bias 7, 3 fraction bits), exact in fp32.
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    const uint32_t e = (code >> 3) & 0xF, f = code & 0x7;
    const float mag = e ? __uint_as_float(((e + 120u) << 23) | (f << 20))  // (1+f/8)*2^(e-7)
                        : (float)f * 0.001953125f;                          // f/8 * 2^-6
    return (code & 0x80) ? -mag : mag;
}

// ---------------------------------------------------------------------------
// cluster helpers (distributed shared memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_peer_f32(const float *local, uint32_t rank) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(local), ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Byte offset of block scale (m, b) in the 128x4 swizzled layout, for b % 4 == 0.
__device__ __forceinline__ int64_t swizzled_group(int64_t m, int b, int Kp4) {
    return ((m >> 7) * Kp4 + (b >> 2)) * 512 + (m & 31) * 16 + ((m >> 5) & 3) * 4;
}

// ---------------------------------------------------------------------------
// the row kernel
// ---------------------------------------------------------------------------
template <typename T, int MODE, bool PARTS, int VPT>
__global__ void __launch_bounds__(1024 / VPT) row_kernel(const __grid_constant__ Params p) {
    __shared__ float warp_ss[32];
    __shared__ float cta_ss;

    const uint32_t C = cluster_size();
    const uint32_t rank = C > 1 ? cluster_rank() : 0;
    const int64_t m = blockIdx.x / C;
    const int NT = blockDim.x;
    const int t = threadIdx.x;
    const int nch = p.seg >> 3;
    const int64_t row = m * (int64_t)p.H;

    int col[VPT];
    bool ok[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * NT + t;
        ok[v] = c < nch;
        col[v] = (int)rank * p.seg + c * 8;
    }

    // ---- issue every load of the row segment up front ----
    uint4 rv[VPT], xv[VPT], wv[VPT];
    const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        rv[v] = (p.residual && ok[v]) ? ld_inout(p.residual + row + col[v]) : zero;
        xv[v] = ok[v] ? ld_stream(p.x + row + col[v]) : zero;
    }
    if (PARTS) {
        // a = dtype(((p0 + p1) + p2) + ...), fp32 accumulation in index order.
        // Partials are fetched four at a time so their loads are in flight
        // together; the adds still run strictly in index order.
        float acc[VPT][8];
#pragma unroll
        for (int v = 0; v < VPT; ++v) Act<T>::unpack(xv[v], acc[v]);
        for (int p0 = 1; p0 < p.k; p0 += 4) {
            uint4 pv[4][VPT];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint16_t *xp = p.x + (p0 + j) * p.part_stride + row;
#pragma unroll
                for (int v = 0; v < VPT; ++v)
                    pv[j][v] = (p0 + j < p.k && ok[v]) ? ld_stream(xp + col[v]) : zero;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (p0 + j < p.k) {
#pragma unroll
                    for (int v = 0; v < VPT; ++v) {
                        float f[8];
                        Act<T>::unpack(pv[j][v], f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[v][i] = __fadd_rn(acc[v][i], f[i]);
                    }
                }
            }
        }
#pragma unroll
        for (int v = 0; v < VPT; ++v) xv[v] = pack8<T>(acc[v]);
    }
#pragma unroll
    for (int v = 0; v < VPT; ++v) wv[v] = ok[v] ? ld_weight(p.w + col[v]) : zero;

    float qscale = 0.f;
    if (MODE == MODE_FP8 || MODE == MODE_NVFP4) qscale = __ldg(p.scale);

    // ---- h = dtype(a + residual), residual <- h, sum of squares ----
    float h[VPT][8];
    float ss = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        Act<T>::unpack(xv[v], h[v]);
        if (p.residual) {
            float r[8];
            Act<T>::unpack(rv[v], r);
#pragma unroll
            for (int i = 0; i < 8; ++i) r[i] = __fadd_rn(h[v][i], r[i]);
            const uint4 hb = pack8<T>(r);
            if (ok[v]) st_v4(p.residual + row + col[v], hb);
            Act<T>::unpack(hb, h[v]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(h[v][i], h[v][i], ss);
    }

    // ---- row reduction: warps, then CTA, then cluster ----
    ss = warp_sum(ss);
    if ((t & 31) == 0) warp_ss[t >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int i = 0; i < (NT >> 5); ++i) tot += warp_ss[i];
    if (C > 1) {
        if (t == 0) cta_ss = tot;
        cluster_arrive_release();
        cluster_wait();
        tot = 0.f;
        for (uint32_t r = 0; r < C; ++r) tot += ld_peer_f32(&cta_ss, r);
        cluster_arrive_relaxed();  // this CTA's reads of its peers are done
    }
    const float inv = __frsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)p.H), p.eps));

    // ---- y = dtype(h * inv * (bias + w)), then quantize the rounded y ----
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        float wf[8], yf[8];
        Act<T>::unpack(wv[v], wf);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            yf[i] = __fmul_rn(__fmul_rn(h[v][i], inv), __fadd_rn(p.weight_bias, wf[i]));
        const uint4 yb = pack8<T>(yf);
        if (p.write_y && ok[v]) st_v4(p.y + row + col[v], yb);
        Act<T>::unpack(yb, yf);  // the rounded y feeds the quantizer

        if (MODE == MODE_FP8) {
            float d[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) d[i] = __fdiv_rn(yf[i], qscale);
            const uint32_t lo = e4m3x2(d[0], d[1]) | (e4m3x2(d[2], d[3]) << 16);
            const uint32_t hi = e4m3x2(d[4], d[5]) | (e4m3x2(d[6], d[7]) << 16);
            if (ok[v]) st_v2(p.q + row + col[v], lo, hi);
        } else if (MODE == MODE_NVFP4) {
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(yf[i]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // 16-element block
            const float sf32 = __fmul_rn(qscale, __fdiv_rn(amax, 6.0f));
            const uint32_t sf = e4m3x2(sf32, 0.f) & 0xFF;
            const float sfv = e4m3_value(sf);
            const float es = sfv == 0.f ? 0.f : __fdiv_rn(qscale, sfv);
#pragma unroll
            for (int i = 0; i < 8; ++i) yf[i] = __fmul_rn(yf[i], es);
            const uint32_t codes = e2m1x4(yf[0], yf[1], yf[2], yf[3]) |
                                   (e2m1x4(yf[4], yf[5], yf[6], yf[7]) << 16);
            if (ok[v]) st_u32(p.q + ((row + col[v]) >> 1), codes);
            // scale bytes of 4 consecutive blocks (lanes 8i, 8i+2, 8i+4, 8i+6)
            const uint32_t s1 = __shfl_down_sync(0xffffffffu, sf, 2);
            const uint32_t s2 = __shfl_down_sync(0xffffffffu, sf, 4);
            const uint32_t s3 = __shfl_down_sync(0xffffffffu, sf, 6);
            if (ok[v] && (t & 7) == 0) {
                const uint32_t word = sf | (s1 << 8) | (s2 << 16) | (s3 << 24);
                st_u32(p.block_scale + swizzled_group(m, col[v] >> 4, p.Kp4), word);
            }
        } else if (MODE == MODE_MXFP8) {
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(yf[i]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));  // 32-element block
            int code = 0;
            if (amax > 0.f) code = min(max(ilogbf(amax) - 8 + 127, 0), 254);
            const float inv_x = ldexpf(1.0f, 127 - code);  // 1 / 2^(code-127), exact
            float d[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) d[i] = __fmul_rn(yf[i], inv_x);
            const uint32_t lo = e4m3x2(d[0], d[1]) | (e4m3x2(d[2], d[3]) << 16);
            const uint32_t hi = e4m3x2(d[4], d[5]) | (e4m3x2(d[6], d[7]) << 16);
            if (ok[v]) st_v2(p.q + row + col[v], lo, hi);
            if (ok[v] && (t & 3) == 0)
                st_u8(p.block_scale + m * (int64_t)(p.H >> 5) + (col[v] >> 5), (uint32_t)code);
        }
    }

    if (C > 1) cluster_wait();  // peers may still be reading this CTA's partial
}

}  // namespace gnq
