// Device building blocks of the fused add + Gemma RMSNorm + quant kernels
// (sm_103a): vector memory access, 16-bit activation packing, the hardware
// FP8/FP4 encoders, exact quotients, cluster and bulk-copy/mbarrier helpers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gnq {

enum { MODE_NONE = -1, MODE_FP8 = 0, MODE_NVFP4 = 1, MODE_MXFP8 = 2 };

// Bits of the device error word (set by a kernel, read by gnq_device_error).
enum { DEVERR_WAIT_TIMEOUT = 1 };

// Compile-time options of a kernel instance (the OPT template argument):
//   OPT_A32     NVFP4: every 16-bit tensor is 32-byte aligned, so a unit's
//               32-byte block of x, residual, partials, w and y moves in one
//               256-bit access;
//   OPT_EARLYW  the weight and the quantizer constants are read before the
//               wait on the preceding grid (the caller guarantees no
//               preceding kernel writes them).
enum { OPT_A32 = 1, OPT_EARLYW = 2 };

struct Params {
    const uint16_t *x;    // the activation, or partial 0 of k
    int64_t part_stride;  // elements from one partial to the next
    int k;                // number of partials (1 = plain activation)
    uint16_t *residual;   // (M, H) or nullptr; updated in place
    const uint16_t *w;    // (H,)
    float eps;
    float inv_h;          // RN(1 / H)
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
    int stages;           // streaming kernel: rows in flight per CTA
    unsigned int *err;    // device error word
    long long wait_limit; // clock cycles a bounded wait may spin
    uint32_t tx_extra;    // test hook: bytes announced per row beyond the copies (0 or 16)
    int pf_ctas;          // row kernel: CTAs below this index prefetch their rows before the wait
};

// ---------------------------------------------------------------------------
// global memory (16-byte vectors; cache hints for a one-pass stream)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;  // read-only input touched once: no L1 allocation
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_inout(const void *p) {
    uint4 r;  // the residual: read, then overwritten by the same thread
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_weight(const void *p) {
    uint4 r;  // the norm weight is re-read by every row: keep it in L1
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
// Predicated stores: the store is skipped when `on` is false, without a
// branch, so the code around it stays one basic block.
__device__ __forceinline__ void st_v4_if(void *p, uint4 v, bool on) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
                 "@q st.global.v4.u32 [%0], {%1,%2,%3,%4};\n\t}" ::"l"(p),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"((int)on)
                 : "memory");
}
__device__ __forceinline__ void st_v2_if(void *p, uint32_t a, uint32_t b, bool on) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %3, 0;\n\t"
                 "@q st.global.v2.u32 [%0], {%1,%2};\n\t}" ::"l"(p), "r"(a), "r"(b), "r"((int)on)
                 : "memory");
}
__device__ __forceinline__ void st_u8_if(void *p, uint32_t a, bool on) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
                 "@q st.global.u8 [%0], %1;\n\t}" ::"l"(p), "r"(a), "r"((int)on)
                 : "memory");
}

// 32-byte (256-bit) accesses of two adjacent 16-byte chunks, for 32-byte
// aligned addresses: one request per warp covers 1 KB of whole sectors.
__device__ __forceinline__ void ld_stream_v8(const void *p, uint4 &a, uint4 &b) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                   "=r"(b.w)
                 : "l"(p));
}
__device__ __forceinline__ void ld_inout_v8(const void *p, uint4 &a, uint4 &b) {
    asm volatile("ld.global.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                   "=r"(b.w)
                 : "l"(p));
}
__device__ __forceinline__ void ld_weight_v8(const void *p, uint4 &a, uint4 &b) {
    asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                   "=r"(b.w)
                 : "l"(p));
}
__device__ __forceinline__ void st_v8(void *p, uint4 a, uint4 b) {
    asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y),
                 "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}
__device__ __forceinline__ void st_v8_if(void *p, uint4 a, uint4 b, bool on) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %9, 0;\n\t"
                 "@q st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n\t}" ::"l"(p),
                 "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w),
                 "r"((int)on)
                 : "memory");
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

// ---------------------------------------------------------------------------
// 16-bit activation types: 8 values <-> one uint4
// ---------------------------------------------------------------------------
template <typename T> struct Act;

template <> struct Act<__nv_bfloat16> {
    static __device__ __forceinline__ void unpack2(uint32_t w, float &lo, float &hi) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xFFFF0000u);
    }
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
    static __device__ __forceinline__ void unpack2(uint32_t w, float &lo, float &hi) {
        const float2 p = __half22float2(*reinterpret_cast<const __half2 *>(&w));
        lo = p.x;
        hi = p.y;
    }
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

// Correctly rounded 16-bit sums of two packed pairs (equal to the fp32 sum
// rounded once: the fp32 sum of two 16-bit values cannot land on a 16-bit
// rounding tie it would not have exactly).
template <typename T> __device__ __forceinline__ uint32_t add16x2(uint32_t a, uint32_t b);
template <> __device__ __forceinline__ uint32_t add16x2<__nv_bfloat16>(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
template <> __device__ __forceinline__ uint32_t add16x2<__half>(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
template <typename T> __device__ __forceinline__ uint4 add16x8(uint4 a, uint4 b) {
    return make_uint4(add16x2<T>(a.x, b.x), add16x2<T>(a.y, b.y), add16x2<T>(a.z, b.z),
                      add16x2<T>(a.w, b.w));
}

// acc + sum of squares of the 8 packed 16-bit values in v: mixed-precision
// fused multiply-adds (the square of a 16-bit value is exact in fp32, one
// rounding per add), two chains for latency.
template <typename T> __device__ __forceinline__ float sumsq16x8(uint4 v, float acc);
#define GNQ_SUMSQ(TY, PTXT)                                                               \
    template <> __device__ __forceinline__ float sumsq16x8<TY>(uint4 v, float acc) {     \
        float a = acc, b = 0.f;                                                           \
        asm("{\n\t.reg .b16 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"                         \
            "mov.b32 {l0, h0}, %2;\n\tmov.b32 {l1, h1}, %3;\n\t"                          \
            "mov.b32 {l2, h2}, %4;\n\tmov.b32 {l3, h3}, %5;\n\t"                          \
            "fma.rn.f32." PTXT " %0, l0, l0, %0;\n\tfma.rn.f32." PTXT " %1, h0, h0, %1;\n\t" \
            "fma.rn.f32." PTXT " %0, l1, l1, %0;\n\tfma.rn.f32." PTXT " %1, h1, h1, %1;\n\t" \
            "fma.rn.f32." PTXT " %0, l2, l2, %0;\n\tfma.rn.f32." PTXT " %1, h2, h2, %1;\n\t" \
            "fma.rn.f32." PTXT " %0, l3, l3, %0;\n\tfma.rn.f32." PTXT " %1, h3, h3, %1;\n\t}" \
            : "+f"(a), "+f"(b)                                                            \
            : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));                                    \
        return a + b;                                                                     \
    }
GNQ_SUMSQ(__nv_bfloat16, "bf16")
GNQ_SUMSQ(__half, "f16")
#undef GNQ_SUMSQ

// a_i = RN(h_i * w_i + h_i * b) for the 8 packed 16-bit h and w and a 16-bit
// b (the low half of `b16`) that is 0 or 1: h_i * b is formed exactly by a
// first mixed-precision FMA (addend -0, so it is h_i, +-0 or -0), then the
// product with w is added in a second (h * w exact, one rounding).  No
// select on the bias, no fp32 copy of h.
template <typename T> __device__ __forceinline__ void biasfma16x8(uint4 h, uint4 w, uint32_t b16, float (&c)[8]);
#define GNQ_BFMA16(TY, PTXT)                                                                     \
    template <>                                                                                  \
    __device__ __forceinline__ void biasfma16x8<TY>(uint4 h, uint4 w, uint32_t b16, float (&c)[8]) { \
        asm("{\n\t.reg .b16 a0, b0, a1, b1, a2, b2, a3, b3, p0, q0, p1, q1, p2, q2, p3, q3, bb, bz;\n\t" \
            ".reg .f32 t0, t1, t2, t3, t4, t5, t6, t7;\n\t"                                          \
            "mov.b32 {a0, b0}, %8;\n\tmov.b32 {a1, b1}, %9;\n\t"                                  \
            "mov.b32 {a2, b2}, %10;\n\tmov.b32 {a3, b3}, %11;\n\t"                                \
            "mov.b32 {p0, q0}, %12;\n\tmov.b32 {p1, q1}, %13;\n\t"                                \
            "mov.b32 {p2, q2}, %14;\n\tmov.b32 {p3, q3}, %15;\n\t"                                \
            "mov.b32 {bb, bz}, %16;\n\t"                                                            \
            "fma.rn.f32." PTXT " t0, a0, bb, 0f80000000;\n\tfma.rn.f32." PTXT " t1, b0, bb, 0f80000000;\n\t" \
            "fma.rn.f32." PTXT " t2, a1, bb, 0f80000000;\n\tfma.rn.f32." PTXT " t3, b1, bb, 0f80000000;\n\t" \
            "fma.rn.f32." PTXT " t4, a2, bb, 0f80000000;\n\tfma.rn.f32." PTXT " t5, b2, bb, 0f80000000;\n\t" \
            "fma.rn.f32." PTXT " t6, a3, bb, 0f80000000;\n\tfma.rn.f32." PTXT " t7, b3, bb, 0f80000000;\n\t" \
            "fma.rn.f32." PTXT " %0, a0, p0, t0;\n\tfma.rn.f32." PTXT " %1, b0, q0, t1;\n\t"     \
            "fma.rn.f32." PTXT " %2, a1, p1, t2;\n\tfma.rn.f32." PTXT " %3, b1, q1, t3;\n\t"     \
            "fma.rn.f32." PTXT " %4, a2, p2, t4;\n\tfma.rn.f32." PTXT " %5, b2, q2, t5;\n\t"     \
            "fma.rn.f32." PTXT " %6, a3, p3, t6;\n\tfma.rn.f32." PTXT " %7, b3, q3, t7;\n\t}"    \
            : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3]), "=f"(c[4]), "=f"(c[5]),             \
              "=f"(c[6]), "=f"(c[7])                                                                \
            : "r"(h.x), "r"(h.y), "r"(h.z), "r"(h.w), "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w),      \
              "r"(b16));                                                                            \
    }
GNQ_BFMA16(__nv_bfloat16, "bf16")
GNQ_BFMA16(__half, "f16")
#undef GNQ_BFMA16

// 1.0 as a 16-bit pattern of T.
template <typename T> __device__ __forceinline__ uint32_t one16();
template <> __device__ __forceinline__ uint32_t one16<__nv_bfloat16>() { return 0x3F80u; }
template <> __device__ __forceinline__ uint32_t one16<__half>() { return 0x3C00u; }

// Per-lane max(|a|, |b|) of two packed pairs (signs of the result are junk).
template <typename T> __device__ __forceinline__ uint32_t absmax16x2(uint32_t a, uint32_t b);
template <> __device__ __forceinline__ uint32_t absmax16x2<__nv_bfloat16>(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
template <> __device__ __forceinline__ uint32_t absmax16x2<__half>(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// max |v| over the 8 values of one packed chunk, as fp32 (exact; NaN lanes
// drop out, as in fmax).
template <typename T> __device__ __forceinline__ float absmax8(uint4 a) {
    const uint32_t m = absmax16x2<T>(absmax16x2<T>(a.x, a.y), absmax16x2<T>(a.z, a.w));
    float lo, hi;
    Act<T>::unpack2(m, lo, hi);
    return fmaxf(fabsf(lo), fabsf(hi));
}

// MXFP8 scale of a block amax (>= 0, or inf): the E8M0 code
// floor(log2(amax)) - 8 + 127 clamped to [0, 254] -- read off the fp32
// exponent field e: e - 8 for a normal amax, 0 for zero and subnormals
// (their floor(log2) is at most -127), 254 for inf -- and the exact
// multiplier 2^(127 - code) that divides the block by the scale.
__device__ __forceinline__ uint32_t e8m0_code(float amax) {
    const uint32_t e = __float_as_uint(amax) >> 23;
    return e == 255u ? 254u : (e > 8u ? e - 8u : 0u);
}
__device__ __forceinline__ float e8m0_inverse(uint32_t code) {
    return code == 254u ? 0x1p-127f : __uint_as_float((254u - code) << 23);
}

// max |v| over the 16 values of two packed chunks, as fp32 (exact).
template <typename T> __device__ __forceinline__ float absmax16(uint4 a, uint4 b) {
    const uint32_t m = absmax16x2<T>(
        absmax16x2<T>(absmax16x2<T>(a.x, a.y), absmax16x2<T>(a.z, a.w)),
        absmax16x2<T>(absmax16x2<T>(b.x, b.y), absmax16x2<T>(b.z, b.w)));
    float lo, hi;
    Act<T>::unpack2(m, lo, hi);
    return fmaxf(fabsf(lo), fabsf(hi));
}

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

// Four E4M3 codes in 32 bits, element 0 in the low byte.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
    uint32_t d;
    asm("{\n\t.reg .b16 a, b;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 a, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 b, %4, %3;\n\t"
        "mov.b32 %0, {a, b};\n\t}"
        : "=r"(d)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
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

// Eight E2M1 codes in 32 bits, element i in bits 4i..4i+3.
__device__ __forceinline__ uint32_t e2m1x8(const float v[8]) {
    uint32_t d;
    asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n\t"
        "mov.b16 lo, {c0, c1};\n\t"
        "mov.b16 hi, {c2, c3};\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(d)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return d;
}

// Value of an E4M3 code (bias 7, 3 fraction bits; S.1111.111 is NaN), exact in fp32.
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    const uint32_t e = (code >> 3) & 0xF, f = code & 0x7;
    float mag = e ? __uint_as_float(((e + 120u) << 23) | (f << 20))  // (1+f/8)*2^(e-7)
                  : (float)f * 0.001953125f;                          // f/8 * 2^-6
    if (e == 0xF && f == 0x7) mag = __uint_as_float(0x7FC00000u);
    return (code & 0x80) ? -mag : mag;
}

// ---------------------------------------------------------------------------
// exact quotients
// ---------------------------------------------------------------------------
// Correctly rounded a / b from r = RN(1/b) with the FMA correction step of
// P. W. Markstein ("Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q0 = RN(a*r) is
// within one ulp of a/b, the remainder a - q0*b is then exact in one fused
// multiply-add, and RN(q0 + rem*r) is the correctly rounded quotient.
// Requires b and r normal and |a| >= 2^-103 (so the remainder cannot
// underflow); a zero or non-finite q0 is returned as is.
__device__ __forceinline__ float div_fma(float a, float b, float r, float &q0) {
    q0 = __fmul_rn(a, r);
    const float rem = __fmaf_rn(-q0, b, a);
    return __fmaf_rn(rem, r, q0);
}

// ---------------------------------------------------------------------------
// paired fp32 arithmetic (Blackwell f32x2: two IEEE round-to-nearest lanes)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pk2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// In-place element-wise helpers on arrays of n (even) floats.
template <int N> __device__ __forceinline__ void mul_arr(float (&v)[N], const float *w) {
#pragma unroll
    for (int i = 0; i < N; i += 2) upk2(mul2(pk2(v[i], v[i + 1]), pk2(w[i], w[i + 1])), v[i], v[i + 1]);
}
template <int N> __device__ __forceinline__ void mul_arr_s(float *v, float c) {
    const uint64_t cc = pk2(c, c);
#pragma unroll
    for (int i = 0; i < N; i += 2) upk2(mul2(pk2(v[i], v[i + 1]), cc), v[i], v[i + 1]);
}

// The static FP8 quotient y / s as the E4M3 encoder needs it.  Two paths,
// chosen once per CTA:
//   FP8_PAIR  (2^-80 <= s <= 2^80): the correction step on pairs, in negated
//             form: n0 = RN(y * -r), rem = y + n0 * s (exact),
//             n1 = RN(rem * -r + n0) = -RN(y / s), signed zeros included; the
//             code signs are flipped back.  The correction is exact for
//             |y| >= 2^-103 (below that |y/s| < 2^-23, a zero code of the
//             right sign either way).  y * (1/s) must be finite: fp16 y is at
//             most 65504 < 2^126 * s; bf16 y is first clamped to
//             |y| <= ylim = RD_bf16(1024 s) with its sign kept (any clamped
//             value has a quotient >= 464 that saturates to 448, like the
//             true one; NaN passes through).
//   FP8_IEEE  other scales: IEEE division.
enum { FP8_IEEE = 0, FP8_PAIR = 2 };

struct Fp8Div {
    float s, r;
    uint32_t ylim2;  // RD_bf16(1024 s), in both halves of a bf16x2 word
    float ylim;      // the same value as fp32
    bool fast;
};

__device__ __forceinline__ Fp8Div make_fp8_div(float s) {
    Fp8Div d;
    d.s = s;
    d.r = __frcp_rn(s);
    d.fast = s >= 0x1p-80f && s <= 0x1p80f;
    const uint32_t t = __float_as_uint(s * 1024.f) >> 16;  // exact product, then toward zero
    d.ylim2 = t | (t << 16);
    d.ylim = __uint_as_float(t << 16);
    return d;
}

__device__ __forceinline__ float min_nan(float a, float b) {
    float d;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// Both bf16 halves of v with their magnitude clamped to ylim2's, signs kept.
__device__ __forceinline__ uint32_t clamp_bf16x2(uint32_t v, uint32_t ylim2) {
    uint32_t d;
    asm("min.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(v), "r"(ylim2));
    return d;
}

// Eight E4M3 codes of y[0..8) / s as two words (y already clamped for bf16).
template <int PATH>
__device__ __forceinline__ void fp8_codes8(const float *y, const Fp8Div &d, uint32_t &lo,
                                           uint32_t &hi) {
    float q[8];
    if constexpr (PATH == FP8_PAIR) {
        const uint64_t nr = pk2(-d.r, -d.r), s2 = pk2(d.s, d.s);
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const uint64_t y2 = pk2(y[i], y[i + 1]);
            const uint64_t n0 = mul2(y2, nr);
            const uint64_t rem = fma2(n0, s2, y2);
            upk2(fma2(rem, nr, n0), q[i], q[i + 1]);
        }
        lo = e4m3x4(q[0], q[1], q[2], q[3]) ^ 0x80808080u;
        hi = e4m3x4(q[4], q[5], q[6], q[7]) ^ 0x80808080u;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(y[i], d.s);
        lo = e4m3x4(q[0], q[1], q[2], q[3]);
        hi = e4m3x4(q[4], q[5], q[6], q[7]);
    }
}

// amax / 6 correctly rounded, for amax the magnitude of a 16-bit value (0,
// finite, inf or NaN).  The correction step above is exact for every finite
// bf16 and fp16 magnitude, subnormals and the largest bf16 values included
// (an exhaustive check in exact rational arithmetic), and gives 0 for 0 and
// NaN for NaN; only inf needs its own answer.
__device__ __forceinline__ float div6(float amax) {
    float q0;
    const float q1 = div_fma(amax, 6.0f, 0.16666667163372039794921875f /* RN(1/6) */, q0);
    return amax == __int_as_float(0x7F800000) ? amax : q1;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// Wait until the grid this one depends on has completed and its memory is
// visible (returns at once when the launch was not programmatic).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the dependent grid to begin launching.  Every grid triggers right
// after its wait, at every batch size: the dependent launches only once all
// of this grid's CTAs have started, so it can only take SMs this grid has
// released.  With a stand-in next-layer kernel as the dependent (the bench's
// PDL consumer sweep, M = 1..8192 at H = 5120) the early trigger led plain
// launches and a trigger at exit at every M in FP8 and NVFP4, including
// M >= 192, where "vllm.models.qwen3_5.nvidia.ops.fused_norm_quant"
// (gemma_add_rms_norm_quant, TRIGGER_EARLY) turns its early trigger off
// because the prelaunched next linear took SMs.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
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

// ---------------------------------------------------------------------------
// bulk copies into shared memory, completed on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after `limit` cycles (2^31, about a second, unless
// a test asks for less) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}
// 1-D bulk copy global -> this CTA's shared memory; bytes and both
// addresses are multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// Cache hints: bring global memory into L2 (no value is read, no effect on
// what a later load returns; L2 is where every SM's accesses meet).
// `last`: with the evict-last priority, kept in L2 ahead of other lines.
__device__ __forceinline__ void prefetch_l2_line(const void *p, bool last) {
    if (last) asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
    else asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte offset of block scale (m, b) in the 128x4 swizzled layout, for b % 4 == 0.
__device__ __forceinline__ int64_t swizzled_group(int64_t m, int b, int Kp4) {
    return ((m >> 7) * Kp4 + (b >> 2)) * 512 + (m & 31) * 16 + ((m >> 5) & 3) * 4;
}

}  // namespace gnq
