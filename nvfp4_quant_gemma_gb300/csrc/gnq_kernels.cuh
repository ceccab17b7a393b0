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
// Two kernels share one per-unit epilogue (y, quantization, stores):
//
//   row_kernel     one CTA per row -- or, for rows wider than 1024 units, a
//                  thread-block cluster of C CTAs meeting through distributed
//                  shared memory -- with the inputs loaded straight into
//                  registers.  Every batch with one activation and a
//                  residual, every batch below 16 x SMs rows, and batches
//                  that write y.
//   stream_kernel  persistent CTAs, each walking rows blockIdx.x, +grid, ...
//                  The inputs of the next `stages` rows stream into a shared
//                  memory ring by 1-D bulk copies completed on mbarriers, so
//                  DRAM latency hides behind the arithmetic of earlier rows.
//                  Large batches without a residual, and k partials.
//
// Each exists as two __global__ wrappers around one inlined body: the
// FP8 / MXFP8 / no-quant instances (register choice left to the compiler)
// and the *_nvfp4 instances (explicit register budgets, RowForm and
// StreamForm).
//
// Work inside a CTA: a thread owns VPT units of U contiguous 16-byte chunks
// (8U elements; U = 2 for NVFP4, so a thread holds whole 16-element blocks,
// else U = 1), unit u = v * blockDim.x + threadIdx.x, so a warp-wide access
// is one contiguous line.  Everything between the load and the stores stays
// in registers.  The sum of squares is an fp32 warp shuffle tree, then a
// second shuffle tree over the per-warp partials, the same in every warp.
// Every rounding that decides a code is an IEEE round-to-nearest operation
// (see gnq_device.cuh), so codes are exactly those of the fp32 reading.
//
// Both kernels wait on the preceding grid (programmatic dependent launch)
// before their first global read, so they may be launched while it drains,
// and every CTA then lets the dependent grid launch: it launches once all of
// this grid's CTAs have started (so it never takes their place), and its
// CTAs fill the SMs this grid's last wave leaves idle while they wait for
// this grid's results.
#pragma once

#include <type_traits>

#include "gnq_device.cuh"

namespace gnq {

template <int MODE> struct Unit {
    static constexpr int U = MODE == MODE_NVFP4 ? 2 : 1;  // chunks per unit
    static constexpr int E = 8 * U;                        // elements per unit
};

// Per-CTA quantization constants.
struct QuantCtx {
    Fp8Div fd;            // FP8: y / s
    float g;              // NVFP4 global scale
    const float *es_tab;  // NVFP4: element scale g / value(sf) per sf code (shared memory)
};

// NVFP4 element scale of a block-scale code: RN(g / value(code)), 0 for a
// zero scale.
__device__ __forceinline__ float element_scale(float g, uint32_t code) {
    const float v = e4m3_value(code);
    return v == 0.f ? 0.f : __fdiv_rn(g, v);
}

// Fill the NVFP4 element-scale table for all 256 codes.
__device__ __forceinline__ void fill_es_table(float *tab, float g, int t, int nt) {
    for (int c = t; c < 256; c += nt) tab[c] = element_scale(g, (uint32_t)c);
}

// TABLE: NVFP4 blocks look their element scale up in a per-CTA table (else
// each block divides once; see row_body).
template <bool TABLE = true>
__device__ __forceinline__ QuantCtx make_quant_ctx(const Params &p, int mode, float *es_smem,
                                                   int t, int nt) {
    QuantCtx qc;
    qc.fd = make_fp8_div(1.f);
    qc.g = 0.f;
    qc.es_tab = es_smem;
    if (mode == MODE_FP8) qc.fd = make_fp8_div(__ldg(p.scale));
    if (mode == MODE_NVFP4) {
        qc.g = __ldg(p.scale);
        if (TABLE) fill_es_table(es_smem, qc.g, t, nt);  // visible after the next __syncthreads
    }
    return qc;
}

// Output pointers of one row (computed once per row).
struct RowOut {
    uint16_t *y;   // y row
    uint8_t *q;    // code row (FP8/MXFP8: H bytes; NVFP4: H/2 bytes)
    uint8_t *sf;   // NVFP4: row part of the swizzled scale offsets; MXFP8: scale row
};

template <int MODE>
__device__ __forceinline__ RowOut row_out(const Params &p, int64_t m) {
    RowOut o;
    const int64_t row = m * (int64_t)p.H;
    o.y = p.y ? p.y + row : nullptr;
    o.q = MODE == MODE_NVFP4 ? p.q + (row >> 1) : p.q + row;
    o.sf = nullptr;
    if (MODE == MODE_NVFP4)  // tile row, then (m%32)*16 + ((m%128)/32)*4 inside the tile
        o.sf = p.block_scale + (m >> 7) * (int64_t)p.Kp4 * 512 + (m & 31) * 16 + ((m >> 5) & 3) * 4;
    if (MODE == MODE_MXFP8) o.sf = p.block_scale + m * (int64_t)(p.H >> 5);
    return o;
}

// Column part of the swizzled scale offset of the block starting at `col`.
__device__ __forceinline__ int sf_col_offset(int col) {
    const int b = col >> 4;
    return (b >> 2) * 512 + (b & 3);
}

// Out-of-range units (a row that is not a whole number of units per
// thread).  NVFP4 (Pred<MODE>): such a unit loads an in-range unit instead,
// adds nothing to the sum of squares and its stores are predicated off, so
// the long per-unit epilogue stays one basic block.  The other modes branch
// around the unit's loads (zero-filled) and stores, which measured faster
// for their shorter epilogues.
template <int MODE> struct Pred {
    static constexpr bool value = MODE == MODE_NVFP4;
};
template <bool PRED> __device__ __forceinline__ void st_v4_unit(void *p, uint4 v, bool ok) {
    if constexpr (PRED) st_v4_if(p, v, ok);
    else if (ok) st_v4(p, v);
}
template <bool PRED> __device__ __forceinline__ void st_v2_unit(void *p, uint32_t a, uint32_t b, bool ok) {
    if constexpr (PRED) st_v2_if(p, a, b, ok);
    else if (ok) st_v2(p, a, b);
}
template <bool PRED> __device__ __forceinline__ void st_v8_unit(void *p, uint4 a, uint4 b, bool ok) {
    if constexpr (PRED) st_v8_if(p, a, b, ok);
    else if (ok) st_v8(p, a, b);
}
template <bool PRED> __device__ __forceinline__ void st_u8_unit(void *p, uint32_t a, bool ok) {
    if constexpr (PRED) st_u8_if(p, a, ok);
    else if (ok) st_u8(p, a);
}

// One unit of y (8U values before rounding): round, store y, quantize the
// rounded values and store codes and scales.  `t` is the thread index;
// FP8PATH is the FP8 quotient path (FP8_*), uniform per CTA; `sfc` is the
// unit's sf_col_offset (NVFP4).  PRED: out-of-range units are predicated
// (Pred<MODE>), unless the instance has none (FULL).  V8: the two chunks of
// an NVFP4 unit's y leave in one 256-bit store (32-byte aligned y).  ESDIV:
// the NVFP4 element scale is divided out per block instead of looked up.
template <typename T, int MODE, int FP8PATH, bool PRED = Pred<MODE>::value, bool V8 = false,
          bool ESDIV = false>
__device__ __forceinline__ void epilogue_unit(const Params &p, const QuantCtx &qc,
                                              float (&yf)[Unit<MODE>::E], const RowOut &o,
                                              int col, int sfc, bool ok, int t) {
    constexpr int U = Unit<MODE>::U;
    uint4 yb[U];
#pragma unroll
    for (int c = 0; c < U; ++c) yb[c] = pack8<T>(&yf[8 * c]);
    if (PRED ? p.write_y != 0 : p.write_y && ok) {
        if constexpr (V8 && U == 2) {
            st_v8_unit<PRED>(o.y + col, yb[0], yb[1], ok);
        } else {
#pragma unroll
            for (int c = 0; c < U; ++c) st_v4_unit<PRED>(o.y + col + 8 * c, yb[c], ok);
        }
    }

    if (MODE == MODE_FP8) {
        uint4 yq = yb[0];
        if (FP8PATH == FP8_PAIR && std::is_same<T, __nv_bfloat16>::value) {
            // keep y * (1/s) finite; clamped values still saturate to 448
            yq.x = clamp_bf16x2(yq.x, qc.fd.ylim2);
            yq.y = clamp_bf16x2(yq.y, qc.fd.ylim2);
            yq.z = clamp_bf16x2(yq.z, qc.fd.ylim2);
            yq.w = clamp_bf16x2(yq.w, qc.fd.ylim2);
        }
        Act<T>::unpack(yq, yf);  // the rounded y feeds the quantizer
        uint32_t lo, hi;
        fp8_codes8<FP8PATH>(yf, qc.fd, lo, hi);
        st_v2_unit<false>(o.q + col, lo, hi, ok);
    } else if (MODE == MODE_NVFP4) {
        // one whole 16-element block per unit
        const float amax = absmax16<T>(yb[0], yb[1]);
        const float sf32 = __fmul_rn(qc.g, div6(amax));
        const uint32_t sf = e4m3x2(sf32, 0.f) & 0xFF;
        Act<T>::unpack(yb[0], &yf[0]);
        Act<T>::unpack(yb[1], &yf[8]);
        mul_arr_s<16>(yf, ESDIV ? element_scale(qc.g, sf) : qc.es_tab[sf]);
        const uint32_t lo = e2m1x8(&yf[0]);
        const uint32_t hi = e2m1x8(&yf[8]);
        st_v2_unit<PRED>(o.q + (col >> 1), lo, hi, ok);
        st_u8_unit<PRED>(o.sf + sfc, sf, ok);
    } else if (MODE == MODE_MXFP8) {
        // a 32-element block is the units of four consecutive lanes
        float amax = absmax8<T>(yb[0]);
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const uint32_t code = e8m0_code(amax);
        Act<T>::unpack(yb[0], yf);
        mul_arr_s<8>(yf, e8m0_inverse(code));  // y / 2^(code-127), exact
        const uint32_t lo = e4m3x4(yf[0], yf[1], yf[2], yf[3]);
        const uint32_t hi = e4m3x4(yf[4], yf[5], yf[6], yf[7]);
        st_v2_unit<false>(o.q + col, lo, hi, ok);
        st_u8_unit<false>(o.sf + (col >> 5), code, ok && (t & 3) == 0);
    }
}

// Sum of the per-warp partials in warp_ss[0..nw): each warp reduces them
// with the same shuffle tree, so every thread gets the same value (one
// shared load and ten shuffle/add steps per thread, whatever the CTA size).
__device__ __forceinline__ float block_total(const float *warp_ss, int nw, int lane) {
    float v = lane < nw ? warp_ss[lane] : 0.f;
    return warp_sum(v);
}

// The same total for CTAs of at most 8 warps: every thread reads the
// partials with two 16-byte shared loads and adds them left to right
// (slots beyond nw masked), in place of the shuffle tree.  Used by the NVFP4
// streaming instances (fp16 16384 x 8192 no-residual batch 57.46 ->
// 56.35 us, k = 4 partials 64.50 -> 64.15 us); the FP8 one measured 1 %
// slower with it.
__device__ __forceinline__ float block_total_small(const float *warp_ss, int nw, int lane) {
    if (nw > 8) return block_total(warp_ss, nw, lane);
    const float4 a = *reinterpret_cast<const float4 *>(warp_ss);
    const float4 b = *reinterpret_cast<const float4 *>(warp_ss + 4);
    float t = a.x;
    t += nw > 1 ? a.y : 0.f;
    t += nw > 2 ? a.z : 0.f;
    t += nw > 3 ? a.w : 0.f;
    if (nw > 4) {
        t += b.x;
        t += nw > 5 ? b.y : 0.f;
        t += nw > 6 ? b.z : 0.f;
        t += nw > 7 ? b.w : 0.f;
    }
    return t;
}

// inv = 1 / sqrt(mean(h^2) + eps); mean via the host-rounded 1/H.
__device__ __forceinline__ float inv_rms(const Params &p, float tot) {
    return rsqrtf(__fadd_rn(__fmul_rn(tot, p.inv_h), p.eps));
}

// ---------------------------------------------------------------------------
// row_kernel: one CTA (or cluster) per row, inputs straight to registers
// ---------------------------------------------------------------------------
// LEAN: h and w stay packed (mixed-precision FMAs; fewest registers).
// Otherwise h is unpacked once to fp32 (fewest instructions).
// Register budget of an NVFP4 row instance (row_kernel_nvfp4; the other
// modes leave the choice to the compiler, which an explicit budget, even
// one equal to the launch bound's, was measured to change for the worse).
// The forms the launch policy picks for one activation: 80 registers at
// four 16-byte chunks per thread (five resident CTAs of 160 threads; 64
// spills), 128 at eight (four CTAs of 128); the others keep what 1024 / VPT
// threads allow.
template <int MODE, int VPT, bool PARTS, bool LEAN> struct RowForm {
    static constexpr int U = Unit<MODE>::U, chunks = VPT * U;
    static constexpr int cap = VPT == 1 ? 64 : VPT == 2 ? 128 : 255;
    static constexpr int occ = chunks <= 2 ? 64
                               : chunks == 4 ? (U == 2 ? 80 : LEAN ? 64 : cap)
                                             : (LEAN ? 128 : cap);
    static constexpr int maxnreg = PARTS ? cap : occ;
};

// FULL: the launch guarantees every unit of the CTA's segment is in range
// (segment = VPT units x threads), so no unit needs a check.  OPT: OPT_A32
// and OPT_EARLYW (see gnq_device.cuh).
template <typename T, int MODE, bool PARTS, int VPT, bool LEAN, bool FULL, int OPT>
__device__ __forceinline__ void row_body(const Params &p, float *warp_ss, float &cta_ss,
                                         float *es_smem) {
    constexpr int U = Unit<MODE>::U, E = Unit<MODE>::E;
    constexpr bool V8 = (OPT & OPT_A32) && U == 2;
    constexpr bool EARLY = (OPT & OPT_EARLYW) != 0;
    // NVFP4 at one unit per thread (the small batches, bound by latency):
    // one division per block instead of a 256-entry table per CTA, which
    // would sit between the scale's load and the first block's codes (M = 1,
    // H = 5120: 1.80 -> 1.68 us).  With EARLY the table is built before the
    // wait and its lookup is the shorter path (1.59 us).
    constexpr bool ESDIV = MODE == MODE_NVFP4 && VPT == 1 && !EARLY;

    const uint32_t C = cluster_size();
    const uint32_t rank = C > 1 ? cluster_rank() : 0;
    const int64_t m = C > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
    const int NT = blockDim.x;
    const int t = threadIdx.x;
    const int nunits = p.seg / E;
    const int64_t row = m * (int64_t)p.H;

    constexpr bool PRED = Pred<MODE>::value;
    int col[VPT], lc[VPT];  // lc: the column a unit loads (PRED: clamped in range)
    bool ok[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int u = v * NT + t;
        ok[v] = FULL || u < nunits;
        col[v] = (int)rank * p.seg + u * E;
        lc[v] = PRED && !ok[v] ? (int)rank * p.seg : col[v];
    }

    uint4 rv[VPT][U], xv[VPT][U], wv[VPT][U];
    const uint4 zero = make_uint4(0, 0, 0, 0);
    auto load_w = [&]() {
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            if constexpr (V8) {
                if (PRED || ok[v]) ld_weight_v8(p.w + lc[v], wv[v][0], wv[v][1]);
                else wv[v][0] = wv[v][1] = zero;
            } else {
#pragma unroll
                for (int c = 0; c < U; ++c)
                    wv[v][c] = (PRED || ok[v]) ? ld_weight(p.w + lc[v] + 8 * c) : zero;
            }
        }
    };
    // The row segment's inputs into L2 while the preceding grid drains: a
    // hint only (the values are read after the wait), one 128-byte line per
    // thread and step.  Only the first wave's CTAs can still be waiting on
    // that grid, so only they prefetch (the M = 2048 NVFP4 batch 15.17 ->
    // 14.44 us, the decode batch 3.39 -> 2.75 us; done by every CTA it cost
    // the fp16 16384 x 8192 NVFP4 batch 1.7 %).
    if ((int)blockIdx.x < p.pf_ctas) {
        const int64_t seg0 = row + (int64_t)rank * p.seg;
        const int lines = (p.seg * 2 + 127) >> 7;
        // Batches of four waves or more keep the prefetched lines with the
        // evict-last priority (fp16 16384 x 8192: FP8 133.34 -> 131.95 us,
        // NVFP4 124.52 -> 123.13 us; below four waves it moved nothing or
        // lost, one-wave M = 256 batches 5-10 %).
        const bool last = p.M * (int64_t)C > 4 * (int64_t)p.pf_ctas;
        for (int op = 0; op < p.k; ++op) {
            const char *b = reinterpret_cast<const char *>(p.x + op * p.part_stride + seg0);
            for (int l = t; l < lines; l += NT) prefetch_l2_line(b + 128 * l, last);
        }
        if (p.residual) {
            const char *b = reinterpret_cast<const char *>(p.residual + seg0);
            for (int l = t; l < lines; l += NT) prefetch_l2_line(b + 128 * l, last);
        }
    }
    QuantCtx qc_early{};
    if constexpr (EARLY) {  // constants first, then the wait on the preceding grid
        load_w();
        qc_early = make_quant_ctx<!ESDIV>(p, MODE, es_smem, t, NT);
    }

    pdl_wait();  // inputs may come from the preceding grid
    pdl_trigger();

    // ---- issue every load of the row segment up front ----
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        if constexpr (V8) {
            if (p.residual && (PRED || ok[v])) ld_inout_v8(p.residual + row + lc[v], rv[v][0], rv[v][1]);
            else rv[v][0] = rv[v][1] = zero;
            if (PRED || ok[v]) ld_stream_v8(p.x + row + lc[v], xv[v][0], xv[v][1]);
            else xv[v][0] = xv[v][1] = zero;
        } else {
#pragma unroll
            for (int c = 0; c < U; ++c) {
                rv[v][c] = (p.residual && (PRED || ok[v])) ? ld_inout(p.residual + row + lc[v] + 8 * c) : zero;
                xv[v][c] = (PRED || ok[v]) ? ld_stream(p.x + row + lc[v] + 8 * c) : zero;
            }
        }
    }
    if (PARTS) {
        // a = dtype(((p0 + p1) + p2) + ...), fp32 accumulation in index order.
        // Partials are fetched four at a time so their loads are in flight
        // together; the adds still run strictly in index order.
        float acc[VPT][E];
#pragma unroll
        for (int v = 0; v < VPT; ++v)
#pragma unroll
            for (int c = 0; c < U; ++c) Act<T>::unpack(xv[v][c], &acc[v][8 * c]);
        for (int p0 = 1; p0 < p.k; p0 += 4) {
            uint4 pv[4][VPT][U];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint16_t *xp = p.x + (p0 + j) * p.part_stride + row;
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    const bool ld = p0 + j < p.k && (PRED || ok[v]);
                    if constexpr (V8) {
                        if (ld) ld_stream_v8(xp + lc[v], pv[j][v][0], pv[j][v][1]);
                        else pv[j][v][0] = pv[j][v][1] = zero;
                    } else {
#pragma unroll
                        for (int c = 0; c < U; ++c) pv[j][v][c] = ld ? ld_stream(xp + lc[v] + 8 * c) : zero;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (p0 + j < p.k) {
#pragma unroll
                    for (int v = 0; v < VPT; ++v)
#pragma unroll
                        for (int c = 0; c < U; ++c) {
                            float f[8];
                            Act<T>::unpack(pv[j][v][c], f);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                acc[v][8 * c + i] = __fadd_rn(acc[v][8 * c + i], f[i]);
                        }
                }
            }
        }
#pragma unroll
        for (int v = 0; v < VPT; ++v)
#pragma unroll
            for (int c = 0; c < U; ++c) xv[v][c] = pack8<T>(&acc[v][8 * c]);
    }
    if constexpr (!EARLY) load_w();

    const QuantCtx qc = EARLY ? qc_early : make_quant_ctx<!ESDIV>(p, MODE, es_smem, t, NT);

    // ---- h = dtype(a + residual), sum of squares ----
    uint4 hb[VPT][U];                        // packed h (the new residual)
    float hf[VPT][LEAN ? 1 : E];             // h in fp32 (not LEAN)
    // PRED: a sum per unit, masked; otherwise one running sum (zero-filled
    // out-of-range units add nothing).
    float ss = 0.f;
    uint64_t ss2 = 0;                        // two fp32 partial sums (not LEAN)
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        float sv = 0.f;
        uint64_t sv2 = 0;
        float &acc = PRED ? sv : ss;
        uint64_t &acc2 = PRED ? sv2 : ss2;
#pragma unroll
        for (int c = 0; c < U; ++c) {
            hb[v][c] = p.residual ? add16x8<T>(xv[v][c], rv[v][c]) : xv[v][c];
            if constexpr (LEAN) {
                acc = sumsq16x8<T>(hb[v][c], acc);
            } else {
                float *hc = &hf[v][8 * c];
                Act<T>::unpack(hb[v][c], hc);
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const uint64_t h2 = pk2(hc[i], hc[i + 1]);
                    acc2 = fma2(h2, h2, acc2);
                }
            }
        }
        if constexpr (PRED) {
            if constexpr (!LEAN) {
                float a, b;
                upk2(sv2, a, b);
                sv = a + b;
            }
            ss += ok[v] ? sv : 0.f;
        }
    }
    if constexpr (!PRED && !LEAN) {
        float a, b;
        upk2(ss2, a, b);
        ss = a + b;
    }
    // A CTA outside a cluster stores the residual now; in a cluster it waits
    // until after the cluster barrier, whose release would otherwise have to
    // wait for these stores.
    auto store_residual = [&]() {
        if (p.residual) {
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                if constexpr (V8) {
                    st_v8_unit<PRED>(p.residual + row + col[v], hb[v][0], hb[v][1], ok[v]);
                } else {
#pragma unroll
                    for (int c = 0; c < U; ++c)
                        st_v4_unit<PRED>(p.residual + row + col[v] + 8 * c, hb[v][c], ok[v]);
                }
            }
        }
    };
    if (C == 1) store_residual();

    // ---- row reduction: warps, then CTA, then cluster ----
    ss = warp_sum(ss);
    if ((t & 31) == 0) warp_ss[t >> 5] = ss;
    __syncthreads();
    float tot = block_total(warp_ss, NT >> 5, t & 31);
    if (C > 1) {
        if (t == 0) cta_ss = tot;
        cluster_arrive_release();
        cluster_wait();
        tot = 0.f;
        for (uint32_t r = 0; r < C; ++r) tot += ld_peer_f32(&cta_ss, r);
        cluster_arrive_relaxed();  // this CTA's reads of its peers are done
        store_residual();
    }
    const float inv = inv_rms(p, tot);

    // ---- y = dtype(h * inv * (bias + w)), then quantize the rounded y ----
    // With bias 1 (Gemma) or 0 (plain) the weighted value is one mixed-
    // precision FMA on the packed h and w: a = RN(h * w + bias * h), then
    // y = RN(a * inv).
    const RowOut o = row_out<MODE>(p, m);
    const bool gemma = p.weight_bias == 1.f;
    const bool plain = p.weight_bias == 0.f;
    const uint32_t b16 = gemma ? one16<T>() : 0u;  // the bias as a 16-bit value (LEAN)
    auto finish = [&](auto path) {
        const uint64_t inv2 = pk2(inv, inv), bias2 = pk2(p.weight_bias, p.weight_bias);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            float yf[E];
#pragma unroll
            for (int c = 0; c < U; ++c) {
                float *a = &yf[8 * c];
                if constexpr (!LEAN) {
                    float wf[8];
                    Act<T>::unpack(wv[v][c], wf);
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        const uint64_t bw2 = add2(bias2, pk2(wf[i], wf[i + 1]));
                        const uint64_t hi2 = mul2(pk2(hf[v][8 * c + i], hf[v][8 * c + i + 1]), inv2);
                        upk2(mul2(hi2, bw2), a[i], a[i + 1]);
                    }
                } else if (gemma || plain) {
                    float hw[8];
                    biasfma16x8<T>(hb[v][c], wv[v][c], b16, hw);
#pragma unroll
                    for (int i = 0; i < 8; i += 2) upk2(mul2(pk2(hw[i], hw[i + 1]), inv2), a[i], a[i + 1]);
                } else {
                    float wf[8], hf[8];
                    Act<T>::unpack(wv[v][c], wf);
                    Act<T>::unpack(hb[v][c], hf);
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        const uint64_t bw2 = add2(bias2, pk2(wf[i], wf[i + 1]));
                        const uint64_t hi2 = mul2(pk2(hf[i], hf[i + 1]), inv2);
                        upk2(mul2(hi2, bw2), a[i], a[i + 1]);
                    }
                }
            }
            epilogue_unit<T, MODE, decltype(path)::value, PRED, V8, ESDIV>(
                p, qc, yf, o, col[v], sf_col_offset(col[v]), ok[v], t);
        }
    };
    if (MODE == MODE_FP8 && !qc.fd.fast) finish(std::integral_constant<int, FP8_IEEE>{});
    else finish(std::integral_constant<int, FP8_PAIR>{});

    if (C > 1) cluster_wait();  // peers may still be reading this CTA's partial
}

#define GNQ_ROW_SMEM                                  \
    __shared__ __align__(16) float warp_ss[32];       \
    __shared__ float cta_ss;                          \
    __shared__ float es_smem[MODE == MODE_NVFP4 ? 256 : 1];

// FP8, MXFP8 and no-quant rows: the compiler's own register choice.
template <typename T, int MODE, bool PARTS, int VPT, bool LEAN, bool FULL, int OPT>
__global__ void __launch_bounds__(1024 / VPT) row_kernel(const __grid_constant__ Params p) {
    GNQ_ROW_SMEM
    row_body<T, MODE, PARTS, VPT, LEAN, FULL, OPT>(p, warp_ss, cta_ss, es_smem);
}

// NVFP4 rows: the RowForm register budget (out-of-range units are
// predicated, so there is no FULL instance).
template <typename T, int MODE, bool PARTS, int VPT, bool LEAN, bool FULL, int OPT>
__global__ void __launch_bounds__(1024 / VPT) __maxnreg__((RowForm<MODE, VPT, PARTS, LEAN>::maxnreg))
    row_kernel_nvfp4(const __grid_constant__ Params p) {
    static_assert(MODE == MODE_NVFP4 && !FULL, "NVFP4 rows only");
    GNQ_ROW_SMEM
    row_body<T, MODE, PARTS, VPT, LEAN, false, OPT>(p, warp_ss, cta_ss, es_smem);
}
#undef GNQ_ROW_SMEM

// ---------------------------------------------------------------------------
// stream_kernel: persistent CTAs, rows streamed through a shared-memory ring
// ---------------------------------------------------------------------------
// Dynamic shared memory: stages x operands x (2H bytes), then one mbarrier
// per stage, then (StreamForm::smem_w) the fp32 table of bias + w.
// Operands of a row: partial 0..k-1, then the residual.
// LEAN: as for row_kernel, the weight kept packed; y comes from the mixed-
// precision FMA of the bias 1 (Gemma) or bias 0 (plain) form -- the host
// launches LEAN only for those two biases.
// NVFP4, not LEAN, several units per thread: bias + w lives in shared
// memory (chunk j of unit u at float4 index j * H/E + u, so a warp's reads
// are conflict-free), which frees the registers for a third resident CTA.

// Thread 0 of a streaming CTA whose wait for local row i (stage s, phase
// parity) gave up: set the error bit and wait, bounded, for every copy still
// in flight (rows i .. i + S - 1) before the CTA's shared memory goes away.
__device__ __forceinline__ void stream_drain(const Params &p, int i, int n_rows, int s, int S,
                                             uint32_t parity, uint32_t bars, uint4 *topup) {
    atomicOr(p.err, (unsigned)DEVERR_WAIT_TIMEOUT);
    for (int j = i; j < n_rows && j < i + S; ++j) {
        if (p.tx_extra)
            bulk_g2s((uint32_t)__cvta_generic_to_shared(&topup[s]), p.w, p.tx_extra, bars + 8u * s);
        mbar_wait_bounded(bars + 8u * s, parity, p.wait_limit);
        if (++s == S) {
            s = 0;
            parity ^= 1u;
        }
    }
}

// Thread 0 of a streaming CTA: its first n rows (m = b, b + G, ...) into L2
// before the wait.  Not inlined, so that the hot loop of the instances that
// call it keeps its own code.
static __device__ __noinline__ void stream_prefetch_rows(const Params &p, int64_t b, int G, int n,
                                                         uint32_t row_bytes) {
    for (int i = 0; i < n; ++i) {
        const int64_t m = b + (int64_t)i * G;
        for (int op = 0; op < p.k; ++op) prefetch_l2_bulk(p.x + op * p.part_stride + m * p.H, row_bytes);
        if (p.residual) prefetch_l2_bulk(p.residual + m * p.H, row_bytes);
    }
}

// maxnreg: the register budget of the NVFP4 instances (stream_kernel_nvfp4):
// 80 for the shared-memory-weight form at two units per thread (three
// resident CTAs of 256 threads), else what the launch bound allows.
template <int MODE, int VPT, bool LEAN> struct StreamForm {
    static constexpr bool smem_w = !LEAN && VPT >= 2 && MODE == MODE_NVFP4;
    static constexpr int maxnreg = VPT == 1 ? 64 : (smem_w && VPT <= 2 ? 80 : 128);
};

// FULL: the launch guarantees the row is exactly VPT units x threads.
// OPT_A32: the residual and y leave in 256-bit stores (NVFP4 units).
template <typename T, int MODE, bool PARTS, int VPT, bool LEAN, bool FULL, int OPT>
__device__ __forceinline__ void stream_body(const Params &p, uint8_t *dsmem, float (*warp_ss)[32],
                                            float *es_smem, uint4 *topup) {
    constexpr int U = Unit<MODE>::U, E = Unit<MODE>::E;
    constexpr bool V8 = (OPT & OPT_A32) && U == 2;
    constexpr bool SW = StreamForm<MODE, VPT, LEAN>::smem_w;
    constexpr bool PRED = Pred<MODE>::value && !FULL;  // FULL: no unit is out of range
    // MERGE: one barrier per row instead of two, where that measured faster:
    // the packed NVFP4 form (fp16 batch without residual 56.20 -> 55.41 us);
    // FP8 (62.07 -> 65.53 us) and the fp32 form with partials lost.
    constexpr bool MERGE = MODE == MODE_NVFP4 && LEAN;

    const int NT = blockDim.x;
    const int t = threadIdx.x;
    const int S = p.stages;
    const int G = gridDim.x;
    const int nops = p.k + (p.residual ? 1 : 0);
    const uint32_t row_bytes = (uint32_t)p.H * 2u;
    const uint32_t stage_bytes = row_bytes * nops;
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(dsmem);
    const uint32_t bars = base + stage_bytes * S;  // 8-byte aligned: row_bytes % 16 == 0
    // bias + w table (SW): 16-byte aligned, after the barriers
    float4 *const bw_s = reinterpret_cast<float4 *>(dsmem + ((stage_bytes * S + 8u * S + 15u) & ~15u));

    // rows of this CTA: m_i = blockIdx.x + i * G, i < n_rows
    const int n_rows = p.M > blockIdx.x ? (int)((p.M - 1 - blockIdx.x) / G + 1) : 0;

    // thread 0: start the loads of local row i into stage s
    auto issue = [&](int i, int s) {
        const int64_t m = blockIdx.x + (int64_t)i * G;
        const uint32_t bar = bars + 8u * s;
        const uint32_t dst = base + stage_bytes * s;
        mbar_expect_tx(bar, stage_bytes + p.tx_extra);
        for (int op = 0; op < p.k; ++op)
            bulk_g2s(dst + row_bytes * op, p.x + op * p.part_stride + m * p.H, row_bytes, bar);
        if (p.residual) bulk_g2s(dst + row_bytes * p.k, p.residual + m * p.H, row_bytes, bar);
    };

    // The first rows' inputs into L2 while the preceding grid drains (a
    // hint).  NVFP4, inlined: fp16 16384 x 8192 without residual 55.42 ->
    // 53.69 us, k = 4 partials 64.07 -> 62.43 us.  The FP8 family through
    // the helper, where it measured faster: bf16 FP8 16384 x 8192 without
    // residual 70.3 -> 63.0 us (4096 rows 21.6 -> 17.5), fp16 MXFP8 67.5 ->
    // 65.0; the fp16 FP8 instances keep their code (with the call compiled
    // in, 62.5 -> 63.2 us, and 65.1 with it skipped at run time).
    if constexpr (MODE != MODE_NVFP4 &&
                  (MODE == MODE_MXFP8 || std::is_same<T, __nv_bfloat16>::value)) {
        if (t == 0) stream_prefetch_rows(p, blockIdx.x, G, n_rows < S ? n_rows : S, row_bytes);
    }
    if (MODE == MODE_NVFP4 && t == 0) {
        for (int i = 0; i < n_rows && i < S; ++i) {
            const int64_t m = blockIdx.x + (int64_t)i * G;
            for (int op = 0; op < p.k; ++op) prefetch_l2_bulk(p.x + op * p.part_stride + m * p.H, row_bytes);
            if (p.residual) prefetch_l2_bulk(p.residual + m * p.H, row_bytes);
        }
    }
    pdl_wait();  // inputs may come from the preceding grid
    pdl_trigger();

    if (t == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bars + 8u * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int i = 0; i < n_rows && i < S; ++i) issue(i, i);
    }

    // per-CTA constants: the weight (packed if LEAN, else bias + w in fp32),
    // quantizer context
    int col[VPT];
    bool ok[VPT];
    uint4 wq[VPT][LEAN ? U : 1];
    float bw[VPT][LEAN || SW ? 1 : E];
    int sfc[VPT];
    int lc[VPT];  // the column a unit loads (PRED: clamped in range)
    const int nunits = p.H / E;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int u = v * NT + t;
        ok[v] = FULL || u < nunits;
        col[v] = u * E;
        lc[v] = PRED && !ok[v] ? 0 : col[v];
        sfc[v] = sf_col_offset(col[v]);
#pragma unroll
        for (int c = 0; c < U; ++c) {
            const uint4 w = (PRED || ok[v]) ? ld_weight(p.w + lc[v] + 8 * c) : make_uint4(0, 0, 0, 0);
            if constexpr (LEAN) {
                wq[v][c] = w;
            } else {
                float f[8];
                Act<T>::unpack(w, f);
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] = __fadd_rn(p.weight_bias, f[i]);
                if constexpr (SW) {  // read back only by this thread (lc: the loaded unit)
                    const int uu = lc[v] / E;
                    bw_s[(2 * c) * nunits + uu] = make_float4(f[0], f[1], f[2], f[3]);
                    bw_s[(2 * c + 1) * nunits + uu] = make_float4(f[4], f[5], f[6], f[7]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) bw[v][8 * c + i] = f[i];
                }
            }
        }
    }
    const uint32_t b16 = p.weight_bias == 1.f ? one16<T>() : 0u;  // LEAN: bias 1 or 0
    const QuantCtx qc = make_quant_ctx(p, MODE, es_smem, t, NT);

    __syncthreads();  // barriers initialised, table filled

    int s = 0;            // stage of row i (i mod S)
    uint32_t parity = 0;  // phase parity of that stage's barrier ((i / S) mod 2)
    for (int i = 0; i < n_rows; ++i) {
        const int64_t m = blockIdx.x + (int64_t)i * G;
        const int64_t row = m * (int64_t)p.H;
        const uint32_t stage = base + stage_bytes * s;

        const bool arrived = mbar_wait_bounded(bars + 8u * s, parity, p.wait_limit);
        // A copy never completed: record it, let the copies still in flight
        // land (bounded again) before the shared memory goes away.  Under the
        // test hook (tx_extra) the missing bytes are this kernel's own
        // announcement: one more valid copy per outstanding row completes
        // each barrier, so every copy has landed when the waits return.
        // MERGE writes nothing before the row barrier (the new residual
        // leaves after it, from the packed h), so the CTA agrees on the
        // arrival of the row's copies there instead.
        if constexpr (!MERGE) {
            if (__syncthreads_or(!arrived)) {
                if (t == 0) stream_drain(p, i, n_rows, s, S, parity, bars, topup);
                __syncthreads();
                return;
            }
        }

        // ---- a = sum of partials (fp32, index order), h = dtype(a + r) ----
        uint4 hb[VPT][LEAN ? U : 1];   // packed h (LEAN)
        float hf[VPT][LEAN ? 1 : E];   // h in fp32 (not LEAN)
        const uint4 zero = make_uint4(0, 0, 0, 0);
        float ss = 0.f;
        uint64_t ss2 = 0;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            float sv = 0.f;
            uint64_t sv2 = 0;
            float &acc_s = PRED ? sv : ss;
            uint64_t &acc_s2 = PRED ? sv2 : ss2;
            const bool ld = PRED || ok[v];
            uint4 hr[U];  // the new residual of the unit (V8: stored once, below)
#pragma unroll
            for (int c = 0; c < U; ++c) {
                const uint32_t off = (uint32_t)(lc[v] + 8 * c) * 2u;
                uint4 xv = ld ? lds_v4(stage + off) : zero;
                if (PARTS) {
                    float acc[8];
                    Act<T>::unpack(xv, acc);
                    for (int op = 1; op < p.k; ++op) {
                        float f[8];
                        Act<T>::unpack(ld ? lds_v4(stage + row_bytes * op + off) : zero, f);
#pragma unroll
                        for (int e = 0; e < 8; e += 2)
                            upk2(add2(pk2(acc[e], acc[e + 1]), pk2(f[e], f[e + 1])), acc[e], acc[e + 1]);
                    }
                    xv = pack8<T>(acc);
                }
                if (p.residual) {
                    xv = add16x8<T>(xv, ld ? lds_v4(stage + row_bytes * p.k + off) : zero);
                    if constexpr (MERGE) {
                        // stored after the row barrier
                    } else if constexpr (V8) {
                        hr[c] = xv;
                    } else {
                        st_v4_unit<PRED>(p.residual + row + col[v] + 8 * c, xv, ok[v]);
                    }
                }
                if constexpr (LEAN) {
                    hb[v][c] = xv;
                    acc_s = sumsq16x8<T>(xv, acc_s);
                } else {
                    float *hc = &hf[v][8 * c];
                    Act<T>::unpack(xv, hc);
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const uint64_t h2 = pk2(hc[e], hc[e + 1]);
                        acc_s2 = fma2(h2, h2, acc_s2);
                    }
                }
            }
            if constexpr (V8 && !MERGE) {
                if (p.residual) st_v8_unit<PRED>(p.residual + row + col[v], hr[0], hr[1], ok[v]);
            }
            if constexpr (PRED) {
                if constexpr (!LEAN) {
                    float a, b;
                    upk2(sv2, a, b);
                    sv = a + b;
                }
                ss += ok[v] ? sv : 0.f;
            }
        }
        if constexpr (!PRED && !LEAN) {
            float a, b;
            upk2(ss2, a, b);
            ss = a + b;
        }

        ss = warp_sum(ss);
        if ((t & 31) == 0) warp_ss[i & 1][t >> 5] = ss;
        // the row barrier: partial sums visible, every thread done reading
        // this stage (MERGE: and the copies' arrival agreed on)
        if constexpr (MERGE) {
            if (__syncthreads_or(!arrived)) {
                if (t == 0) stream_drain(p, i, n_rows, s, S, parity, bars, topup);
                __syncthreads();
                return;
            }
            if (p.residual) {  // the packed h is the new residual
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    if constexpr (V8) {
                        st_v8_unit<PRED>(p.residual + row + col[v], hb[v][0], hb[v][1], ok[v]);
                    } else {
#pragma unroll
                        for (int c = 0; c < U; ++c)
                            st_v4_unit<PRED>(p.residual + row + col[v] + 8 * c, hb[v][c], ok[v]);
                    }
                }
            }
        } else {
            __syncthreads();
        }
        if (t == 0 && i + S < n_rows) {
            fence_async_shared();
            issue(i + S, s);
        }
        float tot;
        if constexpr (MODE == MODE_NVFP4) tot = block_total_small(warp_ss[i & 1], NT >> 5, t & 31);
        else tot = block_total(warp_ss[i & 1], NT >> 5, t & 31);
        const float inv = inv_rms(p, tot);

        // y = RN(RN(h * w + bias * h) * inv): one mixed-precision FMA on the
        // packed h and w (exact product), then the scaling.
        const RowOut o = row_out<MODE>(p, m);
        auto finish = [&](auto path) {
            const uint64_t inv2 = pk2(inv, inv);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                float yf[E];
#pragma unroll
                for (int c = 0; c < U; ++c) {
                    float *a = &yf[8 * c];
                    if constexpr (LEAN) {
                        biasfma16x8<T>(hb[v][c], wq[v][c], b16, *reinterpret_cast<float(*)[8]>(a));
#pragma unroll
                        for (int e = 0; e < 8; e += 2)
                            upk2(mul2(pk2(a[e], a[e + 1]), inv2), a[e], a[e + 1]);
                    } else {
                        float b[8];
                        if constexpr (SW) {
                            const int uu = lc[v] / E;
                            const float4 b0 = bw_s[(2 * c) * nunits + uu];
                            const float4 b1 = bw_s[(2 * c + 1) * nunits + uu];
                            b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
                            b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) b[e] = bw[v][8 * c + e];
                        }
#pragma unroll
                        for (int e = 0; e < 8; e += 2)
                            upk2(mul2(mul2(pk2(hf[v][8 * c + e], hf[v][8 * c + e + 1]), inv2),
                                      pk2(b[e], b[e + 1])),
                                 a[e], a[e + 1]);
                    }
                }
                epilogue_unit<T, MODE, decltype(path)::value, PRED, V8>(p, qc, yf, o, col[v], sfc[v], ok[v], t);
            }
        };
        if (MODE == MODE_FP8 && !qc.fd.fast) finish(std::integral_constant<int, FP8_IEEE>{});
        else finish(std::integral_constant<int, FP8_PAIR>{});
        if (++s == S) {
            s = 0;
            parity ^= 1u;
        }
    }
}

#define GNQ_STREAM_SMEM                                     \
    extern __shared__ __align__(128) uint8_t dsmem[];       \
    __shared__ __align__(16) float warp_ss[2][32];          \
    __shared__ float es_smem[MODE == MODE_NVFP4 ? 256 : 1]; \
    __shared__ __align__(16) uint4 topup[4];

// FP8, MXFP8 and no-quant streaming: the compiler's own register choice.
template <typename T, int MODE, bool PARTS, int VPT, bool LEAN, bool FULL, int OPT>
__global__ void __launch_bounds__(VPT == 1 ? 1024 : 512) stream_kernel(const __grid_constant__ Params p) {
    GNQ_STREAM_SMEM
    stream_body<T, MODE, PARTS, VPT, LEAN, FULL, OPT>(p, dsmem, warp_ss, es_smem, topup);
}

// NVFP4 streaming: the StreamForm register budget.
template <typename T, int MODE, bool PARTS, int VPT, bool LEAN, bool FULL, int OPT>
__global__ void __launch_bounds__(VPT == 1 ? 1024 : 512) __maxnreg__((StreamForm<MODE, VPT, LEAN>::maxnreg))
    stream_kernel_nvfp4(const __grid_constant__ Params p) {
    static_assert(MODE == MODE_NVFP4, "NVFP4 streaming only");
    GNQ_STREAM_SMEM
    stream_body<T, MODE, PARTS, VPT, LEAN, FULL, OPT>(p, dsmem, warp_ss, es_smem, topup);
}
#undef GNQ_STREAM_SMEM

}  // namespace gnq
