/*
 * CPU oracle for the fused Gemma add-RMSNorm + FP8 / NVFP4 input quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously correct
 * restatement of what the method computes, used by the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark.  The product path (the CUDA
 * library) never links, loads or calls it, and it shares no code with it.
 *
 * Sources (the pages are the vLLM documentation and PR text this project is
 * built from):
 *   - "vllm.models.qwen3_5.nvidia.ops.fused_norm_quant", module docstring and
 *     gemma_add_rms_norm_quant (arguments, returns, asserts, allocation);
 *   - same page, _cvt_e2m1x2 (E2M1 packing: low element in the low nibble);
 *   - "vllm.models.qwen3_5.nvidia.ops.fused_allreduce_norm_quant",
 *     fused_allreduce_gemma_rms_norm_quant (fp32 accumulation of the
 *     per-rank partials, 128x4 swizzled scale layout, weight bias 1);
 *   - "vllm.model_executor.layers.fused_allreduce_gemma_rms_norm",
 *     allreduce_gemma_rms_norm_mxfp8 (MXFP8 output: e4m3 values and
 *     row-major E8M0 scales per 32 elements).
 *
 * Bit patterns: 16-bit activations (bf16 or fp16) travel as uint16_t, FP8
 * E4M3 codes, packed E2M1 bytes, E4M3 block scales and E8M0 scales as uint8_t.
 */
#ifndef GNQ_ORACLE_H
#define GNQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OR_BF16 0
#define OR_FP16 1

#define OR_MODE_NONE  (-1) /* add + Gemma RMSNorm only: y is the output        */
#define OR_MODE_FP8     0  /* static per-tensor FP8 E4M3                        */
#define OR_MODE_NVFP4   1  /* E2M1 codes + E4M3 block scales, 128x4 swizzled    */
#define OR_MODE_MXFP8   2  /* E4M3 codes + E8M0 scales per 32, row-major        */

/* --- number formats ---------------------------------------------------- */
double   or_decode16(uint16_t bits, int dtype);
uint16_t or_round16(double v, int dtype);
double   or_e4m3_value(uint8_t code);
uint8_t  or_e4m3_encode(double v);
double   or_e2m1_value(uint8_t code);
uint8_t  or_e2m1_encode(double v);
double   or_e8m0_value(uint8_t code);

/* element-wise array forms of the four routines above (test helpers) */
void or_decode16_array(const uint16_t *bits, double *out, int64_t n, int dtype);
void or_round16_array(const double *v, uint16_t *out, int64_t n, int dtype);
void or_e4m3_encode_array(const double *v, uint8_t *out, int64_t n);
void or_e2m1_encode_array(const double *v, uint8_t *out, int64_t n);

/* --- layout ------------------------------------------------------------- */
int64_t  or_swizzle_offset(int64_t m, int64_t k, int64_t Kp);

/* --- the method ---------------------------------------------------------- */
/*
 * Full pipeline over M rows of H elements.
 *   x         : k partial buffers of (M, H) 16-bit values, part_stride
 *               elements apart (k = 1: the activation itself).  Read only.
 *   residual  : (M, H) or NULL.  Updated in place to the summed input h.
 *   w         : (H,) Gemma weight; the norm multiplies by (1 + w).
 *   weight_bias: 1.0 for the Gemma norm, 0.0 for a plain RMSNorm.
 *   scale     : FP8 static scale s, or the NVFP4 global scale g.
 *   mode      : OR_MODE_*.
 *   q         : FP8/MXFP8 (M, H) bytes; NVFP4 (M, H/2) packed bytes.
 *   block_scale: NVFP4 (round_up(M,128) * round_up(H/16,4)) bytes, swizzled;
 *               MXFP8 (M, H/32) bytes, row-major.  Rows >= M not touched.
 *   y         : (M, H) normed activation, or NULL (it is still rounded to
 *               the activation dtype internally before quantization).
 * Returns 0, or -1 on an argument it does not accept.
 */
int or_gemma_add_rms_norm_quant(const uint16_t *x, int k, int64_t part_stride,
                                uint16_t *residual, const uint16_t *w,
                                float eps, float weight_bias, float scale,
                                int mode, uint8_t *q, uint8_t *block_scale,
                                uint16_t *y, int64_t M, int64_t H, int dtype);

/* Quantization stage alone, applied to a given y (for example one produced
 * by another implementation), so that codes can be compared bit for bit. */
int or_quantize_from_y(const uint16_t *y, float scale, int mode, uint8_t *q,
                       uint8_t *block_scale, int64_t M, int64_t H, int dtype);

/* Number of host threads the row loop may use (1 = serial).  Rows are
 * independent, so the result does not depend on it. */
void or_set_threads(int n);
int  or_get_threads(void);

#ifdef __cplusplus
}
#endif
#endif
