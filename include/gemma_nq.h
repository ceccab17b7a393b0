/*
 * gemma_nq -- fused residual add + Gemma RMSNorm + next-linear input
 * quantization on one GB300 (sm_103a), as a C ABI.
 *
 * The operation ("vllm.models.qwen3_5.nvidia.ops.fused_norm_quant", module
 * docstring and gemma_add_rms_norm_quant):
 *
 *     h  = x + residual                 (rounded to the activation dtype;
 *                                        written back into `residual`)
 *     y  = dtype(h * rsqrt(mean(h^2) + eps) * (1 + w))
 *     q  = quant(y)                     (computed from the rounded y)
 *
 * with quant one of
 *   GNQ_FP8   static per-tensor FP8 E4M3: q = e4m3_satfinite(y / scale);
 *   GNQ_NVFP4 per 16-element block: E4M3 block scale
 *             sf = e4m3_satfinite(g * (amax / 6)), codes
 *             e2m1_satfinite(y * (g / sf)) packed two per byte, the
 *             lower-indexed element in the low nibble; block scales in the
 *             128x4 swizzled layout of shape (round_up(M,128),
 *             round_up(H/16,4)), byte (m, b) at
 *             ((m/128)*(Kp/4) + b/4)*512 + (m%32)*16 + ((m%128)/32)*4 + b%4;
 *   GNQ_MXFP8 per 32-element block ("vllm.model_executor.layers.
 *             fused_allreduce_gemma_rms_norm", allreduce_gemma_rms_norm_mxfp8):
 *             E8M0 scale code floor(log2(amax)) - 8 + 127 clamped to
 *             [0, 254] (0 for an all-zero block), stored row-major (M, H/32);
 *             codes e4m3_satfinite(y / 2^(code - 127)).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are addresses the current CUDA device can access,
 *    in row-major contiguous layout: device memory, or pinned host memory
 *    (mapped into the device's address space; on a Grace-Blackwell node the
 *    kernels then read and write it over NVLink-C2C, with no separate copy).
 *    A call whose activations are not in device memory always runs one CTA
 *    per row (plain loads and stores), never the streaming kernel, whose
 *    bulk copies read device memory.  Activations x, residual, y and the weight
 *    w are 16-bit, of the type named by `dtype` (GNQ_BF16 or GNQ_FP16).
 *  - The caller owns and allocates every buffer.  The library allocates
 *    nothing per call and keeps no state other than cached device properties.
 *  - x, w, scale and the partial buffers are read only.  `residual` (when not
 *    NULL) is updated in place to the rounded x + residual.  q, block_scale
 *    and y are written.  Rows m >= M of the NVFP4 scale tensor are NOT
 *    written (their bytes keep whatever the caller put there).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Nothing is synchronised and no host copy is made.
 *  - M == 0 returns GNQ_OK without launching anything.
 *  - Every call returns a gnq_status; the library never aborts, exits or
 *    traps.  Argument checks happen before any launch; a rejected call has
 *    no effect.
 *  - Alignment: x, residual, w, y, q and every partial buffer must be 16-byte
 *    aligned, block_scale 4-byte aligned, scale 4-byte aligned
 *    (GNQ_ERR_ALIGN).  NVFP4 calls whose 16-bit tensors (and partial
 *    stride) are also 32-byte aligned, as every allocator's tensors are,
 *    move each 16-element block in one 256-bit access; others run one CTA
 *    per row with 128-bit accesses.  H must be a multiple of 8 (GNQ_ERR_SHAPE); NVFP4 needs
 *    H % 64 == 0 (whole 4-column scale tiles, so padded scale columns never
 *    exist) and MXFP8 H % 32 == 0.  H is at most 65536.
 *  - x and residual must not be the same buffer, and y must differ from both
 *    (GNQ_ERR_ALIAS).
 *  - Every buffer must hold at least the elements its shape below states;
 *    the library receives raw pointers and cannot check sizes (the Python
 *    binding does, before any launch).
 */
#ifndef GEMMA_NQ_H
#define GEMMA_NQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GNQ_OK = 0,
    GNQ_ERR_NULL = 1,  /* a required pointer is NULL                        */
    GNQ_ERR_SHAPE = 2, /* M < 0, H out of range or not a supported multiple */
    GNQ_ERR_DTYPE = 3, /* dtype is not GNQ_BF16 / GNQ_FP16                  */
    GNQ_ERR_MODE = 4,  /* unknown quantization mode, or k out of range      */
    GNQ_ERR_ALIAS = 5, /* x == residual, or y aliases x or residual         */
    GNQ_ERR_ALIGN = 6, /* a pointer or the partial stride is misaligned     */
    GNQ_ERR_CUDA = 7   /* the CUDA runtime reported an error at launch (the
                          runtime's last-error state is cleared, so the
                          caller's own later checks do not see it)         */
} gnq_status;

typedef enum { GNQ_BF16 = 0, GNQ_FP16 = 1 } gnq_dtype;

typedef enum { GNQ_FP8 = 0, GNQ_NVFP4 = 1, GNQ_MXFP8 = 2 } gnq_mode;

/*
 * Residual add + Gemma RMSNorm, no quantization
 * ("vllm.model_executor.layers.fused_allreduce_gemma_rms_norm",
 * fused_allreduce_gemma_rms_norm: at tensor-parallel size 1 it is
 * norm(hidden_states, residual), returning (normed, new residual)).
 *
 *   x        (M, H) activation, read only.
 *   residual (M, H) or NULL; updated in place to dtype(x + residual).
 *   w        (H,) Gemma weight; the norm multiplies by (1 + w).
 *   eps      RMSNorm epsilon.
 *   y        (M, H) output, y = dtype(h * rsqrt(mean(h^2) + eps) * (1 + w)).
 */
int gemma_add_rms_norm(const void *x, void *residual, const void *w, float eps,
                       void *y, int64_t M, int64_t H, int dtype, void *stream);

/*
 * Residual add + Gemma RMSNorm + the next linear's input quantization, in one
 * pass ("vllm.models.qwen3_5.nvidia.ops.fused_norm_quant",
 * gemma_add_rms_norm_quant).
 *
 *   x, residual, w, eps   as for gemma_add_rms_norm.
 *   scale        device pointer to ONE fp32: the static FP8 scale s, or the
 *                NVFP4 global scale g (input_global_scale_inv).  Read on the
 *                device, so it may change between graph replays.  Unused
 *                (may be NULL) for GNQ_MXFP8.
 *   mode         GNQ_FP8, GNQ_NVFP4 or GNQ_MXFP8.
 *   write_y      nonzero: also store the normed activation y (M, H).
 *   q            FP8 / MXFP8: (M, H) E4M3 codes.  NVFP4: (M, H/2) bytes of
 *                packed E2M1 codes.
 *   block_scale  NVFP4: the swizzled (round_up(M,128), round_up(H/16,4))
 *                E4M3 scale bytes.  MXFP8: (M, H/32) E8M0 codes.  Unused
 *                (may be NULL) for GNQ_FP8, whose block scale is `scale`.
 *   y            (M, H) if write_y, else ignored (may be NULL).
 */
int gemma_add_rms_norm_quant(const void *x, void *residual, const void *w,
                             float eps, const float *scale, int mode,
                             int write_y, void *q, void *block_scale, void *y,
                             int64_t M, int64_t H, int dtype, void *stream);

/*
 * As gemma_add_rms_norm_quant, with the activation given as k partial
 * buffers, the per-rank partial outputs of a row-parallel linear that a
 * tensor-parallel all-reduce would sum ("vllm.models.qwen3_5.nvidia.ops.
 * fused_allreduce_norm_quant", fused_allreduce_gemma_rms_norm_quant:
 * hidden_states is the per-rank partial, reduced with fp32 accumulation).
 * Here the k partials sit in this GPU's memory and are summed locally:
 * a = dtype(((p0 + p1) + p2) + ...) in fp32, then h = dtype(a + residual).
 *
 *   x_parts      base of k (M, H) buffers; partial p starts at
 *                x_parts + p * part_stride ELEMENTS (part_stride >= M*H and a
 *                multiple of 8, so every partial is 16-byte aligned).
 *   k            number of partials, 1..8 (GNQ_ERR_MODE otherwise).
 *   mode         as above, or -1 for no quantization (then write_y must be
 *                nonzero and q / block_scale / scale are ignored).
 */
int gemma_add_rms_norm_quant_parts(const void *x_parts, int k,
                                   int64_t part_stride, void *residual,
                                   const void *w, float eps,
                                   const float *scale, int mode, int write_y,
                                   void *q, void *block_scale, void *y,
                                   int64_t M, int64_t H, int dtype,
                                   void *stream);

/*
 * Plain (non-Gemma) RMSNorm variant: y = dtype(h * rsqrt(mean(h^2) + eps) * w),
 * i.e. weight bias 0 instead of 1 ("vllm.models.qwen3_5.nvidia.ops.
 * fused_allreduce_norm_quant" passes the weight bias to the fused kernel;
 * weight_bias=1.0 marks the Gemma form on
 * "vllm.model_executor.layers.fused_allreduce_gemma_rms_norm").  Arguments
 * as for gemma_add_rms_norm_quant_parts; k = 1 for a single activation.
 */
int add_rms_norm_quant(const void *x_parts, int k, int64_t part_stride,
                       void *residual, const void *w, float eps,
                       const float *scale, int mode, int write_y, void *q,
                       void *block_scale, void *y, int64_t M, int64_t H,
                       int dtype, void *stream);

/* Human-readable text of a gnq_status (static storage, never NULL). */
const char *gnq_status_string(int status);

/*
 * Tuning hook: force the launch shape of later calls in this process.
 *   kernel   0 = automatic; 1 = one CTA (or cluster) per row; 2 = persistent
 *            streaming kernel (rows staged through shared memory).
 *   cluster  row kernel: 0 = automatic, else 1, 2, 4 or 8 CTAs per row.
 *            Streaming kernel: 0 = automatic grid, else at least that many
 *            rows (2, 4 or 8) per CTA (grid = ceil(M / cluster) CTAs when
 *            that is below one wave).
 *   vpt      0 = automatic, else 1, 2 or 4 units (8 elements; 16 for
 *            NVFP4) per thread.
 *   form     0 = automatic; 1 = h and the weight unpacked to fp32 (fewest
 *            instructions); 2 = kept packed (fewest registers; Gemma or plain
 *            weight bias only).
 * A forced shape that does not fit a call (H, mode, shared memory) falls back
 * to the automatic one for that call.  The shape only changes the order in
 * which a row's squares are summed (so y may move by one rounding step); the
 * residual, and the codes of a given y, never depend on it.  Not
 * synchronised with calls in flight on other host threads.  Returns
 * GNQ_ERR_SHAPE for values outside those sets.
 */
int gnq_set_launch_policy(int kernel, int cluster, int vpt, int form);

/*
 * The launch shape the automatic policy picks for a call on the current
 * device with its activations in device memory, in the terms of
 * gnq_set_launch_policy (a forced policy is not applied): *kernel 1 or 2, *cluster CTAs per row (0 for the streaming
 * kernel), *vpt 1, 2 or 4, *form 1 (fp32) or 2 (packed).  The arguments
 * describe the call: rows M >= 1, width H, k partial buffers (1: one
 * activation), whether it has a residual and writes y, mode, dtype, and the
 * weight bias (1 Gemma, 0 plain).  Forcing the returned shape reproduces
 * the automatic launch, for instance to run a call that writes y with
 * exactly the arithmetic of one that does not.  Returns GNQ_OK;
 * GNQ_ERR_NULL, GNQ_ERR_DTYPE, GNQ_ERR_MODE or GNQ_ERR_SHAPE for arguments a
 * call would reject; GNQ_ERR_CUDA without a usable device.
 */
int gnq_query_launch(int64_t M, int64_t H, int k, int has_residual, int write_y, int mode,
                     int dtype, float weight_bias, int *kernel, int *cluster, int *vpt,
                     int *form);

/*
 * Programmatic dependent launch (on by default): each launch may start while
 * the preceding kernel on the stream drains, and waits inside the kernel
 * (griddepcontrol.wait) until that kernel's results are visible before its
 * first global read of them.  Before the wait, the CTAs that can be waiting
 * (the first wave of a one-CTA-per-row launch; streaming CTAs, for their
 * first rows, in the NVFP4, MXFP8 and bf16 instances) prefetch their rows
 * of x, the partials and the residual
 * into L2: a cache hint, not a read (the values used are loaded after the
 * wait, and L2 is where the preceding kernel's stores land), so the
 * buffers must be valid device-accessible memory at launch, as for any
 * call.  Right after the wait the kernel also lets a programmatic
 * dependent that follows it launch (that kernel must wait in the same way
 * before reading these outputs), so the dependent's CTAs can take the SMs
 * this grid leaves idle and run their own prologue early.  Results are
 * identical either way.  enable = 0 turns it off for later calls in this
 * process, 1 turns it on.  Not synchronised with calls in flight on other
 * host threads.
 */
int gnq_set_pdl(int enable);

/*
 * Constant weights (off by default).  With enable = 1, later small-batch
 * calls (those the policy runs one 16-byte unit -- NVFP4: one 16-element
 * block -- per thread on the one-CTA-per-row kernel, i.e. batches below about
 * one row per SM, with one activation rather than partials) read the norm
 * weight w and the quantization scale, and build their quantizer constants,
 * before they wait for the preceding kernel on their stream (programmatic
 * dependent launch), so that work overlaps its tail; other calls ignore the
 * flag.  The caller guarantees that no kernel that precedes a call on its
 * stream, and may still be running, writes w or scale (true when they are
 * model constants).  x, the partials and the residual are always read after
 * the wait.  Results are identical either way.  enable = 0 restores the
 * default.  Not synchronised with calls in flight on other host threads.
 * Returns GNQ_ERR_SHAPE for other values.
 */
int gnq_set_constant_weights(int enable);

/*
 * Test hook for the failure path of the bounded waits (off by default).
 * With enable = 1, later launches of the persistent streaming kernel in this
 * process announce 16 bytes more per row than their copies deliver and give
 * a wait at most ~2^20 clock cycles, so each CTA's wait for its first row
 * gives up: the kernel sets bit 1 of the device error word, completes each
 * outstanding barrier with one more valid 16-byte copy (from w into its own
 * shared memory, so every copy has landed before it returns), and returns
 * without writing any output.  Nothing outside the call's own buffers is
 * touched; the row kernel is unaffected.  enable = 0 restores normal
 * launches.  Not synchronised with calls in flight on other host threads.
 * Returns GNQ_ERR_SHAPE for other values.
 */
int gnq_inject_wait_timeout(int enable);

/*
 * Device error word of the current device.  Every wait inside a kernel is
 * bounded; a kernel whose wait gives up (about a second without progress)
 * skips the rest of its work, sets bit 1 here and returns, leaving its
 * outputs incomplete.  Copies the word into *flags (synchronising the device)
 * and clears it when `clear` is nonzero.
 */
int gnq_read_device_error(unsigned int *flags, int clear);

/*
 * Diagnostic: a stand-in for the first kernel of the next linear layer, to
 * measure programmatic dependent launch with a real consumer.  Launched as a
 * programmatic dependent of the preceding kernel on `stream`, with `ctas`
 * CTAs of 256 threads: each CTA first reads its share of the wt_bytes at
 * `wt` (an independent buffer, standing for the layer's weight), then waits
 * for the preceding kernel's results (griddepcontrol.wait), then reads its
 * share of the q_bytes at `q` (that kernel's codes), and stores one checksum
 * word per thread to `out` (ctas * 256 words).  Byte counts are multiples of
 * 16 and the pointers 16-byte aligned device memory.  Returns GNQ_ERR_SHAPE,
 * GNQ_ERR_NULL or GNQ_ERR_CUDA on bad arguments or a failed launch.
 */
int gnq_pdl_consumer(const void *q, int64_t q_bytes, const void *wt, int64_t wt_bytes,
                     unsigned int *out, int ctas, void *stream);

/*
 * Diagnostic: the static-FP8 quantizer the kernels use, applied to n fp32
 * values y (device pointer): q[i] = e4m3_satfinite(y[i] / *scale), with
 * `scale` a device pointer to one fp32.  Values go through it in groups of
 * eight on the path the kernels take (paired arithmetic after the magnitude
 * clamp applied to bf16 y, or IEEE division for extreme scales).
 * Lets a test sweep every 16-bit y value against an independent encoder.
 */
int gnq_quantize_fp8_values(const float *y, int64_t n, const float *scale, uint8_t *q,
                            void *stream);

/*
 * Diagnostic: the element encoders the kernels use, applied to n fp32 values
 * v (device pointer): e4m3[i] = the E4M3 satfinite round-to-nearest-even code
 * of v[i], e2m1[i] = the E2M1 satfinite round-to-nearest-even code (low
 * nibble).  Either output may be NULL.  Lets a test compare the hardware
 * conversions with an independent encoder on special values (ties, zero
 * signs, subnormals, saturation).
 */
int gnq_encode_e4m3_e2m1(const float *v, int64_t n, uint8_t *e4m3,
                         uint8_t *e2m1, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* GEMMA_NQ_H */
