/* Plain-C use of the gemma_nq C ABI (no Python, no torch): device buffers
 * from the CUDA runtime, one FP8 call, one NVFP4 call, status checks.
 *
 * Expected values are hand-worked from the method's definition
 * ("vllm.models.qwen3_5.nvidia.ops.fused_norm_quant",
 * gemma_add_rms_norm_quant):
 *   x = 1 (bf16), residual = 2, w = 0, eps = 1e-6, H = 64:
 *   h = 3 (bf16 0x4040) written back; y = dtype(3 / sqrt(9 + 1e-6)) = 1.0;
 *   FP8 with s = 0.02: 1 / 0.02 = 50, the E4M3 tie 48 | 52 -> 48 = 0x64.
 *   NVFP4 with g = 168: every block amax 1 -> g * (1 / 6) = 28 -> E4M3 28
 *   (0x5E); element scale 168 / 28 = 6 -> 1 * 6 = 6 -> E2M1 code 7, so
 *   every byte is 0x77.
 * Exit status 0 on success. */
#include <stdio.h>
#include <stdint.h>
#include <string.h>
#include <cuda_runtime_api.h>

#include "gemma_nq.h"

#define H 64
#define M 3

static int fail(const char *what) {
    fprintf(stderr, "FAIL: %s\n", what);
    return 1;
}

int main(void) {
    uint16_t hx[M * H], hr[M * H], hw[H];
    for (int i = 0; i < M * H; ++i) { hx[i] = 0x3F80; hr[i] = 0x4000; } /* 1.0, 2.0 */
    for (int i = 0; i < H; ++i) hw[i] = 0;
    float s_fp8 = 0.02f, g = 168.0f;

    void *x, *r, *w, *y, *q, *bs;
    float *s;
    if (cudaMalloc(&x, sizeof hx) || cudaMalloc(&r, sizeof hr) || cudaMalloc(&w, sizeof hw) ||
        cudaMalloc(&y, sizeof hx) || cudaMalloc(&q, M * H) || cudaMalloc(&bs, 128 * (H / 16)) ||
        cudaMalloc((void **)&s, 2 * sizeof(float)))
        return fail("cudaMalloc");
    cudaMemcpy(x, hx, sizeof hx, cudaMemcpyHostToDevice);
    cudaMemcpy(r, hr, sizeof hr, cudaMemcpyHostToDevice);
    cudaMemcpy(w, hw, sizeof hw, cudaMemcpyHostToDevice);
    cudaMemcpy(s, &s_fp8, sizeof(float), cudaMemcpyHostToDevice);
    cudaMemcpy(s + 1, &g, sizeof(float), cudaMemcpyHostToDevice);

    /* FP8 with y */
    int st = gemma_add_rms_norm_quant(x, r, w, 1e-6f, s, GNQ_FP8, 1, q, NULL, y, M, H, GNQ_BF16, NULL);
    if (st != GNQ_OK) return fail(gnq_status_string(st));
    if (cudaDeviceSynchronize() != cudaSuccess) return fail("sync");
    uint16_t out_r[M * H], out_y[M * H];
    uint8_t out_q[M * H];
    cudaMemcpy(out_r, r, sizeof out_r, cudaMemcpyDeviceToHost);
    cudaMemcpy(out_y, y, sizeof out_y, cudaMemcpyDeviceToHost);
    cudaMemcpy(out_q, q, sizeof out_q, cudaMemcpyDeviceToHost);
    for (int i = 0; i < M * H; ++i) {
        if (out_r[i] != 0x4040) return fail("residual != 3.0");
        if (out_y[i] != 0x3F80) return fail("y != 1.0");
        if (out_q[i] != 0x64) return fail("fp8 code != 0x64");
    }

    /* NVFP4, residual absent (x = 1 everywhere) */
    cudaMemset(bs, 0xA5, 128 * (H / 16));
    st = gemma_add_rms_norm_quant(x, NULL, w, 1e-6f, s + 1, GNQ_NVFP4, 0, q, bs, NULL, M, H,
                                  GNQ_BF16, NULL);
    if (st != GNQ_OK) return fail(gnq_status_string(st));
    if (cudaDeviceSynchronize() != cudaSuccess) return fail("sync");
    uint8_t out_bs[128 * (H / 16)];
    cudaMemcpy(out_q, q, M * H / 2, cudaMemcpyDeviceToHost);
    cudaMemcpy(out_bs, bs, sizeof out_bs, cudaMemcpyDeviceToHost);
    for (int i = 0; i < M * H / 2; ++i)
        if (out_q[i] != 0x77) return fail("nvfp4 byte != 0x77");
    for (int m = 0; m < 128; ++m)
        for (int b = 0; b < H / 16; ++b) {
            const int off = (m % 32) * 16 + ((m % 128) / 32) * 4 + b; /* one 128x4 tile */
            const uint8_t want = m < M ? 0x5E : 0xA5;
            if (out_bs[off] != want) return fail("nvfp4 scale byte / padding");
        }

    /* rejected calls: statuses, no effect */
    if (gemma_add_rms_norm_quant(x, x, w, 1e-6f, s, GNQ_FP8, 0, q, NULL, NULL, M, H, GNQ_BF16, NULL) != GNQ_ERR_ALIAS)
        return fail("alias status");
    if (gemma_add_rms_norm_quant(x, r, w, 1e-6f, s, GNQ_NVFP4, 0, q, bs, NULL, M, 96, GNQ_BF16, NULL) != GNQ_ERR_SHAPE)
        return fail("shape status");
    if (gemma_add_rms_norm_quant(x, r, w, 1e-6f, s, GNQ_FP8, 0, q, NULL, NULL, 0, H, GNQ_BF16, NULL) != GNQ_OK)
        return fail("empty batch");
    unsigned int flags = 1;
    if (gnq_read_device_error(&flags, 1) != GNQ_OK || flags != 0) return fail("device error word");

    /* the automatic launch shape, and forcing it reproduces the same bits */
    int kernel = 0, cluster = -1, vpt = 0, form = 0;
    if (gnq_query_launch(M, H, 1, 1, 1, GNQ_FP8, GNQ_BF16, 1.0f, &kernel, &cluster, &vpt, &form) !=
        GNQ_OK)
        return fail("query launch");
    if (kernel != 1 || vpt < 1 || vpt > 4 || (form != 1 && form != 2))
        return fail("query launch values");  /* three rows: one CTA per row */
    if (gnq_query_launch(M, H, 1, 1, 1, GNQ_FP8, GNQ_BF16, 1.0f, NULL, &cluster, &vpt, &form) !=
        GNQ_ERR_NULL)
        return fail("query launch NULL status");
    cudaMemcpy(r, hr, sizeof hr, cudaMemcpyHostToDevice);
    if (gnq_set_launch_policy(kernel, cluster, vpt, form) != GNQ_OK) return fail("set policy");
    st = gemma_add_rms_norm_quant(x, r, w, 1e-6f, s, GNQ_FP8, 1, q, NULL, y, M, H, GNQ_BF16, NULL);
    gnq_set_launch_policy(0, 0, 0, 0);
    if (st != GNQ_OK) return fail(gnq_status_string(st));
    if (cudaDeviceSynchronize() != cudaSuccess) return fail("sync");
    cudaMemcpy(out_q, q, sizeof out_q, cudaMemcpyDeviceToHost);
    for (int i = 0; i < M * H; ++i)
        if (out_q[i] != 0x64) return fail("forced shape: fp8 code != 0x64");
    if (strlen(gnq_status_string(GNQ_ERR_ALIGN)) == 0) return fail("status string");
    printf("c abi ok\n");
    return 0;
}
