"""Seeded synthetic workloads for the fused add + Gemma RMSNorm + quant op.

This module holds only input generation: shapes, distributions and seeds.  It
contains none of the method's arithmetic, so the tests can feed the same
inputs to the CUDA library and to the CPU oracle.

Recipe (one torch CPU generator per workload, seeded with ``seed``; draws are
fp32 normals scaled by the standard deviation, then rounded to the activation
dtype; draw order: partials, x, residual, weight):

* ``N(0, v)`` in a workload description is a normal of VARIANCE v.
* Outlier channels: ``randperm(H)[:n_outliers]`` from a second generator
  seeded ``1000 + seed``; those residual columns are multiplied by 20 before
  rounding.
* With ``k > 1`` the activation is k partial buffers (the per-rank partials of
  a row-parallel linear that a tensor-parallel all-reduce would sum) and there
  is no separate x draw.
"""
from __future__ import annotations

import dataclasses
import math

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    H: int
    dtype: str          # "bf16" | "fp16"
    mode: str           # "fp8" | "nvfp4" | "mxfp8" | "none"
    scale: float        # FP8 static scale, or NVFP4 global scale (unused otherwise)
    write_y: bool
    residual: bool
    seed: int
    k: int = 1          # number of partial buffers
    x_var: float = 1.0
    r_var: float = 1.0
    w_var: float = 0.1
    part_var: float = 0.25
    n_outliers: int = 0
    outlier_mult: float = 20.0
    eps: float = 1e-6
    weight_bias: float = 1.0  # 1: Gemma norm (1 + w); 0: plain RMSNorm (w)

    def with_rows(self, M: int) -> "Workload":
        return dataclasses.replace(self, M=M)

    def algorithmic_bytes(self) -> int:
        """HBM bytes one call must move: inputs read once, outputs written
        once, the weight read once; scale padding is never written."""
        e = 2
        M, H = self.M, self.H
        b = self.k * e * M * H + e * H
        if self.residual:
            b += 2 * e * M * H
        if self.write_y or self.mode == "none":
            b += e * M * H
        if self.mode in ("fp8", "mxfp8"):
            b += M * H
        if self.mode == "mxfp8":
            b += M * (H // 32)
        if self.mode == "nvfp4":
            b += M * (H // 2) + M * (H // 16)
        return b


# The five workload configurations of the method's decode, prefill and
# tensor-parallel-partial shapes (config 4 has four variants).
WORKLOADS = {
    w.name: w for w in [
        Workload("decode_m16_h2048_bf16_fp8", 16, 2048, "bf16", "fp8", 0.02,
                 write_y=False, residual=True, seed=0, r_var=4.0),
        Workload("decode_m256_h4096_bf16_fp8_y", 256, 4096, "bf16", "fp8", 0.05,
                 write_y=True, residual=True, seed=1, r_var=9.0, n_outliers=8),
        Workload("prefill_m2048_h5120_bf16_nvfp4_y", 2048, 5120, "bf16", "nvfp4", 168.0,
                 write_y=True, residual=True, seed=2, r_var=9.0, n_outliers=8),
        Workload("prefill_m16384_h8192_fp16_fp8", 16384, 8192, "fp16", "fp8", 0.08,
                 write_y=False, residual=True, seed=3, r_var=16.0),
        Workload("prefill_m16384_h8192_fp16_nvfp4", 16384, 8192, "fp16", "nvfp4", 84.0,
                 write_y=False, residual=True, seed=3, r_var=16.0),
        Workload("prefill_m16384_h8192_fp16_fp8_nores", 16384, 8192, "fp16", "fp8", 0.08,
                 write_y=False, residual=False, seed=3, r_var=16.0),
        Workload("prefill_m16384_h8192_fp16_nvfp4_nores", 16384, 8192, "fp16", "nvfp4", 84.0,
                 write_y=False, residual=False, seed=3, r_var=16.0),
        Workload("parts4_m4096_h7168_bf16_nvfp4_y", 4096, 7168, "bf16", "nvfp4", 112.0,
                 write_y=True, residual=True, seed=4, k=4, r_var=9.0),
    ]
}

# The method's further variants at the same shapes: the MXFP8 output (E4M3
# values + one E8M0 scale per 32 elements, row-major), the plain RMSNorm
# (weight bias 0) and the norm alone (y, no quantization).
EXTRA_WORKLOADS = {
    w.name: w for w in [
        Workload("decode_m256_h4096_bf16_mxfp8_y", 256, 4096, "bf16", "mxfp8", 0.0,
                 write_y=True, residual=True, seed=1, r_var=9.0, n_outliers=8),
        Workload("prefill_m16384_h8192_fp16_mxfp8", 16384, 8192, "fp16", "mxfp8", 0.0,
                 write_y=False, residual=True, seed=3, r_var=16.0),
        Workload("prefill_m16384_h8192_fp16_nvfp4_plain", 16384, 8192, "fp16", "nvfp4", 84.0,
                 write_y=False, residual=True, seed=3, r_var=16.0, weight_bias=0.0),
        Workload("prefill_m16384_h8192_fp16_norm_y", 16384, 8192, "fp16", "none", 0.0,
                 write_y=True, residual=True, seed=3, r_var=16.0),
    ]
}

# The batch the headline throughput is quoted on: the largest configuration
# (prefill, 16384 x 8192 fp16, static FP8 with an in-place residual; 939.5 MB
# per call).
HEADLINE = "prefill_m16384_h8192_fp16_fp8"

# The small-batch sweep: batch sizes M = 1 .. 8192 at H = 5120 (bf16, the
# M = 2048 configuration's distributions), in both the static-FP8 and the
# NVFP4 mode, as the launch-heuristic sweep of "vllm.models.qwen3_5.nvidia.
# ops.fused_norm_quant" (gemma_add_rms_norm_quant) was taken.  129 and 192
# are the batch sizes that sweep singles out.
SMALL_M = (1, 2, 4, 8, 16, 32, 64, 96, 128, 129, 152, 192, 256, 384, 512, 1024, 2048, 4096, 8192)
SWEEP_BASES = {
    "nvfp4": "prefill_m2048_h5120_bf16_nvfp4_y",
    "fp8": "sweep_h5120_bf16_fp8_y",
}


# Shapes used only as the base of the small-batch sweep (not bench lines).
SWEEP_WORKLOADS = {
    w.name: w for w in [
        Workload("sweep_h5120_bf16_fp8_y", 2048, 5120, "bf16", "fp8", 0.05,
                 write_y=True, residual=True, seed=2, r_var=9.0, n_outliers=8),
    ]
}


def all_workloads() -> dict:
    return {**WORKLOADS, **EXTRA_WORKLOADS}


def sweep_workload(mode: str, M: int) -> Workload:
    """The small-batch sweep's workload of one mode at M rows."""
    base = SWEEP_BASES[mode]
    wl = WORKLOADS.get(base) or SWEEP_WORKLOADS[base]
    return wl.with_rows(M)


def outlier_channels(wl: Workload) -> torch.Tensor:
    g = torch.Generator().manual_seed(1000 + wl.seed)
    return torch.randperm(wl.H, generator=g)[: wl.n_outliers]


def make_inputs(wl: Workload, device: str | torch.device = "cpu") -> dict:
    """Seeded inputs of a workload: x (M, H) or partials (k, M, H), residual
    (M, H) or None, weight (H,), scale (1,) fp32, eps."""
    g = torch.Generator().manual_seed(wl.seed)
    T = DTYPES[wl.dtype]
    M, H = wl.M, wl.H
    out = {}
    if wl.k > 1:
        parts = torch.randn(wl.k, M, H, generator=g) * math.sqrt(wl.part_var)
        out["x"] = parts.to(T)
    else:
        out["x"] = (torch.randn(M, H, generator=g) * math.sqrt(wl.x_var)).to(T)
    if wl.residual:
        r = torch.randn(M, H, generator=g) * math.sqrt(wl.r_var)
        if wl.n_outliers:
            r[:, outlier_channels(wl)] *= wl.outlier_mult
        out["residual"] = r.to(T)
    else:
        out["residual"] = None
    out["weight"] = (torch.randn(H, generator=g) * math.sqrt(wl.w_var)).to(T)
    out["scale"] = torch.tensor([wl.scale], dtype=torch.float32)
    out["eps"] = wl.eps
    if device != "cpu":
        out = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in out.items()}
    return out
