"""Batches past 2^31 elements: every 16-bit tensor over 4 GiB, so rows, codes,
scales and partials beyond the 32-bit element and byte offsets are reached.
Each case runs the automatic launch (the row kernel with a residual, the
streaming kernel without one, and k partials), with a ragged row count, and
is checked

* over the whole tensors on the device: the call without y gives the codes,
  scales and residual of a call that writes y in the same launch shape;
* against the oracle on sampled rows (both ends, the 128-row tile edges, the
  first rows whose element offset passes 2^31, and seeded random rows): the
  residual bit-exact, y within one ulp, codes and scales bit-exact from the
  GPU's own y, and the end-to-end rule against the oracle's own pipeline.

Inputs come from a seeded device generator (N(0, 1) x, N(0, 9) residual,
N(0, 0.1) w, partials N(0, 0.25)), drawn in row slabs.
"""
import numpy as np
import pytest
import torch

import oracle
from gnq_testutil import DTYPE_CODE, DTYPES, bits, check_end_to_end, u8, ulp_distance16

pytestmark = pytest.mark.gpu

OMODE = {"fp8": oracle.MODE_FP8, "nvfp4": oracle.MODE_NVFP4}

# (M, H, dtype, mode, scale, residual, k)
CASES = [
    ((1 << 18) + 77, 8192, "bf16", "nvfp4", 84.0, True, 1),
    ((1 << 18) + 77, 8192, "fp16", "fp8", 0.08, False, 1),
    ((1 << 17) + 5, 8192, "bf16", "nvfp4", 112.0, True, 3),
]


@pytest.fixture(scope="module")
def gnq():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from nvfp4_quant_gemma_gb300 import build
    build.build()
    import nvfp4_quant_gemma_gb300 as pkg
    pkg.load()
    pkg.set_launch_policy(0, 0, 0, 0)
    pkg.set_pdl(True)
    import os
    oracle.build()
    oracle.set_threads(os.cpu_count() or 1)
    return pkg


def _normal(shape, std, dtype, seed, dev):
    """Seeded N(0, std^2) in `dtype`, drawn on the device in slabs of rows."""
    g = torch.Generator(device=dev).manual_seed(seed)
    out = torch.empty(shape, dtype=dtype, device=dev)
    flat = out.view(-1, shape[-1])
    step = 1 << 14
    for a in range(0, flat.shape[0], step):
        e = min(flat.shape[0], a + step)
        flat[a:e] = (torch.randn((e - a, shape[-1]), generator=g, device=dev) * std).to(dtype)
    return out


def _sample_rows(M, H):
    m0 = -(-(1 << 31) // H)  # first row whose element offset is at least 2^31
    fixed = [0, 1, 127, 128, 129, m0 - 1, m0, m0 + 1, M - 129, M - 128, M - 2, M - 1]
    rng = np.random.default_rng(M + H)
    rows = sorted({r for r in fixed + list(rng.integers(0, M, 24)) if 0 <= r < M})
    return np.array(rows, dtype=np.int64)


@pytest.mark.parametrize("M,H,dt,mode,scale,residual,k", CASES,
                         ids=[f"{c[3]}_{c[0]}x{c[1]}_k{c[6]}_{'res' if c[5] else 'nores'}" for c in CASES])
def test_past_2_31_elements(gnq, M, H, dt, mode, scale, residual, k):
    dev = torch.device("cuda")
    T = DTYPES[dt]
    om = OMODE[mode]
    assert k * M * H > (1 << 31)
    x = _normal((k, M, H) if k > 1 else (M, H), 0.5 if k > 1 else 1.0, T, 11, dev)
    w = _normal((1, H), 0.1 ** 0.5, T, 12, dev).view(H)
    s = torch.tensor([scale], device=dev)

    def call(write_y):
        r = _normal((M, H), 3.0, T, 13, dev) if residual else None
        out = gnq.alloc_outputs(M, H, mode, write_y, x)
        if out[1] is not None:
            out[1].view(torch.uint8).fill_(oracle.SENTINEL)
        if k > 1:
            gnq.gemma_add_rms_norm_quant_parts(x, r, w, 1e-6, s, mode, write_y=write_y, out=out)
        else:
            gnq.gemma_add_rms_norm_quant(x, r, w, 1e-6, s, mode, write_y=write_y, out=out)
        return r, out

    # the call as configured (no y), then one that writes y in the same shape
    r_a, (q_a, bs_a, _) = call(False)
    shape = gnq.query_launch(M, H, mode, dt, k=k, residual=residual, write_y=False)
    gnq.set_launch_policy(*shape)
    try:
        r_b, (q_b, bs_b, y_b) = call(True)
    finally:
        gnq.set_launch_policy(0, 0, 0, 0)
    torch.cuda.synchronize()
    assert gnq.read_device_error() == 0
    assert torch.equal(q_a.view(torch.uint8), q_b.view(torch.uint8))
    if bs_a is not None:
        assert torch.equal(bs_a.view(torch.uint8), bs_b.view(torch.uint8))
    if residual:
        assert torch.equal(r_a, r_b)
    del q_b, bs_b, r_b

    # sampled rows against the oracle
    rows = _sample_rows(M, H)
    idx = torch.from_numpy(rows).to(dev)
    xs = x.index_select(1 if k > 1 else 0, idx).cpu()
    r_in = _normal((M, H), 3.0, T, 13, dev).index_select(0, idx).cpu() if residual else None
    ref = oracle.gemma_add_rms_norm_quant(bits(xs), None if r_in is None else bits(r_in),
                                          bits(w.cpu()), 1e-6, scale, om, DTYPE_CODE[dt],
                                          write_y=True)
    if residual:
        assert np.array_equal(bits(r_a.index_select(0, idx).cpu()), ref["residual"])
    gy = bits(y_b.index_select(0, idx).cpu())
    assert int(ulp_distance16(gy, ref["y"]).max()) <= 1
    gq = u8(q_a.view(torch.uint8).index_select(0, idx).cpu())
    qo, bso = oracle.quantize_from_y(gy, scale, om, DTYPE_CODE[dt])
    assert np.array_equal(gq, qo)
    gbs = None
    if om == oracle.MODE_NVFP4:
        # the sampled rows' scale bytes, gathered into the sub-batch's own
        # swizzled layout (padding left at the sentinel, as the oracle's)
        kp_full = oracle.round_up(H // 16, 4)
        flat = u8(bs_a.view(torch.uint8).reshape(-1).cpu())
        gbs = np.full(bso.shape, oracle.SENTINEL, np.uint8).reshape(-1)
        for j, m in enumerate(rows):
            for b in range(H // 16):
                gbs[oracle.swizzle_offset(j, b, kp_full)] = flat[oracle.swizzle_offset(int(m), b, kp_full)]
        gbs = gbs.reshape(bso.shape)
        assert np.array_equal(gbs, bso)
    check_end_to_end(gq, gbs, ref, om)
    del x, r_a, q_a, bs_a, y_b
    torch.cuda.empty_cache()
