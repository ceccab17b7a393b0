"""Symmetries of the method, as pins of the oracle.

The fused op is exactly equivariant under a few transformations of its
inputs, and each check below states one as an identity between two oracle
runs.  None retypes the oracle's formulas; each fails on a class of slips:

* scaling x and the residual by a power of two (eps = 0) changes nothing but
  the residual, which scales: fails a norm that is not homogeneous of degree
  zero (a missing square root, a square or a mean taken wrongly, an eps that
  is not added to the mean square);
* negating x negates y and flips every code's sign bit, scales unchanged:
  fails sign handling in any encoder (an unsigned zero, a lost sign nibble);
* permuting columns (FP8), 16-element blocks (NVFP4) or 32-element blocks
  (MXFP8) of x and w permutes the outputs the same way: fails an index,
  stride or swizzle-column slip;
* a subset of rows computed alone equals those rows of the whole batch:
  fails a row stride or swizzle-row slip;
* exchanging x and the residual changes nothing (the add commutes): fails a
  residual that is scaled, rounded or written differently from x.

Inputs that keep every step exact are chosen where the identity needs it:
the column and block permutations use values on a 1/8 grid, so the sum of
squares is exact in any order.
"""
import numpy as np
import pytest
import torch

import oracle
from gnq_testutil import DTYPE_CODE, DTYPES, bits, from_bits

M, H = 37, 256   # 37 rows: a ragged 128-row scale tile; 16 NVFP4 / 8 MXFP8 blocks
MODES = [(oracle.MODE_FP8, 0.05), (oracle.MODE_NVFP4, 168.0), (oracle.MODE_MXFP8, 0.0)]
MODE_IDS = ["fp8", "nvfp4", "mxfp8"]


def _rand(shape, std, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(DTYPES[dtype])


def _grid(shape, dtype, seed):
    """N(0, 1) rounded to multiples of 1/8 in [-4, 4]: exact in both 16-bit
    types, and sums of their squares are exact in fp64 in any order."""
    g = torch.Generator().manual_seed(seed)
    v = torch.clamp(torch.round(torch.randn(shape, generator=g) * 8) / 8, -4, 4)
    return v.to(DTYPES[dtype])


def _run(x, r, w, mode, scale, dtype, eps=1e-6):
    return oracle.gemma_add_rms_norm_quant(bits(x), None if r is None else bits(r), bits(w), eps,
                                           scale, mode, DTYPE_CODE[dtype], write_y=True)


def _scale_rows(bs, mode):
    """(M, blocks) scale bytes of the logical layout (NVFP4: un-swizzled)."""
    if mode == oracle.MODE_NVFP4:
        kp = oracle.round_up(H // 16, 4)
        flat = bs.reshape(-1)
        return np.array([[flat[oracle.swizzle_offset(m, b, kp)] for b in range(H // 16)]
                         for m in range(M)], dtype=np.uint8)
    return bs


@pytest.mark.parametrize("dtype,c", [("bf16", 2.0 ** -20), ("bf16", 16.0), ("fp16", 2.0),
                                     ("fp16", 16.0)])
@pytest.mark.parametrize("mode,scale", MODES, ids=MODE_IDS)
def test_power_of_two_scaling_changes_only_the_residual(oracle_lib, dtype, c, mode, scale):
    x = _rand((M, H), 1.0, dtype, 1)
    r = _rand((M, H), 3.0, dtype, 2)
    w = _rand((H,), 0.3, dtype, 3)
    xs, rs = x * c, r * c
    # the scaled inputs are exact (no value left the normal range: fp16 is
    # only scaled up)
    assert torch.equal(xs / c, x) and torch.equal(rs / c, r)
    a = _run(x, r, w, mode, scale, dtype, eps=0.0)
    b = _run(xs, rs, w, mode, scale, dtype, eps=0.0)
    assert np.array_equal(a["y"], b["y"])
    assert np.array_equal(a["q"], b["q"])
    if a["block_scale"] is not None:
        assert np.array_equal(a["block_scale"], b["block_scale"])
    ha = from_bits(a["residual"], dtype).float()
    hb = from_bits(b["residual"], dtype).float()
    assert torch.equal(hb, ha * c)
    # and eps does enter: a large one moves y
    e = _run(x, r, w, mode, scale, dtype, eps=1.0)
    assert not np.array_equal(a["y"], e["y"])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("mode,scale", MODES, ids=MODE_IDS)
def test_negating_x_negates_y_and_flips_every_code_sign(oracle_lib, dtype, mode, scale):
    x = _rand((M, H), 1.0, dtype, 4)
    x[5, :16] = 0.0            # a zero block: +0 and -0 codes
    w = _rand((H,), 0.3, dtype, 5)
    a = _run(x, None, w, mode, scale, dtype)
    b = _run(-x, None, w, mode, scale, dtype)
    assert np.array_equal(b["y"], a["y"] ^ np.uint16(0x8000))
    if mode == oracle.MODE_NVFP4:
        assert np.array_equal(b["q"], a["q"] ^ np.uint8(0x88))
    else:
        assert np.array_equal(b["q"], a["q"] ^ np.uint8(0x80))
    if a["block_scale"] is not None:
        assert np.array_equal(a["block_scale"], b["block_scale"])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("mode,scale", MODES, ids=MODE_IDS)
def test_permuting_columns_or_blocks_permutes_the_outputs(oracle_lib, dtype, mode, scale):
    x = _grid((M, H), dtype, 6)
    r = _grid((M, H), dtype, 7)
    w = _rand((H,), 0.3, dtype, 8)
    blk = {oracle.MODE_FP8: 1, oracle.MODE_NVFP4: 16, oracle.MODE_MXFP8: 32}[mode]
    pb = np.random.default_rng(9).permutation(H // blk)
    if blk == 1:
        assert not np.array_equal(pb, np.arange(H))
    cols = (pb[:, None] * blk + np.arange(blk)[None, :]).reshape(-1)
    a = _run(x, r, w, mode, scale, dtype)
    b = _run(x[:, cols], r[:, cols], w[cols], mode, scale, dtype)
    assert np.array_equal(b["residual"], a["residual"][:, cols])
    assert np.array_equal(b["y"], a["y"][:, cols])
    if mode == oracle.MODE_NVFP4:
        qa, qb = a["q"].reshape(M, H // 16, 8), b["q"].reshape(M, H // 16, 8)
        assert np.array_equal(qb, qa[:, pb])
    else:
        assert np.array_equal(b["q"], a["q"][:, cols])
    if a["block_scale"] is not None:
        assert np.array_equal(_scale_rows(b["block_scale"], mode), _scale_rows(a["block_scale"], mode)[:, pb])


@pytest.mark.parametrize("mode,scale", MODES, ids=MODE_IDS)
def test_rows_alone_equal_the_same_rows_of_the_batch(oracle_lib, mode, scale):
    dtype = "bf16"
    x = _rand((M, H), 1.0, dtype, 10)
    r = _rand((M, H), 3.0, dtype, 11)
    w = _rand((H,), 0.3, dtype, 12)
    full = _run(x, r, w, mode, scale, dtype)
    rows = [0, 1, 17, 31, 32, 36]
    part = oracle.gemma_add_rms_norm_quant(bits(x[rows]), bits(r[rows]), bits(w), 1e-6, scale,
                                           mode, DTYPE_CODE[dtype], write_y=True)
    for key in ("residual", "y", "q"):
        assert np.array_equal(part[key], full[key][rows])
    if full["block_scale"] is not None:
        if mode == oracle.MODE_NVFP4:
            kp = oracle.round_up(H // 16, 4)
            fa, fp = full["block_scale"].reshape(-1), part["block_scale"].reshape(-1)
            for j, m in enumerate(rows):
                for b in range(H // 16):
                    assert fp[oracle.swizzle_offset(j, b, kp)] == fa[oracle.swizzle_offset(m, b, kp)]
        else:
            assert np.array_equal(part["block_scale"], full["block_scale"][rows])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("mode,scale", MODES, ids=MODE_IDS)
def test_exchanging_x_and_the_residual_changes_nothing(oracle_lib, dtype, mode, scale):
    x = _rand((M, H), 1.0, dtype, 13)
    r = _rand((M, H), 3.0, dtype, 14)
    w = _rand((H,), 0.3, dtype, 15)
    a = _run(x, r, w, mode, scale, dtype)
    b = _run(r, x, w, mode, scale, dtype)
    for key in ("residual", "y", "q", "block_scale"):
        if a[key] is not None:
            assert np.array_equal(a[key], b[key])
