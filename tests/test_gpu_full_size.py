"""Full-size parity: every workload (the five configurations and the MXFP8,
plain-RMSNorm and norm-only variants) at its real size, launched exactly as
bench.py launches it (automatic policy, same inputs recipe).

* Sampled rows (first, last, a seeded random set) against the oracle: the
  updated residual bit for bit, y within one ulp, codes and scales bit for
  bit from the GPU's own y, scale padding untouched.
* Whole-tensor properties from independent library arithmetic: the
  residual equals torch's correctly rounded 16-bit add everywhere; FP8
  codes equal torch's fp32 division + saturating cast of the GPU's y
  everywhere; NVFP4 codes dequantize to within one code step of y; MXFP8
  scales are the E8M0 exponents of the GPU's own block amax and its codes
  torch's saturating cast of y over the exact power-of-two scale.
* The configured write_y=False call gives the same codes as a write_y=True
  call on the same inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from gnq_testutil import DTYPE_CODE, bits, u8, ulp_distance16, unpack_nibbles
from nvfp4_quant_gemma_gb300.workloads import all_workloads, make_inputs

pytestmark = pytest.mark.gpu

OMODE = {"fp8": oracle.MODE_FP8, "nvfp4": oracle.MODE_NVFP4, "mxfp8": oracle.MODE_MXFP8,
         "none": oracle.MODE_NONE}
N_SAMPLE = 24


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


def _call(gnq, wl, x, r, w, s, write_y):
    out = gnq.alloc_outputs(wl.M, wl.H, wl.mode, write_y, x)
    if wl.mode == "nvfp4":
        out[1].view(torch.uint8).fill_(0xA5)
    if wl.weight_bias == 0.0:
        gnq.add_rms_norm_quant(x, r, w, wl.eps, s, wl.mode, write_y=write_y, out=out)
    elif wl.k > 1:
        gnq.gemma_add_rms_norm_quant_parts(x, r, w, wl.eps, s, wl.mode, write_y=write_y, out=out)
    elif wl.mode == "none":
        gnq.gemma_add_rms_norm(x, r, w, wl.eps, y=out[2])
    else:
        gnq.gemma_add_rms_norm_quant(x, r, w, wl.eps, s, wl.mode, write_y=write_y, out=out)
    return out


@pytest.mark.parametrize("name", list(all_workloads()))
def test_workload_full_size(gnq, name):
    wl = all_workloads()[name]
    dev = torch.device("cuda")
    inp = make_inputs(wl)
    x = inp["x"].to(dev)
    w = inp["weight"].to(dev)
    s = inp["scale"].to(dev)
    r0 = inp["residual"]
    dc = DTYPE_CODE[wl.dtype]
    om = OMODE[wl.mode]

    # the configured call (as bench.py times it), then one that also writes y
    # in the configured call's launch shape (the automatic policy may pick
    # another shape once y is written, and the shape may move y by a rounding)
    r_a = None if r0 is None else r0.to(dev)
    q_a, bs_a, y_a = _call(gnq, wl, x, r_a, w, s, wl.write_y)
    shape = gnq.query_launch(wl.M, wl.H, wl.mode, wl.dtype, k=wl.k, residual=r0 is not None,
                             write_y=wl.write_y, weight_bias=wl.weight_bias)
    r_b = None if r0 is None else r0.to(dev)
    gnq.set_launch_policy(*shape)
    try:
        q_b, bs_b, y_b = _call(gnq, wl, x, r_b, w, s, True)
    finally:
        gnq.set_launch_policy(0, 0, 0, 0)
    torch.cuda.synchronize()
    if om != oracle.MODE_NONE:
        assert torch.equal(q_a.view(torch.uint8), q_b.view(torch.uint8))
    if bs_a is not None and om in (oracle.MODE_NVFP4, oracle.MODE_MXFP8):
        assert torch.equal(bs_a.view(torch.uint8), bs_b.view(torch.uint8))
    assert gnq.read_device_error() == 0

    # whole tensor: residual = torch's correctly rounded 16-bit add (of the
    # partials summed in fp32 in index order and rounded once)
    if wl.k > 1:
        acc = x[0].float()
        for i in range(1, wl.k):
            acc = acc + x[i].float()
        h_dev = acc.to(x.dtype)
        del acc
    else:
        h_dev = x
    if r0 is not None:
        ref_r = h_dev + r0.to(dev)
        assert torch.equal(r_a, ref_r) and torch.equal(r_b, ref_r)
    del h_dev

    # whole tensor: codes from the GPU's own y by library arithmetic
    if om == oracle.MODE_FP8:
        ref_q = (y_b.float() / s).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
        assert torch.equal(q_b.view(torch.uint8), ref_q.view(torch.uint8))
        del ref_q
    elif om == oracle.MODE_MXFP8:
        # E8M0 code = floor(log2(block amax)) - 8 + 127 clamped to [0, 254] (0 for
        # an all-zero block); codes = saturating E4M3 of y / 2^(code - 127)
        yb32 = y_b.float().reshape(wl.M, wl.H // 32, 32)
        amax = yb32.abs().amax(dim=-1)
        e = torch.frexp(amax).exponent - 1          # floor(log2(amax)) for amax > 0
        want = torch.where(amax > 0, (e - 8 + 127).clamp(0, 254), torch.zeros_like(e))
        got = bs_b.view(torch.uint8).reshape(wl.M, wl.H // 32).long()
        assert torch.equal(got, want.long())
        inv = torch.ldexp(torch.ones_like(amax), (127 - got).to(torch.int32))
        ref_q = (yb32 * inv[..., None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
        assert torch.equal(q_b.view(torch.uint8), ref_q.view(torch.uint8).reshape(wl.M, wl.H))
        del yb32, amax, e, want, got, inv, ref_q
    elif om == oracle.MODE_NVFP4:
        # decode codes * sf / g and check |dequant - y| <= one code step
        M, H = wl.M, wl.H
        codes = torch.stack([q_b & 0xF, q_b >> 4], dim=-1).reshape(M, H).long()
        table = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6],
                             device=dev)
        vals = table[codes].reshape(M, H // 16, 16)
        Kp = H // 16
        m_idx = torch.arange(M, device=dev)[:, None]
        b_idx = torch.arange(Kp, device=dev)[None, :]
        off = ((m_idx // 128) * (Kp // 4) + b_idx // 4) * 512 + (m_idx % 32) * 16 \
            + ((m_idx % 128) // 32) * 4 + b_idx % 4
        sf = bs_b.view(torch.float8_e4m3fn).reshape(-1)[off.reshape(-1)].float().reshape(M, Kp)
        g = float(wl.scale)
        deq = vals * (sf / g)[..., None]
        yv = y_b.float().reshape(M, H // 16, 16)
        step = (sf / g)[..., None] * 2.0  # the largest E2M1 step is 2
        unsat = ((sf > 0) & (sf < 448))[..., None]  # blocks whose scale neither saturated nor vanished
        assert bool(((deq - yv).abs() <= step * 1.0001 + 1e-30)[unsat.expand_as(yv)].all())
        del codes, vals, deq, yv, step

    # sampled rows against the oracle
    rng = np.random.default_rng(wl.seed)
    rows = sorted({0, wl.M - 1, *rng.choice(wl.M, size=min(N_SAMPLE, wl.M), replace=False).tolist()})
    xs = inp["x"][:, rows] if wl.k > 1 else inp["x"][rows]
    rs = None if r0 is None else r0[rows]
    ref = oracle.gemma_add_rms_norm_quant(bits(xs), None if rs is None else bits(rs),
                                          bits(inp["weight"]), wl.eps, wl.scale, om, dc,
                                          write_y=True, weight_bias=wl.weight_bias)
    if r0 is not None:
        assert np.array_equal(bits(r_a[rows]), ref["residual"])
    gy = bits(y_b[rows])
    assert int(ulp_distance16(gy, ref["y"]).max()) <= 1
    if om == oracle.MODE_NONE:
        assert torch.equal(y_a, y_b)
        return
    qo, bso = oracle.quantize_from_y(gy, wl.scale, om, dc)
    assert np.array_equal(u8(q_a[rows]), qo)
    if om == oracle.MODE_MXFP8:
        assert np.array_equal(u8(bs_a[rows]), bso)
    if om == oracle.MODE_NVFP4:
        Kp = wl.H // 16
        flat = u8(bs_a).reshape(-1)
        for i, m in enumerate(rows):
            got = flat[[oracle.swizzle_offset(m, b, Kp) for b in range(Kp)]]
            want = bso.reshape(-1)[[oracle.swizzle_offset(i, b, Kp) for b in range(Kp)]]
            assert np.array_equal(got, want)
        # padding rows of the last 128-row tile stay untouched
        Mp = oracle.round_up(wl.M, 128)
        if Mp > wl.M:
            pad = [oracle.swizzle_offset(m, b, Kp) for m in range(wl.M, Mp) for b in range(Kp)]
            assert np.all(flat[pad] == 0xA5)
    # end to end on the sampled rows
    if om == oracle.MODE_NVFP4:
        a = unpack_nibbles(u8(q_a[rows])).astype(np.int64)
        b = unpack_nibbles(ref["q"]).astype(np.int64)
        ra = np.where(a & 8, -(a & 7), a & 7)
        rb = np.where(b & 8, -(b & 7), b & 7)
    else:
        a = u8(q_a[rows]).astype(np.int64)
        b = ref["q"].astype(np.int64)
        ra = np.where(a & 0x80, -(a & 0x7F), a & 0x7F)
        rb = np.where(b & 0x80, -(b & 0x7F), b & 0x7F)
    diff = np.abs(ra - rb)
    assert int(diff.max(initial=0)) <= 1
    assert np.count_nonzero(diff) <= max(1, int(1e-4 * diff.size))
