"""Full-size parity: every workload (the five configurations and the MXFP8,
plain-RMSNorm and norm-only variants) at its real size, launched exactly as
bench.py launches it (automatic policy, same inputs recipe), compared with
the oracle over the WHOLE tensor:

* the updated residual bit for bit on every row;
* y within one ulp of the oracle's fp64 norm on every row;
* codes and scales bit for bit on every row when the oracle quantizes the
  GPU's own y, and the NVFP4 scale padding untouched;
* end to end (the oracle's own y -> codes) every differing code and scale
  one step away, and at most 1e-4 of them differing.

Independent library arithmetic pins the same tensors once more: the residual
equals torch's correctly rounded 16-bit add everywhere; FP8 codes equal
torch's fp32 division + saturating cast of the GPU's y; MXFP8 scales are the
E8M0 exponents of the GPU's own block amax and its codes torch's saturating
cast of y over the exact power-of-two scale.  The configured call (y not
written, as bench times it) gives the same codes as a call that writes y in
the same launch shape.
"""
import numpy as np
import pytest
import torch

import oracle
from gnq_testutil import DTYPE_CODE, bits, check_end_to_end, u8, ulp_distance16
from nvfp4_quant_gemma_gb300.workloads import all_workloads, make_inputs

pytestmark = pytest.mark.gpu

OMODE = {"fp8": oracle.MODE_FP8, "nvfp4": oracle.MODE_NVFP4, "mxfp8": oracle.MODE_MXFP8,
         "none": oracle.MODE_NONE}


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

    # every row against the oracle
    r_in = None if r0 is None else bits(r0)
    ref = oracle.gemma_add_rms_norm_quant(bits(inp["x"]), r_in, bits(inp["weight"]), wl.eps,
                                          wl.scale, om, dc, write_y=True,
                                          weight_bias=wl.weight_bias)
    del r_in
    if r0 is not None:
        assert np.array_equal(bits(r_a), ref["residual"])
    gy = bits(y_b)
    assert int(ulp_distance16(gy, ref["y"]).max()) <= 1
    if om == oracle.MODE_NONE:
        assert torch.equal(y_a, y_b)
        return
    qo, bso = oracle.quantize_from_y(gy, wl.scale, om, dc)
    gq = u8(q_a)
    assert np.array_equal(gq, qo)
    gbs = None if bs_a is None or om == oracle.MODE_FP8 else u8(bs_a)
    if gbs is not None:
        # NVFP4: the whole swizzled buffer, so the padding rows (filled with
        # the oracle's sentinel before the call) must also be untouched
        assert np.array_equal(gbs, bso)
    check_end_to_end(gq, gbs, ref, om)
