"""GPU parity: the sm_103a library against the CPU oracle, through the C ABI.

Rules (the method's correctness contract):
  * the updated residual is bit-exact;
  * y is within 1 unit in the last place of the activation dtype (relative
    2^-8 for bf16, 2^-11 for fp16) of the oracle's fp64 norm;
  * codes and block scales are bit-exact when the oracle quantizes the GPU's
    own y (the same fp32 decisions on both sides);
  * end to end (oracle y -> oracle codes vs GPU codes) every differing code
    is an adjacent code, and at most 1e-4 of the elements differ (checked
    where a tensor holds at least 1e5 codes: below that the fraction is
    under ten codes and the bound is not meaningful); the same rule for the
    NVFP4 E4M3 block-scale bytes and the MXFP8 E8M0 scale codes (MXFP8 codes
    are compared where the two scales agree: a scale one code apart
    rescales its whole block by 2);
  * NVFP4 scale rows >= M, and bytes around every output, are untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from gnq_testutil import DTYPE_CODE, DTYPES, bits, check_end_to_end, u8, ulp_distance16

pytestmark = pytest.mark.gpu

OMODE = {"none": oracle.MODE_NONE, "fp8": oracle.MODE_FP8, "nvfp4": oracle.MODE_NVFP4,
         "mxfp8": oracle.MODE_MXFP8}
SENT = 0xA5
GUARD = 256


@pytest.fixture(scope="module")
def gnq():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from nvfp4_quant_gemma_gb300 import build
    build.build()
    import nvfp4_quant_gemma_gb300 as pkg
    pkg.load()
    pkg.set_launch_policy(0, 0, 0, 0)
    oracle.build()
    import os
    oracle.set_threads(os.cpu_count() or 1)
    return pkg


def _guarded(shape, dtype, dev):
    """A tensor inside a sentinel-filled buffer with GUARD bytes on each side."""
    nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    buf = torch.full((nbytes + 2 * GUARD,), SENT, dtype=torch.uint8, device=dev)
    t = buf[GUARD:GUARD + nbytes].view(dtype).view(shape)
    return buf, t


def _guards_intact(buf):
    b = buf.cpu().numpy()
    return bool(np.all(b[:GUARD] == SENT) and np.all(b[-GUARD:] == SENT))


def _make(M, H, dtype, seed, k=1, residual=True, r_std=3.0, w_std=0.3, special=True):
    g = torch.Generator().manual_seed(seed)
    T = DTYPES[dtype]
    x = torch.randn((k, M, H) if k > 1 else (M, H), generator=g)
    if k > 1:
        x = x * 0.5
    r = torch.randn(M, H, generator=g) * r_std if residual else None
    w = torch.randn(H, generator=g) * w_std
    if special and M >= 3 and residual:
        r[:, :: max(1, H // 7)] *= 20.0  # outlier channels (saturate FP8/NVFP4)
        r[1] = 0.0                       # row 1: residual zero
        x[..., 2, :] = 0.0               # row 2: x zero
        if M >= 4:
            r[3] = 0.0
            x[..., 3, :] = 0.0           # row 3: all zero -> y = 0, scales 0
    return x.to(T), (None if r is None else r.to(T)), w.to(T)


def run_case(gnq, x, r, w, mode, scale, write_y, dtype, eps=1e-6, weight_bias=1.0, check_e2e=True):
    """Run GPU and oracle on the same inputs and assert every parity rule."""
    dev = torch.device("cuda")
    T = DTYPES[dtype]
    dc = DTYPE_CODE[dtype]
    k = x.shape[0] if x.dim() == 3 else 1
    M, H = x.shape[-2:]
    om = OMODE[mode]
    ref = oracle.gemma_add_rms_norm_quant(bits(x), None if r is None else bits(r), bits(w), eps,
                                          scale, om, dc, write_y=True, weight_bias=weight_bias)

    xd, wd = x.to(dev), w.to(dev)
    sd = torch.tensor([scale], dtype=torch.float32, device=dev)
    results = {}
    for wy in sorted({True, bool(write_y)}):
        rd_buf, rd = (None, None) if r is None else _guarded((M, H), T, dev)
        if rd is not None:
            rd.copy_(r.to(dev))
        qb = bsb = yb = None
        q = bs = y = None
        if om in (oracle.MODE_FP8, oracle.MODE_MXFP8):
            qb, q = _guarded((M, H), torch.uint8, dev)
        elif om == oracle.MODE_NVFP4:
            qb, q = _guarded((M, H // 2), torch.uint8, dev)
        if om == oracle.MODE_NVFP4:
            bsb, bs = _guarded(oracle.scale_shape(M, H, om), torch.uint8, dev)
        elif om == oracle.MODE_MXFP8:
            bsb, bs = _guarded(oracle.scale_shape(M, H, om), torch.uint8, dev)
        if wy or om == oracle.MODE_NONE:
            yb, y = _guarded((M, H), T, dev)
        if k == 1 and weight_bias == 1.0:
            if om == oracle.MODE_NONE:
                gnq.gemma_add_rms_norm(xd, rd, wd, eps, y=y)
            else:
                gnq.gemma_add_rms_norm_quant(xd, rd, wd, eps, sd, mode, write_y=wy, out=(q, bs, y))
        else:
            fn = gnq.gemma_add_rms_norm_quant_parts if weight_bias == 1.0 else gnq.add_rms_norm_quant
            fn(xd, rd, wd, eps, sd, mode, write_y=wy, out=(q, bs, y))
        torch.cuda.synchronize()
        for b in (rd_buf, qb, bsb, yb):
            if b is not None:
                assert _guards_intact(b), "a write landed outside its buffer"
        results[wy] = dict(r=rd, q=q, bs=bs, y=y)

    full = results[True]
    # residual: bit-exact
    if r is not None:
        assert np.array_equal(bits(full["r"]), ref["residual"])
    # y: within one ulp of the fp64 oracle
    gy = bits(full["y"])
    assert int(ulp_distance16(gy, ref["y"]).max()) <= 1
    if om == oracle.MODE_NONE:
        return
    # write_y does not change the codes
    if not write_y:
        assert np.array_equal(u8(results[False]["q"]), u8(full["q"]))
        if full["bs"] is not None:
            assert np.array_equal(u8(results[False]["bs"]), u8(full["bs"]))
        if r is not None:
            assert np.array_equal(bits(results[False]["r"]), ref["residual"])
    # codes from the GPU's own y: bit-exact
    qo, bso = oracle.quantize_from_y(gy, scale, om, dc)
    gq = u8(full["q"])
    assert np.array_equal(gq, qo)
    if om == oracle.MODE_NVFP4:
        gbs = u8(full["bs"]).reshape(-1)
        Kp = oracle.round_up(H // 16, 4)
        written = np.zeros(gbs.size, bool)
        for m in range(M):
            for b in range(H // 16):
                written[oracle.swizzle_offset(m, b, Kp)] = True
        assert np.array_equal(gbs[written], bso.reshape(-1)[written])
        assert np.all(gbs[~written] == SENT), "padding rows of the scale tensor were written"
    elif om == oracle.MODE_MXFP8:
        assert np.array_equal(u8(full["bs"]), bso)
    # end to end: oracle codes vs GPU codes
    if check_e2e:
        check_end_to_end(gq, None if full["bs"] is None else u8(full["bs"]), ref, om)


# --- hardware encoders vs the oracle's reading ----------------------------------

def test_hardware_encoders_match_oracle(gnq):
    rng = np.random.default_rng(0)
    e4_vals = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = (e4_vals[:-1] + e4_vals[1:]) / 2
    e2_vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6.0])
    mids2 = (e2_vals[:-1] + e2_vals[1:]) / 2
    v = np.concatenate([
        rng.standard_normal(100000) * np.ldexp(1.0, rng.integers(-14, 10, 100000)),
        mids, -mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
        np.nextafter(mids.astype(np.float32), np.float32(1e9)),
        mids2, -mids2, e4_vals, -e4_vals,
        [0.0, -0.0, 1e-30, -1e-30, 2.0 ** -10, 3 * 2.0 ** -11, 448.0, 464.0, 500.0, 1e30,
         -1e30, 6.0, 6.5, 7.0, -100.0, np.inf, -np.inf, 1e-45, -1e-45]]).astype(np.float32)
    vd = torch.from_numpy(v).cuda()
    e4, e2 = gnq.encode_e4m3_e2m1(vd)
    torch.cuda.synchronize()
    v64 = v.astype(np.float64)
    assert np.array_equal(e4.cpu().numpy(), oracle.e4m3_encode(v64))
    assert np.array_equal(e2.cpu().numpy(), oracle.e2m1_encode(v64))


# --- small shapes: several tiles, ragged tails, every mode ---------------------

SMALL_M = [1, 3, 127, 129, 300]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("mode,scale", [("fp8", 0.05), ("nvfp4", 168.0), ("mxfp8", 0.0)])
@pytest.mark.parametrize("M", SMALL_M)
@pytest.mark.parametrize("H", [64, 2048, 5120])
def test_small_shapes(gnq, dtype, mode, scale, M, H):
    x, r, w = _make(M, H, dtype, seed=M * 7 + H)
    run_case(gnq, x, r, w, mode, scale, write_y=(M % 2 == 1), dtype=dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("mode,scale", [("fp8", 0.08), ("nvfp4", 84.0)])
def test_no_residual(gnq, dtype, mode, scale):
    x, _, w = _make(200, 8192, dtype, seed=11, residual=False)
    run_case(gnq, x, None, w, mode, scale, write_y=False, dtype=dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("M,H", [(1, 8), (5, 24), (130, 4096), (64, 8192)])
def test_norm_only(gnq, dtype, M, H):
    x, r, w = _make(M, H, dtype, seed=5)
    run_case(gnq, x, r, w, "none", 0.0, write_y=True, dtype=dtype)


@pytest.mark.parametrize("k", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("mode,scale", [("nvfp4", 112.0), ("fp8", 0.05), ("none", 0.0)])
def test_partials(gnq, k, mode, scale):
    x, r, w = _make(150, 7168, "bf16", seed=k, k=k)
    run_case(gnq, x, r, w, mode, scale, write_y=True, dtype="bf16")


@pytest.mark.parametrize("mode,scale", [("fp8", 0.05), ("nvfp4", 168.0)])
@pytest.mark.parametrize("kernel,form", [(1, 1), (1, 2), (2, 1), (2, 2)])
def test_plain_rmsnorm_variant(gnq, mode, scale, kernel, form):
    x, r, w = _make(100, 2048, "bf16", seed=3, w_std=1.0)
    with forced_policy(gnq, kernel, 0, 0, form):
        run_case(gnq, x, r, w, mode, scale, write_y=True, dtype="bf16", weight_bias=0.0)


def test_odd_h_fp8(gnq):
    # H a multiple of 8 but not of 16 or 64 (FP8 and the plain norm accept it)
    x, r, w = _make(37, 8 * 129, "bf16", seed=1)
    run_case(gnq, x, r, w, "fp8", 0.02, write_y=True, dtype="bf16")


def test_max_h(gnq):
    x, r, w = _make(3, 65536, "bf16", seed=2)
    run_case(gnq, x, r, w, "nvfp4", 168.0, write_y=True, dtype="bf16")
    run_case(gnq, x, r, w, "fp8", 0.05, write_y=False, dtype="bf16")


class forced_policy:
    def __init__(self, gnq, kernel, cluster=0, vpt=0, form=0):
        self.gnq, self.args = gnq, (kernel, cluster, vpt, form)

    def __enter__(self):
        self.gnq.set_launch_policy(*self.args)

    def __exit__(self, *exc):
        self.gnq.set_launch_policy(0, 0, 0, 0)


@pytest.mark.parametrize("kernel,cluster,vpt", [(1, c, v) for c in (1, 2, 4, 8) for v in (1, 2, 4)]
                         + [(2, 0, v) for v in (1, 2, 4)] + [(2, r, 2) for r in (2, 8)])
@pytest.mark.parametrize("form", [1, 2])
def test_every_launch_shape(gnq, kernel, cluster, vpt, form):
    """Forced kernels, cluster sizes (for the streaming kernel: at least that
    many rows per CTA), units per thread and register forms give the same
    contract."""
    x, r, w = _make(133, 4096, "bf16", seed=cluster * 10 + vpt + kernel)
    with forced_policy(gnq, kernel, cluster, vpt, form):
        run_case(gnq, x, r, w, "nvfp4", 168.0, write_y=True, dtype="bf16")
        run_case(gnq, x, r, w, "mxfp8", 0.0, write_y=False, dtype="bf16")
        run_case(gnq, x, r, w, "fp8", 0.05, write_y=False, dtype="bf16")
    assert gnq.read_device_error() == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("mode,scale", [("fp8", 0.08), ("nvfp4", 84.0), ("mxfp8", 0.0), ("none", 0.0)])
@pytest.mark.parametrize("M,H,k,res", [(1, 64, 1, True), (7, 2048, 1, False), (333, 5120, 1, True),
                                       (1000, 8192, 1, True), (610, 7168, 4, True),
                                       (300, 16384, 1, True), (160, 1024, 3, False)])
@pytest.mark.parametrize("form", [1, 2])
def test_streaming_kernel(gnq, dtype, mode, scale, M, H, k, res, form):
    """The persistent shared-memory-ring kernel on ragged row counts (rows per
    CTA differ), every mode, with and without residual and partials, in both
    register forms."""
    x, r, w = _make(M, H, dtype, seed=M + H + k, k=k, residual=res)
    with forced_policy(gnq, 2, 0, 0, form):
        run_case(gnq, x, r, w, mode, scale, write_y=(M % 2 == 0), dtype=dtype)
    assert gnq.read_device_error() == 0


@pytest.mark.parametrize("kernel", [1, 2])
def test_fp8_clamped_path_with_huge_weights(gnq, kernel):
    """bf16 weights near 1e36 make y * (1/s) overflow fp32: the kernels must
    take the clamped quotient and still saturate exactly like the oracle."""
    M, H = 400, 2048
    x, r, w = _make(M, H, "bf16", seed=41)
    w = w.float()
    w[::5] = 1e36
    w[1::5] = -3e35
    w = w.to(torch.bfloat16)
    with forced_policy(gnq, kernel):
        run_case(gnq, x, r, w, "fp8", 0.001, write_y=True, dtype="bf16")


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_extreme_scales(gnq, kernel, dtype):
    """The fused kernels at the edges of their scale handling: static FP8
    scales at and beyond the FMA-corrected quotient's range [2^-80, 2^80]
    (outside it, and for a negative scale, the kernels divide), and NVFP4
    global scales across the fp32 range (block scales saturating at 448,
    subnormal, or zero so every code is a signed zero)."""
    M, H = 70, 1024
    x, r, w = _make(M, H, dtype, seed=53)
    with forced_policy(gnq, kernel):
        for s in (2.0 ** -90, 2.0 ** -80, 2.0 ** 80, 2.0 ** 81, 1e30, -0.05):
            run_case(gnq, x, r, w, "fp8", s, write_y=True, dtype=dtype)
        for g in (2.0 ** -60, 1e-6, 1.0, 1e6, 2.0 ** 100):
            run_case(gnq, x, r, w, "nvfp4", g, write_y=False, dtype=dtype)
    assert gnq.read_device_error() == 0


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_mxfp8_overflowing_blocks(gnq, kernel, dtype):
    """Weights that push y past the 16-bit range (fp16: inf; bf16: huge
    finite values): blocks holding an inf take the top E8M0 code, the rest
    of the row its own codes, exactly as the oracle quantizes the GPU's y."""
    M, H = 300, 1024
    x, r, w = _make(M, H, dtype, seed=43)
    w = w.float()
    w[5:37:3] = 6.0e4 if dtype == "fp16" else 1e38
    w = w.to(DTYPES[dtype])
    with forced_policy(gnq, kernel):
        run_case(gnq, x, r, w, "mxfp8", 0.0, write_y=True, dtype=dtype)


@pytest.mark.parametrize("M,H,res,write_y,mode,scale,kernel", [
    (2048, 5120, True, True, "nvfp4", 168.0, 1),    # residual: one CTA per row
    (2560, 2048, False, False, "fp8", 0.05, 2),     # no residual, no y: streaming
    (2560, 2048, False, False, "nvfp4", 168.0, 2),
    (2560, 2048, False, False, "mxfp8", 0.0, 2),
    (2560, 2048, False, True, "fp8", 0.05, 1),      # no residual, y written: one CTA per row
])
def test_automatic_policy_large_batch(gnq, M, H, res, write_y, mode, scale, kernel):
    """The automatic launch shape of prefill-sized batches in each branch of
    the policy (from 16 x SMs rows): the kernel it picks, and parity of the
    automatic launch (a call without y in the shape the query reports for
    it, compared with a call that writes y in that same shape)."""
    x, r, w = _make(M, H, "bf16", seed=77)
    shape = gnq.query_launch(M, H, mode, "bf16", residual=res, write_y=write_y)
    if torch.cuda.get_device_properties(0).multi_processor_count * 16 <= M:
        assert shape[0] == kernel
        if shape[2] == 4:
            assert shape[3] == 2  # packed form at four units per thread
    if write_y:
        run_case(gnq, x, r if res else None, w, mode, scale, write_y=True, dtype="bf16")
    else:
        # the automatic shape of the call without y, forced on both of
        # run_case's calls (with and without y) so they share its arithmetic
        gnq.set_launch_policy(*shape)
        try:
            run_case(gnq, x, r if res else None, w, mode, scale, write_y=False, dtype="bf16")
        finally:
            gnq.set_launch_policy(0, 0, 0, 0)
    assert gnq.read_device_error() == 0


def _all_finite_16bit(dtype):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = torch.from_numpy(pats.view(np.int16)).view(DTYPES[dtype]).float()
    return v[torch.isfinite(v)].contiguous()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fp8_quotient_every_16bit_value(gnq, dtype):
    """The kernels' y / s (FMA-corrected reciprocal path, IEEE division for
    extreme scales) against the oracle on every finite 16-bit y."""
    y = _all_finite_16bit(dtype)
    yd = y.cuda()
    rng = np.random.default_rng(5)
    scales = [0.02, 0.05, 0.08, 1.0, 0.03, 3.0, 448.0, 2.0 ** -80, 2.0 ** 80, 2.0 ** -81,
              1e-30, 1e30, -0.05, 7e-5]
    scales += list(np.exp(rng.uniform(np.log(1e-4), np.log(1e4), 40)))
    y64 = y.double().numpy()
    for s in scales:
        s32 = np.float32(s)
        q = gnq.quantize_fp8_values(yd, torch.tensor([s32], device="cuda")).cpu().numpy()
        ref = oracle.e4m3_encode((y.numpy() / s32).astype(np.float64))  # fp32 IEEE division
        assert np.array_equal(q, ref), f"scale {s}"


def test_special_rows(gnq):
    """Zero rows, a weight of -1 (y is a signed zero), and tiny values."""
    M, H = 8, 256
    x = torch.randn(M, H).to(torch.bfloat16)
    x[0] = 0.0
    x[1] = 2.0 ** -120
    x[2, ::2] = -x[2, ::2].abs()
    r = torch.zeros(M, H, dtype=torch.bfloat16)
    w = torch.randn(H).to(torch.bfloat16)
    w[:32] = -1.0
    for mode, s in (("fp8", 0.02), ("nvfp4", 168.0), ("mxfp8", 0.0)):
        run_case(gnq, x, r, w, mode, s, write_y=True, dtype="bf16")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("kernel", [1, 2])
def test_subnormal_and_cancelling_residuals(gnq, dtype, kernel):
    """Residual sums that are subnormal, cancel to +-0, or round at ties are
    bit-exact (the packed 16-bit add keeps subnormals)."""
    M, H = 300, 1024
    T = DTYPES[dtype]
    tiny = 2.0 ** (-133 if dtype == "bf16" else -24)   # smallest subnormal
    g = torch.Generator().manual_seed(3)
    x = (torch.randint(-40, 40, (M, H), generator=g).float() * tiny)
    r = (torch.randint(-40, 40, (M, H), generator=g).float() * tiny)
    r[::3] = -x[::3]                                    # exact cancellation
    x[1, :64] = -0.0
    r[1, :64] = -0.0                                    # -0 + -0 = -0
    x[5:, :] = torch.randn(M - 5, H, generator=g)       # normal rows for the quantizers
    x, r = x.to(T), r.to(T)
    w = torch.randn(H, generator=g).to(T)
    with forced_policy(gnq, kernel):
        for mode, s in (("fp8", 0.05), ("nvfp4", 168.0)):
            run_case(gnq, x, r, w, mode, s, write_y=True, dtype=dtype, check_e2e=False)


def test_empty_batch(gnq):
    dev = torch.device("cuda")
    x = torch.empty(0, 128, dtype=torch.bfloat16, device=dev)
    w = torch.zeros(128, dtype=torch.bfloat16, device=dev)
    s = torch.ones(1, dtype=torch.float32, device=dev)
    q, bs, y = gnq.gemma_add_rms_norm_quant(x, None, w, 1e-6, s, "nvfp4", write_y=True)
    assert q.shape == (0, 64) and bs.shape == (0, 8) and y.shape == (0, 128)


def test_stream_and_graph_capture(gnq):
    """A side stream and a captured CUDA graph give the eager results."""
    dev = torch.device("cuda")
    x, r, w = _make(256, 4096, "bf16", seed=9)
    xd, wd = x.to(dev), w.to(dev)
    sd = torch.tensor([0.05], device=dev)
    r1 = r.to(dev)
    q1, _, y1 = gnq.gemma_add_rms_norm_quant(xd, r1, wd, 1e-6, sd, "fp8", write_y=True)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    r2 = r.to(dev)
    with torch.cuda.stream(side):
        q2, _, y2 = gnq.gemma_add_rms_norm_quant(xd, r2, wd, 1e-6, sd, "fp8", write_y=True)
    side.synchronize()
    r3 = r.to(dev)
    out = gnq.alloc_outputs(256, 4096, "fp8", True, xd)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gnq.gemma_add_rms_norm_quant(xd, r3, wd, 1e-6, sd, "fp8", write_y=True, out=out)
    r3.copy_(r.to(dev))
    g.replay()
    torch.cuda.synchronize()
    for qq, yy, rr in ((q2, y2, r2), (out[0], out[2], r3)):
        assert torch.equal(qq.view(torch.uint8), q1.view(torch.uint8))
        assert torch.equal(yy, y1) and torch.equal(rr, r1)


@pytest.mark.parametrize("mode,scale,M,k", [("fp8", 0.05, 256, 1), ("nvfp4", 168.0, 256, 1),
                                            ("fp8", 0.05, 4096, 1), ("nvfp4", 168.0, 4096, 1),
                                            ("nvfp4", 168.0, 4096, 2), ("fp8", 0.05, 4096, 2)])
def test_pdl_on_and_off_agree(gnq, mode, scale, M, k):
    """Programmatic dependent launch changes launch timing only: a chain of
    dependent calls (each consuming the previous residual) gives the same
    bits with it on and off, eagerly and in a captured graph -- one-wave and
    many-wave row grids, and the persistent streaming grid (k partials)."""
    dev = torch.device("cuda")
    x, r, w = _make(M, 4096, "bf16", seed=31)
    xd, wd = x.to(dev), w.to(dev)
    if k > 1:
        xd = torch.stack([xd, (xd * 0.5).to(xd.dtype)])
    sd = torch.tensor([scale], device=dev)

    def chain(pdl, graph):
        gnq.set_pdl(pdl)
        try:
            rd = r.to(dev)
            outs = [gnq.alloc_outputs(M, 4096, mode, True, xd) for _ in range(4)]
            def run():
                for o in outs:  # each call reads the residual the previous one wrote
                    if k > 1:
                        gnq.gemma_add_rms_norm_quant_parts(xd, rd, wd, 1e-6, sd, mode, write_y=True, out=o)
                    else:
                        gnq.gemma_add_rms_norm_quant(xd, rd, wd, 1e-6, sd, mode, write_y=True, out=o)
            if graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    run()
                rd.copy_(r.to(dev))
                g.replay()
            else:
                run()
            torch.cuda.synchronize()
            return [rd.clone()] + [t.view(torch.uint8).clone() if t.dtype != torch.bfloat16 else t.clone()
                                   for o in outs for t in o if t is not None]
        finally:
            gnq.set_pdl(True)

    ref = chain(False, False)
    for pdl, graph in ((True, False), (True, True), (False, True)):
        got = chain(pdl, graph)
        assert all(torch.equal(a, b) for a, b in zip(ref, got))


@pytest.mark.parametrize("mode,scale", [("fp8", 0.05), ("nvfp4", 168.0), ("mxfp8", 0.0)])
@pytest.mark.parametrize("M", [64, 2048])
def test_pdl_chain_whose_x_is_the_previous_y(gnq, mode, scale, M):
    """A chain in which every call's activation x is the y the previous call
    wrote (and its residual the residual it updated), as when the producing
    kernel writes x: the rows each call prefetches before its wait are still
    being written by its predecessor.  PDL on (eagerly and in a captured
    graph) gives the bits of plain launches, in one-wave and many-wave
    grids."""
    dev = torch.device("cuda")
    H = 4096
    x, r, w = _make(M, H, "bf16", seed=37)
    wd = w.to(dev)
    sd = torch.tensor([scale], device=dev)

    def chain(pdl, graph):
        gnq.set_pdl(pdl)
        try:
            rd = r.to(dev)
            x0 = x.to(dev)
            outs = [gnq.alloc_outputs(M, H, mode, True, x0) for _ in range(4)]
            for o in outs:  # NVFP4 scale padding rows are never written
                if o[1] is not None:
                    o[1].view(torch.uint8).fill_(0xA5)
            def run():
                xi = x0
                for o in outs:
                    gnq.gemma_add_rms_norm_quant(xi, rd, wd, 1e-6, sd, mode, write_y=True, out=o)
                    xi = o[2]  # the next call normalizes this call's y
            if graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    run()
                rd.copy_(r.to(dev))
                for o in outs:
                    o[2].zero_()
                g.replay()
            else:
                run()
            torch.cuda.synchronize()
            return [rd.clone()] + [t.view(torch.uint8).clone() for o in outs for t in o if t is not None]
        finally:
            gnq.set_pdl(True)

    ref = chain(False, False)
    for pdl, graph in ((True, False), (True, True)):
        got = chain(pdl, graph)
        assert all(torch.equal(a, b) for a, b in zip(ref, got))
    assert gnq.read_device_error() == 0


def test_status_codes_with_device_buffers(gnq):
    lib = gnq.load()
    import ctypes
    dev = torch.device("cuda")
    x = torch.zeros(4, 128, dtype=torch.bfloat16, device=dev)
    r = torch.zeros(4, 128, dtype=torch.bfloat16, device=dev)
    w = torch.zeros(128, dtype=torch.bfloat16, device=dev)
    q = torch.zeros(4, 128, dtype=torch.uint8, device=dev)
    s = torch.ones(1, dtype=torch.float32, device=dev)
    P = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)
    call = lib.gemma_add_rms_norm_quant
    # x aliased with residual
    assert call(P(x), P(x), P(w), 1e-6, P(s), 0, 0, P(q), None, None, 4, 128, 0, None) == 5
    # misaligned x
    assert call(P(x, 2), P(r), P(w), 1e-6, P(s), 0, 0, P(q), None, None, 3, 64, 0, None) == 6
    # NVFP4 needs H % 64 == 0
    assert call(P(x), P(r), P(w), 1e-6, P(s), 1, 0, P(q), P(q), None, 4, 96, 0, None) == 2
    # missing scale / block scale
    assert call(P(x), P(r), P(w), 1e-6, None, 0, 0, P(q), None, None, 4, 128, 0, None) == 1
    assert call(P(x), P(r), P(w), 1e-6, P(s), 1, 0, P(q), None, None, 4, 128, 0, None) == 1
    # bad dtype / mode
    assert call(P(x), P(r), P(w), 1e-6, P(s), 0, 0, P(q), None, None, 4, 128, 7, None) == 3
    assert call(P(x), P(r), P(w), 1e-6, P(s), 9, 0, P(q), None, None, 4, 128, 0, None) == 4
    torch.cuda.synchronize()
    assert torch.count_nonzero(r) == 0  # rejected calls had no effect


@pytest.mark.parametrize("M,H,mode,scale,res,write_y", [
    (256, 4096, "fp8", 0.05, True, True),      # the decode batch: one CTA per row
    (40, 5120, "nvfp4", 168.0, True, True),
    (3000, 2048, "fp8", 0.05, False, False),   # would stream on device: host input keeps rows
])
def test_pinned_host_buffers(gnq, M, H, mode, scale, res, write_y):
    """Every buffer in pinned host memory (read and written by the kernels
    through the host link, no copy): the same bits as the device buffers."""
    x, r, w = _make(M, H, "bf16", seed=47)
    r = r if res else None
    s = torch.tensor([scale], dtype=torch.float32)
    outs = {}
    for where in ("cuda", "host"):
        def place(t):
            if t is None:
                return None
            return t.to("cuda") if where == "cuda" else t.clone().pin_memory()
        xd, rd, wd, sd = place(x), place(r), place(w), place(s)
        out = gnq.alloc_outputs(M, H, mode, write_y, xd)
        if mode == "nvfp4":
            out[1].view(torch.uint8).fill_(0xA5)
        # host activations always take the row kernel; run the device side
        # in it too, so both sum the squares in the same order
        with forced_policy(gnq, 1 if where == "cuda" else 0):
            gnq.gemma_add_rms_norm_quant(xd, rd, wd, 1e-6, sd, mode, write_y=write_y, out=out)
        torch.cuda.synchronize()
        outs[where] = [t.cpu().view(torch.uint8) if t.dtype != torch.bfloat16 else t.cpu()
                       for t in out if t is not None] + ([rd.cpu()] if rd is not None else [])
        if where == "host":
            assert all(t.is_pinned() for t in out if t is not None)
    assert all(torch.equal(a, b) for a, b in zip(outs["cuda"], outs["host"]))
    assert gnq.read_device_error() == 0


def test_binding_rejects_bad_buffers(gnq):
    """The binding checks every buffer's size, dtype, layout and placement
    before it launches anything (the C ABI cannot see a buffer's size), so
    a short or mistyped buffer raises instead of being written past."""
    dev = torch.device("cuda")
    M, H = 8, 256
    x = torch.randn(M, H, device=dev).to(torch.bfloat16)
    r = torch.randn(M, H, device=dev).to(torch.bfloat16)
    w = torch.randn(H, device=dev).to(torch.bfloat16)
    s = torch.tensor([168.0], device=dev)
    q, bs, y = gnq.alloc_outputs(M, H, "nvfp4", True, x)
    r0 = r.clone()
    bad = [
        dict(out=(q[:-1], bs, y)),                                   # q one row short
        dict(out=(q, bs.view(torch.uint8)[:-1], y)),                 # scale padding missing
        dict(out=(q, bs, y.float())),                                # y of the wrong dtype
        dict(out=(q, bs, y.t().contiguous().t())),                   # y not contiguous
        dict(out=(q, bs, None)),                                     # y missing with write_y
        dict(weight=w.float()),                                      # weight of the wrong dtype
        dict(weight=w[: H // 2]),                                    # weight too short
        dict(residual=r[: M // 2]),                                  # residual too short
        dict(residual=r.cpu()),                                      # pageable host memory
    ]
    for case in bad:
        kw = dict(out=(q, bs, y), weight=w, residual=r)
        kw.update(case)
        with pytest.raises(ValueError):
            gnq.gemma_add_rms_norm_quant(x, kw["residual"], kw["weight"], 1e-6, s, "nvfp4",
                                         write_y=True, out=kw["out"])
    torch.cuda.synchronize()
    assert torch.equal(r, r0)  # nothing ran
    with pytest.raises(ValueError):
        gnq.gemma_add_rms_norm(x, r, w, 1e-6, y=y[: M // 2])
    with pytest.raises(ValueError):
        gnq.gemma_add_rms_norm_quant_parts(torch.stack([x, x]), r, w, 1e-6, s, "fp8",
                                           out=(q, None, None))              # q sized for NVFP4


@pytest.mark.parametrize("mode,scale,vpt,form,residual", [
    ("fp8", 0.05, 0, 0, False),
    # the packed NVFP4 form agrees on the copies' arrival at its row barrier
    # and stores the new residual after it
    ("nvfp4", 168.0, 4, 2, False),
    ("nvfp4", 168.0, 4, 2, True),
    ("nvfp4", 168.0, 2, 1, True),
])
def test_bounded_wait_gives_up_and_the_next_call_is_clean(gnq, mode, scale, vpt, form, residual):
    """The failure path of the streaming kernel's bounded waits, on the GPU
    without a fault: under the library's test hook every row announces 16
    bytes more than its copies deliver, so no barrier can complete and each
    CTA's first wait runs out (after ~2^20 cycles).  The kernel must set the
    timeout bit of the device error word, complete its barriers itself with
    one more valid copy, and return without writing any output (codes,
    scales, y, the residual); the next normal call must then pass the whole
    parity contract."""
    dev = torch.device("cuda")
    M, H = 700, 2048
    x, r, w = _make(M, H, "bf16", seed=61, residual=residual)
    xd, wd = x.to(dev), w.to(dev)
    rd = None if r is None else r.to(dev)
    sd = torch.tensor([scale], device=dev)
    assert gnq.read_device_error(clear=True) == 0
    q, bs, y = gnq.alloc_outputs(M, H, mode, True, xd)
    for t in (q, bs, y):
        if t is not None:
            t.view(torch.uint8).fill_(0xA5)
    with forced_policy(gnq, 2, 0, vpt, form):
        gnq.inject_wait_timeout(True)
        try:
            gnq.gemma_add_rms_norm_quant(xd, rd, wd, 1e-6, sd, mode, write_y=True, out=(q, bs, y))
            torch.cuda.synchronize()
        finally:
            gnq.inject_wait_timeout(False)
        assert gnq.read_device_error(clear=True) & 1, "the timeout bit was not set"
        for name, t in (("codes", q), ("scales", bs), ("y", y)):
            if t is not None:
                assert bool((t.view(torch.uint8) == 0xA5).all()), f"a timed-out call wrote {name}"
        if r is not None:
            assert torch.equal(rd.cpu(), r), "a timed-out call wrote the residual"
        run_case(gnq, x, r, w, mode, scale, write_y=True, dtype="bf16")
    assert gnq.read_device_error() == 0


@pytest.mark.parametrize("M,kernel", [(100, 1), (300, 1), (300, 2)])
@pytest.mark.parametrize("mode,scale", [("fp8", 0.05), ("nvfp4", 168.0), ("mxfp8", 0.0)])
def test_constant_weights_flag(gnq, M, kernel, mode, scale):
    """With the constant-weights flag, small batches (one unit per thread on
    the row kernel, M = 100 here) read w and the scale before they wait on
    the preceding kernel; other launches ignore it.  Single calls keep the
    parity contract, and a dependent chain (each call consuming the residual
    the previous one wrote) gives the bits of the default launches."""
    dev = torch.device("cuda")
    x, r, w = _make(M, 4096, "bf16", seed=67)
    gnq.set_constant_weights(True)
    try:
        with forced_policy(gnq, kernel):
            run_case(gnq, x, r, w, mode, scale, write_y=True, dtype="bf16")
    finally:
        gnq.set_constant_weights(False)
    xd, wd = x.to(dev), w.to(dev)
    sd = torch.tensor([scale], device=dev)

    def chain(const_w):
        gnq.set_constant_weights(const_w)
        try:
            rd = r.to(dev)
            outs = [gnq.alloc_outputs(M, 4096, mode, True, xd) for _ in range(4)]
            for o in outs:  # NVFP4 scale rows M..round_up(M, 128) are never written
                if o[1] is not None:
                    o[1].view(torch.uint8).fill_(0xA5)
            with forced_policy(gnq, kernel):
                for o in outs:
                    gnq.gemma_add_rms_norm_quant(xd, rd, wd, 1e-6, sd, mode, write_y=True, out=o)
            torch.cuda.synchronize()
            return [rd.clone()] + [t.view(torch.uint8).clone() for o in outs for t in o
                                   if t is not None]
        finally:
            gnq.set_constant_weights(False)

    assert all(torch.equal(a, b) for a, b in zip(chain(False), chain(True)))
    assert gnq.read_device_error() == 0


@pytest.mark.parametrize("pdl", [True, False])
@pytest.mark.parametrize("M", [64, 2048])
def test_pdl_consumer_reads_the_finished_codes(gnq, pdl, M):
    """The stand-in consumer (launched as a programmatic dependent of each
    call, reading its own weight before it waits and the call's codes after)
    sees every call's final codes, with the calls launched as programmatic
    dependents or not: its checksum equals the one computed on the host from
    the codes."""
    dev = torch.device("cuda")
    H, ctas = 5120, 40
    x, r, w = _make(M, H, "bf16", seed=71)
    xd, wd = x.to(dev), w.to(dev)
    sd = torch.tensor([168.0], device=dev)
    wt = torch.randint(0, 255, (ctas * 4096,), dtype=torch.uint8, device=dev)
    outs, sums, rds = [], [], []
    gnq.set_pdl(pdl)
    try:
        for i in range(3):
            rd = r.to(dev)
            o = gnq.alloc_outputs(M, H, "nvfp4", False, xd)
            s_out = torch.zeros(ctas * 256, dtype=torch.int32, device=dev)
            gnq.gemma_add_rms_norm_quant(xd, rd, wd, 1e-6, sd, "nvfp4", out=o)
            gnq.pdl_consumer(o[0], wt, s_out, ctas)
            outs.append(o)
            sums.append(s_out)
            rds.append(rd)
        torch.cuda.synchronize()
    finally:
        gnq.set_pdl(True)

    def host_checksum(q_bytes):
        n_thr = ctas * 256
        wv = wt.cpu().numpy().view(np.uint32).reshape(-1, 4)
        wx = wv[:, 0] ^ wv[:, 1] ^ wv[:, 2] ^ wv[:, 3]
        acc = np.zeros(n_thr, np.uint32)
        for i0 in range(0, wx.size, n_thr):
            seg = wx[i0:i0 + n_thr]
            acc[:seg.size] ^= seg
        qv = q_bytes.view(np.uint32).reshape(-1, 4)
        qx = (qv[:, 0] ^ qv[:, 1] ^ qv[:, 2] ^ qv[:, 3]).astype(np.uint64)
        acc = acc.astype(np.uint64)
        for i0 in range(0, qx.size, n_thr):
            seg = qx[i0:i0 + n_thr]
            acc[:seg.size] += seg
        return (acc & 0xFFFFFFFF).astype(np.uint32)

    for o, s_out in zip(outs, sums):
        want = host_checksum(u8(o[0]).reshape(-1))
        assert np.array_equal(s_out.cpu().numpy().view(np.uint32), want)
    run_case(gnq, x, r, w, "nvfp4", 168.0, write_y=False, dtype="bf16")


@pytest.mark.parametrize("kernel", [0, 1, 2])
@pytest.mark.parametrize("M,H,k", [(200, 2048, 1), (700, 4096, 1), (90, 1024, 3)])
def test_nvfp4_16_byte_aligned_buffers(gnq, kernel, M, H, k):
    """NVFP4 calls whose 16-bit tensors are 16-byte but not 32-byte aligned
    (views 8 elements into larger buffers) take the instances without
    256-bit accesses -- the row kernel, whatever shape is forced -- and give
    the bits of the same call on 32-byte aligned buffers."""
    dev = torch.device("cuda")
    x, r, w = _make(M, H, "bf16", seed=73, k=k)
    sd = torch.tensor([168.0], device=dev)

    def off16(t):
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=dev)
        v = buf[8:].view(t.shape)
        v.copy_(t.to(dev))
        assert v.data_ptr() % 32 == 16
        return v

    results = []
    for place in (lambda t: t.to(dev).clone(), off16):
        xd, rd, wd = place(x), place(r), place(w)
        yb = torch.empty(M * H + 8, dtype=torch.bfloat16, device=dev)
        y = yb[8:].view(M, H) if place is off16 else yb[:M * H].view(M, H)
        q, bs, _ = gnq.alloc_outputs(M, H, "nvfp4", False, xd)
        bs.view(torch.uint8).fill_(0xA5)
        with forced_policy(gnq, kernel):
            if k > 1:
                gnq.gemma_add_rms_norm_quant_parts(xd, rd, wd, 1e-6, sd, "nvfp4", write_y=True,
                                                   out=(q, bs, y))
            else:
                gnq.gemma_add_rms_norm_quant(xd, rd, wd, 1e-6, sd, "nvfp4", write_y=True,
                                             out=(q, bs, y))
        torch.cuda.synchronize()
        results.append([rd.cpu(), y.cpu(), q.cpu(), bs.view(torch.uint8).cpu()])
    (r_a, y_a, q_a, s_a), (r_b, y_b, q_b, s_b) = results
    assert torch.equal(r_a, r_b)
    if kernel != 2:
        # the same launch shape on both sides: the same bits everywhere
        assert torch.equal(y_a, y_b) and torch.equal(q_a, q_b) and torch.equal(s_a, s_b)
    else:
        # the forced streaming shape fell back to the row kernel on the
        # misaligned side, which sums the squares in another order
        assert int(ulp_distance16(bits(y_a), bits(y_b)).max()) <= 1
    # and the misaligned call passes the whole contract against the oracle
    with forced_policy(gnq, kernel):
        run_case(gnq, x, r, w, "nvfp4", 168.0, write_y=True, dtype="bf16")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("mode,scale", [("fp8", 0.08), ("nvfp4", 84.0), ("mxfp8", 0.0)])
@pytest.mark.parametrize("M,H", [(700, 8192), (333, 8192 + 64), (160, 2048)])
def test_streaming_without_residual_or_y(gnq, dtype, mode, scale, M, H):
    """The streaming instances compiled for launches with neither a residual
    nor y (four units per thread, packed form), on rows that are and are not
    a whole number of units per thread: the call without y must give the
    codes of the same launch shape writing y (a generic instance), and the
    whole contract against the oracle."""
    x, _, w = _make(M, H, dtype, seed=M + 3, residual=False)
    with forced_policy(gnq, 2, 0, 4, 2):
        run_case(gnq, x, None, w, mode, scale, write_y=False, dtype=dtype)
    assert gnq.read_device_error() == 0
