"""Pins of the oracle's add + Gemma RMSNorm + quantization pipeline against
hand-worked examples, library routines and invariants of the mathematics.

Each test is chosen so that a plausible slip in the oracle fails it: a dropped
or flipped (1 + w), a wrong divisor in the mean, a dropped eps, a residual that
is not written back or not used, a wrong partial-sum order or precision, a
swapped nibble order, a wrong scale formula or rounding rule."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gnq_testutil import DTYPE_CODE, DTYPES, bits, from_bits, unpack_nibbles

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *vals = line.split()
                d[key] = vals
    return d


def _rand(shape, std, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(DTYPES[dtype])


# --- hand-worked examples ------------------------------------------------------

def test_fp8_row_golden(oracle_lib):
    d = _golden("fp8_row_example.txt")
    H = int(d["H"][0])
    x = bits(torch.full((1, H), float(d["x"][0]), dtype=torch.bfloat16))
    w = bits(torch.full((H,), float(d["w"][0]), dtype=torch.bfloat16))
    out = oracle.gemma_add_rms_norm_quant(x, None, w, float(d["eps"][0]), float(d["scale"][0]),
                                          oracle.MODE_FP8, oracle.BF16, write_y=True)
    assert np.all(out["y"] == int(d["y_bf16_bits"][0], 16))
    assert np.all(out["q"] == int(d["q"][0], 16))


def test_nvfp4_block_golden(oracle_lib):
    d = _golden("nvfp4_block_example.txt")
    y16 = np.array([float(v) for v in d["y"]])
    # a 64-wide row: the worked block first, then three zero blocks
    y = np.zeros((1, 64))
    y[0, :16] = y16
    yb = bits(torch.tensor(y, dtype=torch.bfloat16))
    q, bs = oracle.quantize_from_y(yb, float(d["g"][0]), oracle.MODE_NVFP4, oracle.BF16)
    assert list(q[0, :8]) == [int(v, 16) for v in d["q"]]
    assert bs.reshape(-1)[oracle.swizzle_offset(0, 0, 4)] == int(d["scale_byte"][0], 16)
    # all-zero blocks: scale 0 and zero codes
    assert np.all(q[0, 8:] == 0)
    for b in range(1, 4):
        assert bs.reshape(-1)[oracle.swizzle_offset(0, b, 4)] == 0


def test_mxfp8_row_example(oracle_lib):
    """Hand-worked MXFP8 row (tests/golden/mxfp8_block_example.txt): scale
    codes from floor(log2(amax)), an E4M3 tie, subnormal codes and a
    half-subnormal tie, an all-zero block, saturation."""
    d = _golden("mxfp8_block_example.txt")
    y = np.zeros((1, 128))
    for b in range(4):
        vals = [float(v) for v in d.get(f"y{b}", [])]
        y[0, 32 * b: 32 * b + len(vals)] = vals
    yt = torch.tensor(y, dtype=torch.bfloat16)
    assert torch.equal(yt.double(), torch.tensor(y))  # every listed value is a bf16
    yt[0, 6] = -0.0                                     # block 0's signed zero
    q, bs = oracle.quantize_from_y(bits(yt), 0.0, oracle.MODE_MXFP8, oracle.BF16)
    for b in range(4):
        assert bs[0, b] == int(d[f"code{b}"][0])
        want = [int(v, 16) for v in d.get(f"q{b}", [])]
        got = list(q[0, 32 * b: 32 * (b + 1)])
        assert got[: len(want)] == want and all(c == 0 for c in got[len(want):])


# --- residual add --------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_residual_written_back_as_rounded_sum(oracle_lib, dtype):
    M, H = 5, 256
    x = _rand((M, H), 1.0, dtype, 1)
    r = _rand((M, H), 3.0, dtype, 2)
    w = _rand((H,), 0.3, dtype, 3)
    out = oracle.gemma_add_rms_norm_quant(bits(x), bits(r), bits(w), 1e-6, 0.05,
                                          oracle.MODE_FP8, DTYPE_CODE[dtype])
    # torch's CPU add of two 16-bit tensors is the correctly rounded sum
    assert np.array_equal(out["residual"], bits(x + r))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_residual_feeds_the_norm(oracle_lib, dtype):
    """norm(x, residual) equals norm(x + residual, no residual)."""
    M, H = 4, 512
    x = _rand((M, H), 1.0, dtype, 4)
    r = _rand((M, H), 2.0, dtype, 5)
    w = _rand((H,), 0.3, dtype, 6)
    c = DTYPE_CODE[dtype]
    a = oracle.gemma_add_rms_norm_quant(bits(x), bits(r), bits(w), 1e-6, 0.0, oracle.MODE_NONE, c)
    b = oracle.gemma_add_rms_norm_quant(bits(x + r), None, bits(w), 1e-6, 0.0, oracle.MODE_NONE, c)
    assert b["residual"] is None
    assert np.array_equal(a["y"], b["y"])


def test_partials_summed_in_fp32_in_index_order(oracle_lib):
    """Partials [2^24, 1, -2^24, 1]: fp32 left to right gives
    (2^24 + 1 -> 2^24, ties to even) - 2^24 + 1 = 1; the exact sum is 2 and
    any other order or a wider accumulator gives 2 or more."""
    H = 64
    parts = np.zeros((4, 1, H))
    parts[:, 0, :] = np.array([2.0 ** 24, 1.0, -(2.0 ** 24), 1.0])[:, None]
    xb = bits(torch.tensor(parts, dtype=torch.bfloat16))
    w = bits(torch.zeros(H, dtype=torch.bfloat16))
    r = bits(torch.zeros(1, H, dtype=torch.bfloat16))
    out = oracle.gemma_add_rms_norm_quant(xb, r, w, 1e-6, 0.0, oracle.MODE_NONE, oracle.BF16)
    assert np.all(oracle.decode16(out["residual"], oracle.BF16) == 1.0)


def test_partials_rounded_once_then_added_to_residual(oracle_lib):
    """With exact sums (small multiples of 2^-4) the partial path reduces to the
    single-buffer path on the exact sum."""
    M, H, k = 3, 128, 4
    g = torch.Generator().manual_seed(7)
    parts = torch.randint(-64, 64, (k, M, H), generator=g).float() / 16
    r = (torch.randint(-64, 64, (M, H), generator=g).float() / 16).to(torch.bfloat16)
    w = _rand((H,), 0.3, "bf16", 8)
    total = parts.sum(0).to(torch.bfloat16)  # exact in fp32, then one rounding
    a = oracle.gemma_add_rms_norm_quant(bits(parts.to(torch.bfloat16)), bits(r), bits(w), 1e-6,
                                        0.05, oracle.MODE_FP8, oracle.BF16)
    b = oracle.gemma_add_rms_norm_quant(bits(total), bits(r), bits(w), 1e-6,
                                        0.05, oracle.MODE_FP8, oracle.BF16)
    for key in ("residual", "y", "q"):
        assert np.array_equal(a[key], b[key])


# --- the norm ------------------------------------------------------------------

def test_unit_rms_with_zero_weight(oracle_lib):
    """w = 0, eps = 0: the output row has mean square 1 (up to bf16 rounding);
    a divisor other than H, or a missing square root, breaks it."""
    M, H = 6, 16
    x = _rand((M, H), 3.0, "bf16", 9)
    w = bits(torch.zeros(H, dtype=torch.bfloat16))
    out = oracle.gemma_add_rms_norm_quant(bits(x), None, w, 0.0, 0.0, oracle.MODE_NONE, oracle.BF16)
    y = oracle.decode16(out["y"], oracle.BF16)
    ms = (y ** 2).mean(axis=1)
    assert np.all(np.abs(ms - 1.0) < 2 * 2.0 ** -8)


def test_matches_unit_vector_from_library_norm(oracle_lib):
    """w = 0, eps = 0: y = x * sqrt(H) / ||x||_2, with the norm from numpy."""
    M, H = 4, 1024
    x = _rand((M, H), 1.0, "bf16", 10)
    w = bits(torch.zeros(H, dtype=torch.bfloat16))
    out = oracle.gemma_add_rms_norm_quant(bits(x), None, w, 0.0, 0.0, oracle.MODE_NONE, oracle.BF16)
    xv = oracle.decode16(bits(x), oracle.BF16)
    ref = xv * math.sqrt(H) / np.linalg.norm(xv, axis=1, keepdims=True)
    got = oracle.decode16(out["y"], oracle.BF16)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)


def test_weight_enters_as_one_plus_w(oracle_lib):
    """y(w = c) / y(w = 0) = 1 + c for a constant weight c."""
    M, H = 3, 256
    x = _rand((M, H), 1.0, "bf16", 11)
    for c in (0.5, -0.75, 2.0):
        w0 = bits(torch.zeros(H, dtype=torch.bfloat16))
        wc = bits(torch.full((H,), c, dtype=torch.bfloat16))
        y0 = oracle.decode16(oracle.gemma_add_rms_norm_quant(bits(x), None, w0, 1e-6, 0.0,
                                                             oracle.MODE_NONE, oracle.BF16)["y"], 0)
        yc = oracle.decode16(oracle.gemma_add_rms_norm_quant(bits(x), None, wc, 1e-6, 0.0,
                                                             oracle.MODE_NONE, oracle.BF16)["y"], 0)
        assert np.all(np.abs(yc - (1 + c) * y0) <= np.abs((1 + c) * y0) * 2.0 ** -7)


def test_plain_rmsnorm_when_weight_bias_zero(oracle_lib):
    """weight_bias = 0 gives the plain RMSNorm: y(w = 1) equals the Gemma y(w = 0)."""
    M, H = 3, 256
    x = _rand((M, H), 1.0, "bf16", 12)
    ones = bits(torch.ones(H, dtype=torch.bfloat16))
    zeros = bits(torch.zeros(H, dtype=torch.bfloat16))
    a = oracle.gemma_add_rms_norm_quant(bits(x), None, ones, 1e-6, 0.0, oracle.MODE_NONE,
                                        oracle.BF16, weight_bias=0.0)
    b = oracle.gemma_add_rms_norm_quant(bits(x), None, zeros, 1e-6, 0.0, oracle.MODE_NONE,
                                        oracle.BF16)
    assert np.array_equal(a["y"], b["y"])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_eps_closed_form_on_constant_row(oracle_lib, dtype):
    """x = c on every element, w = 0: y = c / sqrt(c^2 + eps)."""
    H = 64
    c, eps = 2.0 ** -10, 1e-6
    x = bits(torch.full((1, H), c, dtype=DTYPES[dtype]))
    w = bits(torch.zeros(H, dtype=DTYPES[dtype]))
    out = oracle.gemma_add_rms_norm_quant(x, None, w, eps, 0.0, oracle.MODE_NONE, DTYPE_CODE[dtype])
    want = c / math.sqrt(c * c + float(np.float32(eps)))
    got = oracle.decode16(out["y"], DTYPE_CODE[dtype])
    tol = 2.0 ** (-8 if dtype == "bf16" else -11)
    assert np.all(np.abs(got - want) <= want * tol)
    assert abs(want - 1.0) > 0.1  # eps matters here


def test_zero_row_and_cancelling_weight(oracle_lib):
    H = 64
    z = bits(torch.zeros(2, H, dtype=torch.bfloat16))
    w = bits(torch.zeros(H, dtype=torch.bfloat16))
    out = oracle.gemma_add_rms_norm_quant(z, None, w, 1e-6, 168.0, oracle.MODE_NVFP4, oracle.BF16)
    assert np.all(out["y"] == 0) and np.all(out["q"] == 0)
    flat = out["block_scale"].reshape(-1)
    assert np.all(flat[[oracle.swizzle_offset(m, b, 4) for m in range(2) for b in range(4)]] == 0)
    # w = -1 cancels the Gemma bias: y is a zero of h's sign
    x = torch.tensor([[1.5, -2.0] * (H // 2)], dtype=torch.bfloat16)
    wm = bits(torch.full((H,), -1.0, dtype=torch.bfloat16))
    out = oracle.gemma_add_rms_norm_quant(bits(x), None, wm, 1e-6, 0.02, oracle.MODE_FP8, oracle.BF16)
    assert list(out["y"][0, :2]) == [0x0000, 0x8000]
    assert list(out["q"][0, :2]) == [0x00, 0x80]


# --- quantizers ----------------------------------------------------------------

def _y_sample(M, H, seed, dtype="bf16"):
    g = torch.Generator().manual_seed(seed)
    y = torch.randn(M, H, generator=g) * 3
    y[:, ::97] *= 40  # outliers that saturate
    y[0, :32] = 0.0
    return y.to(DTYPES[dtype])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fp8_codes_match_library_cast(oracle_lib, dtype):
    M, H, s = 8, 512, 0.05
    y = _y_sample(M, H, 13, dtype)
    q, bs = oracle.quantize_from_y(bits(y), s, oracle.MODE_FP8, DTYPE_CODE[dtype])
    assert bs is None
    v = y.float() / torch.tensor(s, dtype=torch.float32)   # fp32 IEEE division
    ref = v.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


@pytest.mark.parametrize("s", [0.03, 0.05])
def test_fp8_is_a_division_over_all_bf16_values(oracle_lib, s):
    """Every finite bf16 y: the oracle's codes equal torch's fp32 y / s cast.
    For s = 0.03 some codes differ from the y * (1/s) form, which pins the
    division reading."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    y = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16)
    y = y[torch.isfinite(y.float())].reshape(1, -1)
    y = y[:, : y.shape[1] // 16 * 16]
    q, _ = oracle.quantize_from_y(bits(y), s, oracle.MODE_FP8, oracle.BF16)
    st = torch.tensor(s, dtype=torch.float32)
    ref = (y.float() / st).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


def _e2m1_grid(v):
    a = np.abs(v)
    r = np.where(a < 2.0, np.rint(a / 0.5) * 0.5,
                 np.where(a < 4.0, np.rint(a), np.rint(a / 2.0) * 2.0))
    r = np.minimum(r, 6.0)
    code = np.searchsorted(np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]), r)
    return (code | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("M", [1, 130])
def test_nvfp4_codes_and_scales_from_library_arithmetic(oracle_lib, dtype, M):
    """Block scale = e4m3(g * (amax / 6)) and codes = e2m1(y * (g / sf)),
    evaluated here with torch fp32 tensor ops and casts, the E2M1 rounding by
    the per-binade grid formulation; scales read back through the layout."""
    H, g = 256, 168.0
    y = _y_sample(M, H, 14, dtype)
    q, bs = oracle.quantize_from_y(bits(y), g, oracle.MODE_NVFP4, DTYPE_CODE[dtype])
    yf = y.float().reshape(M, H // 16, 16)
    amax = yf.abs().amax(dim=2)
    gt = torch.tensor(g, dtype=torch.float32)
    sf32 = gt * (amax / torch.tensor(6.0))
    sf = sf32.clamp(max=448.0).to(torch.float8_e4m3fn)
    sfv = sf.float()
    es = torch.where(sfv == 0, torch.zeros_like(sfv), gt / sfv)
    v = (yf * es[..., None]).reshape(M, H).numpy()
    codes = unpack_nibbles(q)
    assert np.array_equal(codes, _e2m1_grid(v))
    Kp = H // 16
    flat = bs.reshape(-1)
    got_sf = np.array([[flat[oracle.swizzle_offset(m, b, Kp)] for b in range(Kp)] for m in range(M)])
    assert np.array_equal(got_sf, sf.view(torch.uint8).numpy())
    # rows M..round_up(M,128) of the scale tensor are never written
    Mp = oracle.round_up(M, 128)
    written = np.zeros(Mp * Kp, bool)
    for m in range(M):
        for b in range(Kp):
            written[oracle.swizzle_offset(m, b, Kp)] = True
    assert np.all(flat[~written] == oracle.SENTINEL)


def test_nvfp4_dequantized_error_bound(oracle_lib):
    """Decoding code * sf / g lands within half a code step of y (relative to
    the block scale), except where the block's amax saturates the E4M3 range."""
    M, H, g = 16, 512, 168.0
    y = _y_sample(M, H, 15)
    y[:, ::97] /= 40  # keep the block scales below 448
    yb = bits(y)
    q, bs = oracle.quantize_from_y(yb, g, oracle.MODE_NVFP4, oracle.BF16)
    codes = unpack_nibbles(q)
    vals = np.array([oracle.e2m1_value(int(c)) for c in range(16)])[codes]
    flat = bs.reshape(-1)
    Kp = H // 16
    yv = oracle.decode16(yb, oracle.BF16)
    for m in range(M):
        for b in range(Kp):
            sf = oracle.e4m3_value(int(flat[oracle.swizzle_offset(m, b, Kp)]))
            blk = slice(16 * b, 16 * b + 16)
            deq = vals[m, blk] * sf / g
            amax = np.abs(yv[m, blk]).max()
            # the largest E2M1 step is 2 (between 4 and 6): error <= 1 code unit
            assert np.all(np.abs(deq - yv[m, blk]) <= 1.0 * sf / g * 1.0001 + 1e-12)
            # block amax maps to the top of the E2M1 range (4 or 6)
            if amax > 0:
                assert np.abs(vals[m, blk]).max() >= 4.0


def test_mxfp8_scales_and_codes_from_library_arithmetic(oracle_lib):
    """Scale code = floor(log2(amax)) - 8 + 127 (numpy frexp), codes =
    e4m3(y / 2^(code - 127)) via torch's cast with saturation."""
    M, H = 5, 256
    y = _y_sample(M, H, 16)
    q, bs = oracle.quantize_from_y(bits(y), 0.0, oracle.MODE_MXFP8, oracle.BF16)
    yf = y.double().numpy().reshape(M, H // 32, 32)
    amax = np.abs(yf).max(axis=2)
    _, e = np.frexp(amax)
    code = np.where(amax == 0, 0, np.clip(e - 1 - 8 + 127, 0, 254))
    assert np.array_equal(bs, code.astype(np.uint8))
    X = np.ldexp(1.0, code - 127)[..., None]
    ref = torch.from_numpy((yf / X).reshape(M, H)).float().clamp(-448, 448)
    assert np.array_equal(q, ref.to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_mxfp8_infinite_block_takes_the_top_code(oracle_lib):
    """A block whose amax is inf (y overflowed): floor(log2(inf)) = +inf
    clamps to code 254, X = 2^127; inf saturates to 448, finite values
    divided by 2^127 fall below E4M3's smallest subnormal and keep their
    sign (0x00 / 0x80).  The next block is unaffected."""
    y = torch.zeros(1, 64, dtype=torch.bfloat16)
    y[0, 3] = float("inf")
    y[0, 5] = -2.0
    y[0, 40] = 3.0
    q, bs = oracle.quantize_from_y(bits(y), 0.0, oracle.MODE_MXFP8, oracle.BF16)
    assert bs[0, 0] == 254
    assert bs[0, 1] == 1 - 8 + 127           # floor(log2(3)) = 1
    assert q[0, 3] == 0x7E                   # +448
    assert q[0, 5] == 0x80                   # -2 / 2^127 -> -0
    assert q[0, 0] == 0x00
    assert q[0, 40] == 0x7C                  # 3 / 2^(1-8) = 384 = 1.5 * 2^8: exponent field 15, mantissa 100


def test_quantize_from_y_agrees_with_full_pipeline(oracle_lib):
    M, H = 7, 512
    x = _rand((M, H), 1.0, "bf16", 17)
    r = _rand((M, H), 3.0, "bf16", 18)
    w = _rand((H,), 0.3, "bf16", 19)
    for mode, s in ((oracle.MODE_FP8, 0.05), (oracle.MODE_NVFP4, 168.0), (oracle.MODE_MXFP8, 0.0)):
        full = oracle.gemma_add_rms_norm_quant(bits(x), bits(r), bits(w), 1e-6, s, mode,
                                               oracle.BF16, write_y=True)
        q, bs = oracle.quantize_from_y(full["y"], s, mode, oracle.BF16)
        assert np.array_equal(q, full["q"])
        if bs is not None:
            assert np.array_equal(bs, full["block_scale"])
        no_y = oracle.gemma_add_rms_norm_quant(bits(x), bits(r), bits(w), 1e-6, s, mode,
                                               oracle.BF16, write_y=False)
        assert no_y["y"] is None and np.array_equal(no_y["q"], full["q"])


def test_threads_do_not_change_results(oracle_lib):
    M, H = 33, 256
    x = _rand((M, H), 1.0, "fp16", 20)
    r = _rand((M, H), 3.0, "fp16", 21)
    w = _rand((H,), 0.3, "fp16", 22)
    old = oracle.get_threads()
    try:
        oracle.set_threads(1)
        a = oracle.gemma_add_rms_norm_quant(bits(x), bits(r), bits(w), 1e-6, 84.0,
                                            oracle.MODE_NVFP4, oracle.FP16)
        oracle.set_threads(4)
        b = oracle.gemma_add_rms_norm_quant(bits(x), bits(r), bits(w), 1e-6, 84.0,
                                            oracle.MODE_NVFP4, oracle.FP16)
    finally:
        oracle.set_threads(old)
    for key in ("residual", "y", "q", "block_scale"):
        assert np.array_equal(a[key], b[key])
