"""Arithmetic claims the CUDA kernels rely on, checked exhaustively on the CPU
with exact rational arithmetic (no GPU, no oracle).

The NVFP4 block scale is g * (amax / 6): two fp32 operations, the first a
division of the block's largest magnitude by 6.  The kernel computes it as
q0 = RN(amax * RN(1/6)), rem = RN(amax - 6 q0) in one fused multiply-add,
q1 = RN(q0 + rem * RN(1/6)) in another, and uses q1 for every finite amax
with no range check (only inf is special-cased).  amax is the magnitude of a
16-bit value, so the claim can be checked for all of them: q1 must equal the
correctly rounded amax / 6 for every finite non-negative bf16 and fp16 value.
"""
from fractions import Fraction

import numpy as np
import pytest

F32_MIN_EXP = -126  # smallest normal exponent
F32_MANT = 23


def rn32(x: Fraction) -> Fraction:
    """x rounded to the nearest float32 (ties to even), subnormals included."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, F32_MIN_EXP)
    ulp = Fraction(2) ** (e - F32_MANT)
    n = a / ulp
    whole = n.numerator // n.denominator
    frac = n - whole
    if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and whole % 2 == 1):
        whole += 1
    r = whole * ulp
    assert r < Fraction(2) ** 128, "overflow is outside the claim"
    return sign * r


def fma_div6(a: Fraction, r6: Fraction) -> Fraction:
    q0 = rn32(a * r6)
    rem = rn32(a - 6 * q0)   # one fused multiply-add: exact, then one rounding
    return rn32(q0 + rem * r6)


def magnitudes(dtype: str) -> np.ndarray:
    if dtype == "bf16":  # every finite positive bf16 pattern
        return (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    return np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)


def test_rn32_matches_numpy_float32():
    # the rounding helper itself, against the library's float32 division
    rng = np.random.default_rng(5)
    a = rng.standard_normal(200).astype(np.float32) * np.float32(1e3)
    b = rng.standard_normal(200).astype(np.float32)
    got = [rn32(Fraction(float(x)) / Fraction(float(y))) for x, y in zip(a, b)]
    want = (a / b).astype(np.float32)
    assert [Fraction(float(w)) for w in want] == got
    # a subnormal quotient
    x = np.float32(2.0 ** -140)
    assert rn32(Fraction(float(x)) / 3) == Fraction(float(x / np.float32(3)))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fma_corrected_div6_is_correctly_rounded(dtype):
    r6 = rn32(Fraction(1, 6))
    assert r6 == Fraction(float(np.float32(1) / np.float32(6)))
    bad = []
    for v in magnitudes(dtype):
        a = Fraction(float(v))
        if fma_div6(a, r6) != rn32(a / 6):
            bad.append(float(v))
    assert not bad, bad[:5]
    assert fma_div6(Fraction(0), r6) == 0


def test_single_rounding_alone_is_not_enough():
    # without the correction step a third of the values would be off
    r6 = rn32(Fraction(1, 6))
    vals = magnitudes("fp16")[::37]
    off = sum(rn32(Fraction(float(v)) * r6) != rn32(Fraction(float(v)) / 6) for v in vals)
    assert off > len(vals) // 10


# --- MXFP8: the E8M0 scale code read off the exponent field -------------------
#
# The kernel takes code = floor(log2(amax)) - 8 + 127 clamped to [0, 254]
# from the fp32 exponent field e of amax: e - 8 if e > 8, 0 below (zero and
# subnormals), 254 for inf; and divides by the scale with the exact
# multiplier 2^(127 - code), built as the fp32 pattern (254 - code) << 23
# (2^-127, a subnormal, for code 254).

def _kernel_code(amax: np.ndarray) -> np.ndarray:
    e = amax.astype(np.float32).view(np.uint32) >> 23
    return np.where(e == 255, 254, np.where(e > 8, e.astype(np.int64) - 8, 0))


def _definition_code(amax: np.ndarray) -> np.ndarray:
    a = amax.astype(np.float64)
    _, e2 = np.frexp(np.where(np.isinf(a), 1.0, a))
    code = np.clip(e2 - 1 - 8 + 127, 0, 254)
    return np.where(a == 0, 0, np.where(np.isinf(a), 254, code))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_e8m0_code_from_exponent_field(dtype):
    vals = np.concatenate([[0.0], magnitudes(dtype), [np.inf]]).astype(np.float32)
    assert np.array_equal(_kernel_code(vals), _definition_code(vals))


def test_e8m0_inverse_is_the_exact_power_of_two():
    for code in range(255):
        bits = 0x00400000 if code == 254 else (254 - code) << 23
        got = np.array([bits], dtype=np.uint32).view(np.float32)[0]
        assert Fraction(float(got)) == Fraction(2) ** (127 - code)
