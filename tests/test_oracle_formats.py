"""Pins of the oracle's number-format routines against things other than
itself: library casts (torch, numpy), golden tables from the format
definitions, and an independent per-binade rounding formulation."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gnq_testutil import bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# --- 16-bit activation formats -------------------------------------------------

def test_decode16_bf16_all_patterns_match_torch(oracle_lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = oracle.decode16(pats, oracle.BF16)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def test_decode16_fp16_all_patterns_match_numpy(oracle_lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = oracle.decode16(pats, oracle.FP16)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def _fp32_sweep(rng, n):
    """fp32 values over the whole exponent range, plus exact bf16/fp16 ties."""
    mant = rng.uniform(1.0, 2.0, n)
    exp = rng.integers(-140, 128, n)
    sign = rng.choice([-1.0, 1.0], n)
    v = (sign * np.ldexp(mant, exp)).astype(np.float32)
    # bf16 midpoints: a bf16 value plus half of its spacing (exact in fp32)
    b = rng.integers(0, 0x7F7F, 4096).astype(np.uint16)
    bv = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    ties = np.nextafter(bv, np.float32(np.inf)).astype(np.float32)
    ties_exact = (bv.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    return np.concatenate([v, ties, ties_exact, -ties_exact,
                           np.array([0.0, -0.0, 3.3895314e38, 3.39e38, 1e-45], np.float32)])


def test_round16_bf16_matches_torch_cast(oracle_lib):
    rng = np.random.default_rng(0)
    v = _fp32_sweep(rng, 200000)
    ref = bits(torch.from_numpy(v).to(torch.bfloat16))
    got = oracle.round16(v.astype(np.float64), oracle.BF16)
    assert np.array_equal(ref, got)


def test_round16_fp16_matches_numpy_cast(oracle_lib):
    rng = np.random.default_rng(1)
    mant = rng.uniform(1.0, 2.0, 200000)
    exp = rng.integers(-27, 17, 200000)
    v = np.ldexp(mant, exp) * rng.choice([-1.0, 1.0], 200000)
    # exact fp16 midpoints and their neighbours
    h = rng.integers(0, 0x7BFF, 4096).astype(np.uint16).view(np.float16).astype(np.float64)
    spacing = np.spacing(h.astype(np.float16)).astype(np.float64)
    mids = h + spacing / 2
    v = np.concatenate([v, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                        [65504.0, 65519.99, 65520.0, 1e6, 2.0**-25, 2.0**-25 * 1.0000001]])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    got = oracle.round16(v, oracle.FP16)
    assert np.array_equal(ref, got)


def test_round16_bf16_is_nearest_for_fp64_inputs(oracle_lib):
    """Brute force on doubles that fp32 cannot hold: the result is the nearer
    of the two bf16 neighbours, the even one on a tie."""
    rng = np.random.default_rng(2)
    v = rng.standard_normal(20000) * np.ldexp(1.0, rng.integers(-30, 30, 20000))
    got = oracle.round16(v, oracle.BF16)
    gv = oracle.decode16(got, oracle.BF16)
    # neighbours of the result on the bf16 line
    up = oracle.decode16((got.astype(np.int32) + 1).astype(np.uint16), oracle.BF16)
    dn = oracle.decode16((got.astype(np.int32) - 1).astype(np.uint16), oracle.BF16)
    err = np.abs(gv - v)
    assert np.all(err <= np.abs(up - v))
    assert np.all(err <= np.abs(dn - v))


# --- FP8 E4M3 ------------------------------------------------------------------

def test_e4m3_values_all_codes_match_torch(oracle_lib):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_cast_in_range(oracle_lib):
    rng = np.random.default_rng(3)
    # every midpoint between neighbouring finite codes, and its fp32 neighbours
    vals = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    rand = (rng.uniform(-1, 1, 100000) * np.ldexp(1.0, rng.integers(-12, 9, 100000))).astype(np.float32)
    v = np.concatenate([mids, -mids, np.nextafter(mids, np.float32(0)),
                        np.nextafter(mids, np.float32(1e9)), rand,
                        np.float32([463.99997, 448.0, 0.0, -0.0])])
    v = v[np.abs(v) < 464]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(v.astype(np.float64))
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates_and_keeps_nan(oracle_lib):
    big = np.array([464.0, 480.0, 1e6, 3e38, math.inf])
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    assert oracle.e4m3_encode(np.array([math.nan]))[0] & 0x7F == 0x7F
    # the sign survives a zero result
    assert oracle.e4m3_encode(np.array([-0.0, -1e-9]))[0] == 0x80
    assert oracle.e4m3_encode(np.array([-0.0, -1e-9]))[1] == 0x80


# --- FP4 E2M1 ------------------------------------------------------------------

def test_e2m1_table_golden(oracle_lib):
    for code, val in _read_rows("e2m1_table.txt"):
        got = oracle.e2m1_value(int(code))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e2m1_rounding_golden(oracle_lib):
    rows = _read_rows("e2m1_rounding.txt")
    v = np.array([float(r[0]) for r in rows])
    want = np.array([int(r[1]) for r in rows])
    assert np.array_equal(oracle.e2m1_encode(v), want)


def _e2m1_by_binade(v):
    """Independent formulation: inside each binade the E2M1 values sit on an
    even grid (0.5 below 2, 1 in [2, 4), 2 in [4, 6]); rounding to the grid
    with numpy's rint (ties to even) is ties-to-even on the code."""
    a = np.abs(v)
    r = np.where(a < 2.0, np.rint(a / 0.5) * 0.5,
                 np.where(a < 4.0, np.rint(a), np.rint(a / 2.0) * 2.0))
    r = np.minimum(r, 6.0)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    code = np.searchsorted(mags, r)
    return (code | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def test_e2m1_encode_matches_binade_rint(oracle_lib):
    rng = np.random.default_rng(4)
    v = rng.uniform(-8, 8, 200000)
    grid = np.arange(-800, 801) / 100.0  # includes every tie point
    v = np.concatenate([v, grid, np.nextafter(grid, 100), np.nextafter(grid, -100)])
    assert np.array_equal(oracle.e2m1_encode(v), _e2m1_by_binade(v))


def test_e8m0_values(oracle_lib):
    assert oracle.e8m0_value(127) == 1.0
    assert oracle.e8m0_value(0) == 2.0 ** -127
    assert oracle.e8m0_value(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_value(255))
    codes = np.arange(255, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).double().numpy()
    assert np.array_equal(ref, [oracle.e8m0_value(int(c)) for c in codes])
