"""Pins of the oracle's 128x4 swizzled scale layout: hand-worked offsets, a
bijection check, and an independent reshape/transpose construction."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_swizzle_golden_points(oracle_lib):
    with open(os.path.join(GOLDEN, "swizzle_points.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert rows
    for m, k, Kp, off in rows:
        assert oracle.swizzle_offset(int(m), int(k), int(Kp)) == int(off), (m, k, Kp)


@pytest.mark.parametrize("M,H", [(1, 64), (127, 128), (128, 256), (129, 2048), (300, 5120)])
def test_swizzle_is_bijection_and_matches_tiled_transpose(oracle_lib, M, H):
    Mp = oracle.round_up(M, 128)
    Kp = oracle.round_up(H // 16, 4)
    ids = np.arange(Mp * Kp).reshape(Mp, Kp)  # id of (m, k) = m*Kp + k
    # Independent construction of the layout: cut the scale matrix into
    # 128x4 tiles, tile-major along k; within a tile, the 128 rows are split
    # as (4 groups of 32) and stored [m%32][(m%128)/32][k%4].
    tiled = ids.reshape(Mp // 128, 4, 32, Kp // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
    offs = np.empty(Mp * Kp, np.int64)
    for m in range(Mp):
        for k in range(Kp):
            offs[m * Kp + k] = oracle.swizzle_offset(m, k, Kp)
    assert np.array_equal(np.sort(offs), np.arange(Mp * Kp))  # bijection
    assert np.array_equal(offs[tiled], np.arange(Mp * Kp))    # same layout
