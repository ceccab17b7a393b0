"""Shared helpers for the test suite: bit-pattern views and code comparisons.

Holds none of the method's arithmetic."""
from __future__ import annotations

import numpy as np
import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}
DTYPE_CODE = {"bf16": 0, "fp16": 1}


def bits(t: torch.Tensor) -> np.ndarray:
    """16-bit tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray, dtype: str) -> torch.Tensor:
    """numpy uint16 bit patterns -> CPU tensor of the 16-bit dtype."""
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(DTYPES[dtype])


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.uint8).numpy()


def ulp_distance16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in units of the last place between 16-bit patterns of the same
    format (sign-magnitude mapped onto a monotonic integer line; +0 == -0)."""
    def key(x):
        x = x.astype(np.int64)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(key(a) - key(b))


E2M1_MAGS = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_signed_rank(code: np.ndarray) -> np.ndarray:
    """Position of an E2M1 code on the ordered value line, -7..7 (+-0 -> 0)."""
    code = code.astype(np.int64)
    mag = code & 7
    return np.where(code & 8, -mag, mag)


def e4m3_signed_rank(code: np.ndarray) -> np.ndarray:
    """Position of a finite E4M3 code on the ordered value line (+-0 -> 0)."""
    code = code.astype(np.int64)
    mag = code & 0x7F
    return np.where(code & 0x80, -mag, mag)


def unpack_nibbles(q: np.ndarray) -> np.ndarray:
    """(M, H/2) packed bytes -> (M, H) codes, low nibble first."""
    lo = q & 0xF
    hi = q >> 4
    return np.stack([lo, hi], axis=-1).reshape(q.shape[0], q.shape[1] * 2)


def adjacent_codes(a_rank: np.ndarray, b_rank: np.ndarray, n: int | None = None) -> None:
    """End-to-end rule between two code tensors given as value-line ranks:
    every differing code is one step away, and where the tensor holds at
    least 1e5 codes (`n`, default its size) at most 1e-4 of them differ."""
    diff = np.abs(a_rank.astype(np.int64) - b_rank.astype(np.int64))
    assert int(diff.max(initial=0)) <= 1, "an end-to-end code is more than one step off"
    n = diff.size if n is None else n
    if n >= 100000:
        assert np.count_nonzero(diff) <= int(1e-4 * n), \
            f"{np.count_nonzero(diff)} of {n} end-to-end codes differ"


def check_end_to_end(gq: np.ndarray, gbs, ref: dict, om: int) -> None:
    """GPU codes and scales against the oracle's own pipeline (its fp64 y).

    FP8: the E4M3 codes.  NVFP4: the packed E2M1 codes, and the E4M3 block
    scale bytes (both buffers were filled with the same sentinel before the
    calls, so unwritten padding compares equal and only the M * H/16 written
    scales count).  MXFP8: the E8M0 scale codes, then the E4M3 codes of the
    blocks whose two scales agree (a scale one code apart rescales its whole
    block by 2, so those codes are not comparable)."""
    import oracle
    if om == oracle.MODE_FP8:
        adjacent_codes(e4m3_signed_rank(gq), e4m3_signed_rank(ref["q"]))
    elif om == oracle.MODE_NVFP4:
        adjacent_codes(e2m1_signed_rank(unpack_nibbles(gq)),
                       e2m1_signed_rank(unpack_nibbles(ref["q"])))
        M, H = gq.shape[0], 2 * gq.shape[1]
        adjacent_codes(e4m3_signed_rank(gbs.reshape(-1)),
                       e4m3_signed_rank(ref["block_scale"].reshape(-1)), n=M * (H // 16))
    elif om == oracle.MODE_MXFP8:
        ga, gb = gbs.astype(np.int64), ref["block_scale"].astype(np.int64)
        adjacent_codes(ga, gb)
        same = np.repeat(ga == gb, 32, axis=1)
        adjacent_codes(e4m3_signed_rank(gq)[same], e4m3_signed_rank(ref["q"])[same])
