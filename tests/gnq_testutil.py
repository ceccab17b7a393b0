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
