"""CPU oracle for the fused Gemma add-RMSNorm + FP8 / NVFP4 input quantization.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` import this package; the product library
never does, and the two share no code.  The arithmetic lives in ``oracle.c``
(plain C11); this module builds it with gcc and marshals numpy arrays.

Parity pins for every function are in ``tests/test_oracle_*.py``.  What each
routine follows on the pages:

* ``gemma_add_rms_norm_quant`` -- "vllm.models.qwen3_5.nvidia.ops.fused_norm_quant",
  ``gemma_add_rms_norm_quant`` (residual updated in place to x + residual,
  norm scaled by (1 + weight), quantized values computed from the
  activation-dtype-rounded normed output, FP8 codes or packed E2M1 with
  swizzled 128x4 E4M3 block scales, rows >= M of the scales left unwritten);
  k-partial input per "...fused_allreduce_norm_quant",
  ``fused_allreduce_gemma_rms_norm_quant`` (partials of a row-parallel linear
  summed with fp32 accumulation).
* ``quantize_from_y`` -- the quantization stage alone, on a given y.
* MXFP8 mode -- "vllm.model_executor.layers.fused_allreduce_gemma_rms_norm",
  ``allreduce_gemma_rms_norm_mxfp8`` (e4m3 values [M, N], row-major E8M0 scales
  [M, N // 32]).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")

BF16, FP16 = 0, 1
MODE_NONE, MODE_FP8, MODE_NVFP4, MODE_MXFP8 = -1, 0, 1, 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (no CUDA involved)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or (
        os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC),
                                     os.path.getmtime(os.path.join(_HERE, "oracle.h"))))
    if force or stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
               "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # GNQ_ORACLE_LIB points the suite at another build of oracle.c; the
        # mutation test uses it to check that the pins catch planted slips.
        lib = ctypes.CDLL(os.environ.get("GNQ_ORACLE_LIB") or build())
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.or_decode16.restype = ctypes.c_double
        lib.or_decode16.argtypes = [ctypes.c_uint16, ctypes.c_int]
        lib.or_round16.restype = ctypes.c_uint16
        lib.or_round16.argtypes = [ctypes.c_double, ctypes.c_int]
        lib.or_e4m3_value.restype = ctypes.c_double
        lib.or_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.or_e4m3_encode.restype = ctypes.c_uint8
        lib.or_e4m3_encode.argtypes = [ctypes.c_double]
        lib.or_e2m1_value.restype = ctypes.c_double
        lib.or_e2m1_value.argtypes = [ctypes.c_uint8]
        lib.or_e2m1_encode.restype = ctypes.c_uint8
        lib.or_e2m1_encode.argtypes = [ctypes.c_double]
        lib.or_e8m0_value.restype = ctypes.c_double
        lib.or_e8m0_value.argtypes = [ctypes.c_uint8]
        lib.or_swizzle_offset.restype = i64
        lib.or_swizzle_offset.argtypes = [i64, i64, i64]
        for name, argt in (("or_decode16_array", [P, P, i64, ctypes.c_int]),
                           ("or_round16_array", [P, P, i64, ctypes.c_int]),
                           ("or_e4m3_encode_array", [P, P, i64]),
                           ("or_e2m1_encode_array", [P, P, i64])):
            fn = getattr(lib, name)
            fn.restype = None
            fn.argtypes = argt
        lib.or_gemma_add_rms_norm_quant.restype = ctypes.c_int
        lib.or_gemma_add_rms_norm_quant.argtypes = [
            P, ctypes.c_int, i64, P, P, ctypes.c_float, ctypes.c_float,
            ctypes.c_float, ctypes.c_int, P, P, P, i64, i64, ctypes.c_int]
        lib.or_quantize_from_y.restype = ctypes.c_int
        lib.or_quantize_from_y.argtypes = [P, ctypes.c_float, ctypes.c_int, P, P,
                                           i64, i64, ctypes.c_int]
        lib.or_set_threads.restype = None
        lib.or_set_threads.argtypes = [ctypes.c_int]
        lib.or_get_threads.restype = ctypes.c_int
        lib.or_get_threads.argtypes = []
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    _load().or_set_threads(int(n))


def get_threads() -> int:
    return _load().or_get_threads()


# --- number formats --------------------------------------------------------

def decode16(bits, dtype: int) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().or_decode16_array(_ptr(b), _ptr(out), b.size, dtype)
    return out


def round16(values, dtype: int) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().or_round16_array(_ptr(v), _ptr(out), v.size, dtype)
    return out


def e4m3_value(code: int) -> float:
    return _load().or_e4m3_value(code)


def e4m3_encode(values) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    _load().or_e4m3_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def e2m1_value(code: int) -> float:
    return _load().or_e2m1_value(code)


def e2m1_encode(values) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    _load().or_e2m1_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def e8m0_value(code: int) -> float:
    return _load().or_e8m0_value(code)


def swizzle_offset(m: int, k: int, Kp: int) -> int:
    return _load().or_swizzle_offset(m, k, Kp)


# --- the method --------------------------------------------------------------

def round_up(a: int, b: int) -> int:
    return (a + b - 1) // b * b


def scale_shape(M: int, H: int, mode: int) -> tuple[int, int]:
    """Byte shape of the block-scale output (NVFP4 swizzled, MXFP8 row-major)."""
    if mode == MODE_NVFP4:
        return round_up(M, 128), round_up(H // 16, 4)
    if mode == MODE_MXFP8:
        return M, H // 32
    return 0, 0


SENTINEL = 0xA5  # fill of the block-scale buffer before a call


def gemma_add_rms_norm_quant(x, residual, w, eps: float, scale: float, mode: int,
                             dtype: int, write_y: bool = True,
                             weight_bias: float = 1.0):
    """Run the oracle over 16-bit bit patterns (numpy uint16).

    ``x`` is (M, H), or (k, M, H) for k partial buffers.  ``residual`` is (M, H)
    or None and is NOT modified; the updated residual is returned.  Returns a
    dict with ``residual`` (updated copy or None), ``y`` (uint16 or None),
    ``q`` and ``block_scale`` (uint8; block_scale is None for FP8 and for
    mode NONE, and is pre-filled with SENTINEL so untouched bytes show).
    """
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if x.ndim == 2:
        k, (M, H) = 1, x.shape
    else:
        k, M, H = x.shape
    r = None if residual is None else np.array(residual, dtype=np.uint16, copy=True, order="C")
    wv = np.ascontiguousarray(w, dtype=np.uint16)
    assert wv.shape == (H,)
    y = np.empty((M, H), np.uint16) if (write_y or mode == MODE_NONE) else None
    q = None
    bs = None
    if mode == MODE_FP8 or mode == MODE_MXFP8:
        q = np.empty((M, H), np.uint8)
    elif mode == MODE_NVFP4:
        q = np.empty((M, H // 2), np.uint8)
    if mode in (MODE_NVFP4, MODE_MXFP8):
        bs = np.full(scale_shape(M, H, mode), SENTINEL, np.uint8)
    rc = lib.or_gemma_add_rms_norm_quant(
        _ptr(x), k, M * H, _ptr(r), _ptr(wv), float(eps), float(weight_bias),
        float(scale), mode, _ptr(q), _ptr(bs), _ptr(y), M, H, dtype)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return {"residual": r, "y": y, "q": q, "block_scale": bs}


def quantize_from_y(y, scale: float, mode: int, dtype: int):
    """Quantize a given (M, H) y (uint16 bit patterns); returns (q, block_scale)."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.uint16)
    M, H = y.shape
    if mode == MODE_NVFP4:
        q = np.empty((M, H // 2), np.uint8)
    else:
        q = np.empty((M, H), np.uint8)
    bs = None
    if mode in (MODE_NVFP4, MODE_MXFP8):
        bs = np.full(scale_shape(M, H, mode), SENTINEL, np.uint8)
    rc = lib.or_quantize_from_y(_ptr(y), float(scale), mode, _ptr(q), _ptr(bs), M, H, dtype)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return q, bs
