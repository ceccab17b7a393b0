"""Python binding of libgemma_nq.so: argument marshalling only.

Every step of the operation runs in the library's CUDA kernels; this module
checks tensor metadata, allocates outputs with PyTorch the way
"vllm.models.qwen3_5.nvidia.ops.fused_norm_quant" (gemma_add_rms_norm_quant)
does, passes raw pointers (CUDA or pinned host memory) and the current CUDA
stream through ctypes,
and turns a nonzero status into an exception.  There is no fallback: if the
library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

GNQ_OK = 0
_DTYPE = {torch.bfloat16: 0, torch.float16: 1}
_MODES = {"none": -1, "fp8": 0, "nvfp4": 1, "mxfp8": 2}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load the in-tree libgemma_nq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        P, i64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        sigs = {
            "gemma_add_rms_norm": [P, P, P, F, P, i64, i64, I, P],
            "gemma_add_rms_norm_quant": [P, P, P, F, P, I, I, P, P, P, i64, i64, I, P],
            "gemma_add_rms_norm_quant_parts": [P, I, i64, P, P, F, P, I, I, P, P, P, i64, i64, I, P],
            "add_rms_norm_quant": [P, I, i64, P, P, F, P, I, I, P, P, P, i64, i64, I, P],
            "gnq_set_launch_policy": [I, I, I, I],
            "gnq_query_launch": [i64, i64, I, I, I, I, I, F, P, P, P, P],
            "gnq_read_device_error": [P, I],
            "gnq_set_pdl": [I],
            "gnq_set_constant_weights": [I],
            "gnq_inject_wait_timeout": [I],
            "gnq_quantize_fp8_values": [P, i64, P, P, P],
            "gnq_pdl_consumer": [P, i64, P, i64, P, I, P],
            "gnq_encode_e4m3_e2m1": [P, i64, P, P, P],
        }
        for name, argt in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = argt
            fn.restype = ctypes.c_int
        lib.gnq_status_string.argtypes = [ctypes.c_int]
        lib.gnq_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


# Names the C ABI exports (checked by the test suite against include/gemma_nq.h).
EXPORTS = ("gemma_add_rms_norm", "gemma_add_rms_norm_quant", "gemma_add_rms_norm_quant_parts",
           "add_rms_norm_quant", "gnq_status_string", "gnq_set_launch_policy",
           "gnq_read_device_error", "gnq_set_pdl", "gnq_encode_e4m3_e2m1",
           "gnq_quantize_fp8_values", "gnq_query_launch", "gnq_set_constant_weights",
           "gnq_inject_wait_timeout", "gnq_pdl_consumer")


def status_string(status: int) -> str:
    return load().gnq_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != GNQ_OK:
        raise RuntimeError(f"{what}: {status_string(status)} (status {status})")


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _mode(mode) -> int:
    if isinstance(mode, bool):  # the pages' signature: nvfp4=True / False
        return _MODES["nvfp4"] if mode else _MODES["fp8"]
    if isinstance(mode, str):
        return _MODES[mode]
    return int(mode)


def _reachable(t: torch.Tensor) -> bool:
    """A tensor the GPU can address: CUDA memory or pinned (mapped) host memory."""
    return t.is_cuda or t.is_pinned()


def _check_act(x: torch.Tensor, name: str) -> None:
    if not _reachable(x) or not x.is_contiguous() or x.dtype not in _DTYPE:
        raise ValueError(f"{name} must be a contiguous bf16/fp16 tensor in CUDA or pinned memory")


def _check_buf(t, name: str, nbytes: int, dtype=None, required: bool = True) -> None:
    """A buffer the kernels read or write: contiguous, of `dtype` if given, at
    least `nbytes` long, in CUDA or pinned memory.  Raises before any launch
    (the library itself cannot see a buffer's size)."""
    if t is None:
        if required:
            raise ValueError(f"{name} is required here")
        return
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes; the call needs {nbytes}")
    if not _reachable(t):
        raise ValueError(f"{name} must be in CUDA or pinned host memory")


def _check_call(M: int, H: int, k: int, dt, residual, weight, mode: int, write_y: bool, out):
    """Sizes of every buffer a call touches (x itself checked by the caller)."""
    e = 2
    _check_buf(residual, "residual", M * H * e, dt, required=False)
    _check_buf(weight, "weight", H * e, dt)
    q, bs, y = out
    if mode in (0, 2):
        _check_buf(q, "q", M * H)
    elif mode == 1:
        _check_buf(q, "q", M * H // 2)
    if mode == 1:
        _check_buf(bs, "block_scale", round_up(M, 128) * round_up(H // 16, 4))
    elif mode == 2:
        _check_buf(bs, "block_scale", M * (H // 32))
    if write_y or mode == -1:
        _check_buf(y, "y", M * H * e, dt)


def round_up(a: int, b: int) -> int:
    return (a + b - 1) // b * b


def alloc_outputs(M: int, H: int, mode, write_y: bool, like: torch.Tensor):
    """(q, block_scale, y) buffers as the pages allocate them; block_scale is
    None for FP8 (whose block scale is the static scale tensor).  Placed like
    `like`: on its CUDA device, or in pinned host memory for a host tensor."""
    m = _mode(mode)
    kw = {"device": like.device} if like.is_cuda else {"pin_memory": True}
    q = bs = None
    if m in (0, 2):
        q = torch.empty((M, H), dtype=torch.float8_e4m3fn, **kw)
    elif m == 1:
        q = torch.empty((M, H // 2), dtype=torch.uint8, **kw)
    if m == 1:
        bs = torch.empty((round_up(M, 128), round_up(H // 16, 4) // 4), dtype=torch.int32,
                         **kw).view(torch.float8_e4m3fn)
    elif m == 2:
        bs = torch.empty((M, H // 32), dtype=torch.uint8, **kw)
    y = torch.empty((M, H), dtype=like.dtype, **kw) if (write_y or m == -1) else None
    return q, bs, y


def gemma_add_rms_norm(x, residual, weight, eps, y=None, stream=None):
    """Residual add + Gemma RMSNorm.  Returns (y, residual); residual (if
    given) is updated in place to x + residual."""
    _check_act(x, "x")
    M, H = x.shape
    if y is None:
        y = torch.empty_like(x) if x.is_cuda else torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    _check_call(M, H, 1, x.dtype, residual, weight, -1, True, (None, None, y))
    st = load().gemma_add_rms_norm(_ptr(x), _ptr(residual), _ptr(weight), float(eps), _ptr(y),
                                   M, H, _DTYPE[x.dtype], _stream(stream))
    _check(st, "gemma_add_rms_norm")
    return y, residual


def _scale_ptr(scale):
    if scale is None:
        return None
    if not (_reachable(scale) and scale.dtype == torch.float32 and scale.numel() == 1):
        raise ValueError("scale must be a 1-element fp32 tensor in CUDA or pinned memory")
    return _ptr(scale)


def gemma_add_rms_norm_quant(x, residual, weight, eps, scale, nvfp4=False, write_y=False,
                             out=None, stream=None):
    """Gemma RMSNorm of x (+ residual) quantized for the next linear.

    ``nvfp4`` may be a bool (the pages' signature) or one of "fp8", "nvfp4",
    "mxfp8".  Returns (q, block_scale, y) like the pages' op: block_scale is
    the swizzled E4M3 scale tensor for NVFP4, the (M, H/32) E8M0 codes for
    MXFP8, and ``scale`` itself for FP8; y is None unless write_y.  ``out``
    may supply preallocated (q, block_scale, y)."""
    _check_act(x, "x")
    M, H = x.shape
    m = _mode(nvfp4)
    q, bs, y = out if out is not None else alloc_outputs(M, H, m, write_y, x)
    _check_call(M, H, 1, x.dtype, residual, weight, m, write_y, (q, bs, y))
    st = load().gemma_add_rms_norm_quant(
        _ptr(x), _ptr(residual), _ptr(weight), float(eps), _scale_ptr(scale), m,
        1 if write_y else 0, _ptr(q), _ptr(bs), _ptr(y), M, H, _DTYPE[x.dtype], _stream(stream))
    _check(st, "gemma_add_rms_norm_quant")
    return q, (scale if m == 0 else bs), (y if write_y else None)


def _parts_call(fn_name, x_parts, residual, weight, eps, scale, mode, write_y, out, stream):
    if x_parts.dim() == 2:
        x_parts = x_parts.unsqueeze(0)
    if not _reachable(x_parts) or not x_parts.is_contiguous() or x_parts.dtype not in _DTYPE:
        raise ValueError("x_parts must be a contiguous bf16/fp16 tensor (k, M, H) in CUDA or "
                         "pinned memory")
    k, M, H = x_parts.shape
    m = _mode(mode)
    q, bs, y = out if out is not None else alloc_outputs(M, H, m, write_y, x_parts)
    _check_call(M, H, k, x_parts.dtype, residual, weight, m, write_y, (q, bs, y))
    st = getattr(load(), fn_name)(
        _ptr(x_parts), k, M * H, _ptr(residual), _ptr(weight), float(eps), _scale_ptr(scale), m,
        1 if (write_y or m == -1) else 0, _ptr(q), _ptr(bs), _ptr(y), M, H,
        _DTYPE[x_parts.dtype], _stream(stream))
    _check(st, fn_name)
    return q, (scale if m == 0 else bs), (y if (write_y or m == -1) else None)


def gemma_add_rms_norm_quant_parts(x_parts, residual, weight, eps, scale, mode, write_y=False,
                                   out=None, stream=None):
    """As gemma_add_rms_norm_quant with the activation given as k partial
    buffers (k, M, H), summed in fp32 on the GPU before the residual add."""
    return _parts_call("gemma_add_rms_norm_quant_parts", x_parts, residual, weight, eps, scale,
                       mode, write_y, out, stream)


def add_rms_norm_quant(x_parts, residual, weight, eps, scale, mode, write_y=False, out=None,
                       stream=None):
    """Plain RMSNorm variant (y = h * rsqrt(mean(h^2) + eps) * w)."""
    return _parts_call("add_rms_norm_quant", x_parts, residual, weight, eps, scale, mode,
                       write_y, out, stream)


def set_launch_policy(kernel: int = 0, cluster: int = 0, vpt: int = 0, form: int = 0) -> None:
    """Force the launch shape (0 = automatic): kernel 1 = row kernel, 2 =
    streaming kernel; cluster = CTAs per row; vpt = units per thread; form
    1 = fp32 (fewest instructions), 2 = packed (fewest registers)."""
    _check(load().gnq_set_launch_policy(int(kernel), int(cluster), int(vpt), int(form)),
           "gnq_set_launch_policy")


def query_launch(M: int, H: int, mode, dtype: str = "bf16", k: int = 1, residual: bool = True,
                 write_y: bool = False, weight_bias: float = 1.0) -> tuple[int, int, int, int]:
    """The automatic launch shape of a call, as (kernel, cluster, vpt, form) in
    set_launch_policy's terms; forcing it reproduces the automatic launch."""
    out = [ctypes.c_int(0) for _ in range(4)]
    dt = {"bf16": 0, "fp16": 1}[dtype] if isinstance(dtype, str) else _DTYPE[dtype]
    _check(load().gnq_query_launch(int(M), int(H), int(k), int(bool(residual)), int(bool(write_y)),
                                   _mode(mode), dt, float(weight_bias),
                                   *[ctypes.byref(o) for o in out]), "gnq_query_launch")
    return tuple(o.value for o in out)


def set_pdl(enable: bool) -> None:
    """Programmatic dependent launch on (default) or off for later calls."""
    _check(load().gnq_set_pdl(1 if enable else 0), "gnq_set_pdl")


def pdl_consumer(q: torch.Tensor, wt: torch.Tensor, out: torch.Tensor, ctas: int,
                 stream=None) -> None:
    """Diagnostic stand-in for the next layer's first kernel: reads wt, waits
    on the preceding kernel, reads q, writes ctas * 256 checksum words."""
    for t, name in ((q, "q"), (wt, "wt")):
        if not (t.is_cuda and t.is_contiguous() and (t.numel() * t.element_size()) % 16 == 0):
            raise ValueError(f"{name} must be a contiguous CUDA tensor of whole 16-byte units")
    if not (out.is_cuda and out.dtype == torch.int32 and out.numel() >= ctas * 256):
        raise ValueError("out must be an int32 CUDA tensor of at least ctas * 256 words")
    _check(load().gnq_pdl_consumer(_ptr(q), q.numel() * q.element_size(), _ptr(wt),
                                   wt.numel() * wt.element_size(), _ptr(out), int(ctas),
                                   _stream(stream)), "gnq_pdl_consumer")


def set_constant_weights(enable: bool) -> None:
    """Read w and the scale before waiting on the preceding kernel (the caller
    guarantees no preceding kernel writes them); off by default."""
    _check(load().gnq_set_constant_weights(1 if enable else 0), "gnq_set_constant_weights")


def inject_wait_timeout(enable: bool) -> None:
    """Test hook: later streaming launches make their bounded waits give up
    (device error bit 1, no outputs written); off by default."""
    _check(load().gnq_inject_wait_timeout(1 if enable else 0), "gnq_inject_wait_timeout")


def read_device_error(clear: bool = True) -> int:
    """The device error word (bit 1: a bounded wait in a kernel gave up)."""
    flags = ctypes.c_uint(0)
    _check(load().gnq_read_device_error(ctypes.byref(flags), 1 if clear else 0),
           "gnq_read_device_error")
    return int(flags.value)


def quantize_fp8_values(y: torch.Tensor, scale: torch.Tensor, stream=None) -> torch.Tensor:
    """The kernels' static-FP8 quantizer on raw fp32 values (diagnostic)."""
    if not (y.is_cuda and y.dtype == torch.float32 and y.is_contiguous()):
        raise ValueError("y must be a contiguous fp32 CUDA tensor")
    q = torch.empty(y.shape, dtype=torch.uint8, device=y.device)
    _check(load().gnq_quantize_fp8_values(_ptr(y), y.numel(), _scale_ptr(scale), _ptr(q),
                                          _stream(stream)), "gnq_quantize_fp8_values")
    return q


def encode_e4m3_e2m1(v: torch.Tensor, stream=None):
    """Hardware E4M3 and E2M1 codes of fp32 values (diagnostic)."""
    if not (v.is_cuda and v.dtype == torch.float32 and v.is_contiguous()):
        raise ValueError("v must be a contiguous fp32 CUDA tensor")
    e4 = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    e2 = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    _check(load().gnq_encode_e4m3_e2m1(_ptr(v), v.numel(), _ptr(e4), _ptr(e2), _stream(stream)),
           "gnq_encode_e4m3_e2m1")
    return e4, e2
