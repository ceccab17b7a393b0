"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports every
symbol the header declares, and rejects bad arguments on the host before any
CUDA call.  No call here reaches a kernel launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemma_nq.h")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_quant_gemma_gb300 import build
    build.build()
    import nvfp4_quant_gemma_gb300 as pkg
    return pkg.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    for n in ("gemma_add_rms_norm", "gemma_add_rms_norm_quant", "gemma_add_rms_norm_quant_parts",
              "add_rms_norm_quant", "gnq_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from nvfp4_quant_gemma_gb300 import _binding
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in gemma_nq.h but not exported"
    assert set(names) == set(_binding.EXPORTS)


def test_status_strings(lib):
    lib.gnq_status_string.restype = ctypes.c_char_p
    texts = {lib.gnq_status_string(i).decode() for i in range(8)}
    assert len(texts) == 8
    assert lib.gnq_status_string(99).decode() == "unknown status"


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails validation


@pytest.mark.parametrize("args,status", [
    # (M, H, dtype, mode, x, residual, w, scale, q, bs, y, write_y) -> status
    ((0, 64, 0, 1, None, None, None, None, None, None, None, 1), 0),   # empty batch: no launch
    ((4, 64, 2, 0, FAKE, None, FAKE, FAKE, FAKE, None, None, 0), 3),   # dtype
    ((4, 64, 0, 3, FAKE, None, FAKE, FAKE, FAKE, None, None, 0), 4),   # mode
    ((4, 60, 0, 0, FAKE, None, FAKE, FAKE, FAKE, None, None, 0), 2),   # H % 8
    ((4, 96, 0, 1, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, 0), 2),   # NVFP4 H % 64
    ((4, 48, 0, 2, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, 0), 2),   # MXFP8 H % 32
    ((4, 65544, 0, 0, FAKE, None, FAKE, FAKE, FAKE, None, None, 0), 2),  # H too large
    ((-1, 64, 0, 0, FAKE, None, FAKE, FAKE, FAKE, None, None, 0), 2),  # M < 0
    ((4, 64, 0, 0, None, None, FAKE, FAKE, FAKE, None, None, 0), 1),   # x NULL
    ((4, 64, 0, 0, FAKE, None, FAKE, None, FAKE, None, None, 0), 1),   # scale NULL
    ((4, 64, 0, 1, FAKE, None, FAKE, FAKE, FAKE, None, None, 0), 1),   # block_scale NULL
    ((4, 64, 0, 0, FAKE, None, FAKE, FAKE, FAKE, None, None, 1), 1),   # y NULL with write_y
    ((4, 64, 0, 0, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 0), 5),   # x == residual
    ((4, 64, 0, 0, ctypes.c_void_p(0x10002), None, FAKE, FAKE, FAKE, None, None, 0), 6),  # align
])
def test_host_validation(lib, args, status):
    M, H, dt, mode, x, r, w, s, q, bs, y, wy = args
    got = lib.gemma_add_rms_norm_quant(x, r, w, ctypes.c_float(1e-6), s, mode, wy, q, bs, y,
                                       ctypes.c_int64(M), ctypes.c_int64(H), dt, None)
    assert got == status


def test_parts_validation(lib):
    f = lib.gemma_add_rms_norm_quant_parts
    args = lambda k, stride: (FAKE, k, ctypes.c_int64(stride), None, FAKE, ctypes.c_float(1e-6),
                              FAKE, 0, 0, FAKE, None, None, ctypes.c_int64(4), ctypes.c_int64(64),
                              0, None)
    assert f(*args(0, 256)) == 4    # k < 1
    assert f(*args(9, 256)) == 4    # k > 8
    assert f(*args(4, 255)) == 6    # stride below M*H
    assert f(*args(4, 260)) == 6    # stride not a multiple of 8
    assert lib.gnq_set_launch_policy(0, 3, 0, 0) == 2
    assert lib.gnq_set_launch_policy(0, 0, 3, 0) == 2
    assert lib.gnq_set_launch_policy(3, 0, 0, 0) == 2
    assert lib.gnq_set_launch_policy(0, 0, 0, 3) == 2
    assert lib.gnq_set_launch_policy(0, 0, 0, 0) == 0
    assert lib.gnq_read_device_error(None, 0) == 1


def test_query_launch_validation(lib):
    """gnq_query_launch rejects what a call would reject (before any device
    query), and fails with GNQ_ERR_CUDA only for a valid call."""
    q = lib.gnq_query_launch
    outs = [ctypes.c_int(0) for _ in range(4)]
    ptrs = [ctypes.byref(o) for o in outs]
    i64, f = ctypes.c_int64, ctypes.c_float

    def call(M=256, H=4096, k=1, res=1, wy=1, mode=0, dt=0, bias=1.0, p=ptrs):
        return q(i64(M), i64(H), k, res, wy, mode, dt, f(bias), *p)

    assert call(p=[None] + ptrs[1:]) == 1      # NULL output
    assert call(dt=2) == 3                     # dtype
    assert call(mode=3) == 4                   # mode
    assert call(k=9) == 4                      # partial count
    assert call(M=0) == 2                      # rows
    assert call(H=100) == 2                    # H % 8
    assert call(mode=1, H=96) == 2             # NVFP4 H % 64
    assert call(H=65544) == 2                  # H too large
    assert call() in (0, 7)                    # valid: a shape, or no device here


def test_switches_and_diagnostics_validate_their_arguments(lib):
    """The process-wide switches accept only their documented values, the
    tuning hook only its documented sets, and the stand-in consumer rejects
    bad sizes and missing buffers -- all on the host, before any CUDA call.
    Valid switch values are restored to the defaults afterwards."""
    P = ctypes.c_void_p
    for fn in (lib.gnq_set_pdl, lib.gnq_set_constant_weights, lib.gnq_inject_wait_timeout):
        assert fn(2) == 2 and fn(-1) == 2
        assert fn(0) == 0
    assert lib.gnq_set_pdl(1) == 0                              # back to the default
    assert lib.gnq_set_launch_policy(3, 0, 0, 0) == 2            # kernel
    assert lib.gnq_set_launch_policy(2, 3, 0, 0) == 2            # rows per CTA not a power of 2
    assert lib.gnq_set_launch_policy(2, 16, 0, 0) == 2           # more than 8
    assert lib.gnq_set_launch_policy(1, 0, 3, 0) == 2            # units per thread
    assert lib.gnq_set_launch_policy(1, 0, 0, 3) == 2            # form
    assert lib.gnq_set_launch_policy(2, 2, 0, 0) == 0            # streaming, >= 2 rows per CTA
    assert lib.gnq_set_launch_policy(0, 0, 0, 0) == 0
    c = lib.gnq_pdl_consumer
    i64 = ctypes.c_int64
    buf = P(4096)  # never dereferenced: every call below is rejected first
    assert c(buf, i64(24), buf, i64(16), buf, 1, None) == 2      # q bytes not a multiple of 16
    assert c(buf, i64(16), buf, i64(-16), buf, 1, None) == 2     # negative weight bytes
    assert c(buf, i64(16), buf, i64(16), buf, 0, None) == 2      # no CTA
    assert c(buf, i64(16), buf, i64(16), None, 1, None) == 1     # no output
    assert c(None, i64(16), buf, i64(16), buf, 1, None) == 1     # no codes


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    from nvfp4_quant_gemma_gb300 import _binding, build
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        _binding.load()


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "nvfp4_quant_gemma_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "oracle.h" not in text and "liboracle" not in text, f
