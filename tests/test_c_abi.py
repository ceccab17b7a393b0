"""The C ABI from a plain C program (no Python or torch on the call path):
compiled with gcc against include/gemma_nq.h, linked to the in-tree
libgemma_nq.so and the CUDA runtime, and run on the GPU."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_c_program_compiles_against_the_header(tmp_path):
    """CPU: the header is valid C and the program links against the library."""
    from nvfp4_quant_gemma_gb300 import build
    lib = build.build()
    exe = tmp_path / "abi_smoke"
    cuda = _cuda_home()
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", os.path.join(ROOT, "tests", "c", "abi_smoke.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", os.path.dirname(lib), "-lgemma_nq", "-L", os.path.join(cuda, "lib64"),
           "-lcudart", "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)]
    subprocess.run(cmd, check=True)
    assert exe.exists()


@pytest.mark.gpu
def test_c_program_runs(tmp_path):
    from nvfp4_quant_gemma_gb300 import build
    lib = build.build()
    exe = tmp_path / "abi_smoke"
    cuda = _cuda_home()
    subprocess.run(["gcc", "-std=c99", os.path.join(ROOT, "tests", "c", "abi_smoke.c"),
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    "-L", os.path.dirname(lib), "-lgemma_nq", "-L", os.path.join(cuda, "lib64"),
                    "-lcudart", "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr + res.stdout
    assert "c abi ok" in res.stdout
