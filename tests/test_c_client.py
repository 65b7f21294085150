"""A plain C11 program against include/rdx.h and librdx.so: the boundary is a
C ABI (no C++, no PyTorch types).  Compiled on the CPU; run on the GPU."""
import os
import shutil
import subprocess

import pytest

from reduction_rdx_sum_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "rdx_client.c")
EXE = os.path.join(ROOT, "_build", "rdx_client")


def compile_client() -> str:
    build.build()
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    os.makedirs(os.path.dirname(EXE), exist_ok=True)
    pkg = os.path.dirname(build.LIB)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O1", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), SRC, "-o", EXE, "-L", pkg, "-lrdx",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{pkg}",
                    f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"], check=True)
    return EXE


def test_header_is_c_and_client_links():
    assert os.path.exists(compile_client())


@pytest.mark.gpu
def test_c_client_runs():
    exe = compile_client()
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c client ok" in r.stdout
