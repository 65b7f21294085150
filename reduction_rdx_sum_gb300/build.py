"""Build librdx.so (the CUDA library) in-tree for sm_103a.

Each translation unit is compiled by its own nvcc process (in parallel), then
linked into ``reduction_rdx_sum_gb300/librdx.so`` against the shared CUDA
runtime (the one PyTorch has already loaded, when it has).  ptxas resource
usage (registers, spills, shared memory) is written to ``_build/ptxas.txt``.
Nothing is rebuilt while the library is newer than every source and header.

    python -m reduction_rdx_sum_gb300.build [--force] [-DNAME=VALUE ...]
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "librdx.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build librdx.so")
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, defines: list[str] | None = None, out: str = LIB, verbose: bool = False) -> str:
    """Compile and link librdx.so; returns its path."""
    if not force and not defines and out == LIB and up_to_date(out):
        return out
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    extra = list(defines or [])

    def compile_one(src: str):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + f".{os.getpid()}.o")
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    srcs = sources()
    with ThreadPoolExecutor(len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    objs = [o for o, _ in results]
    with open(os.path.join(BUILD, "ptxas.txt"), "w") as f:
        for src, (_, log) in zip(srcs, results):
            f.write(f"== {os.path.basename(src)}\n{log}\n")
    tmp = out + f".tmp{os.getpid()}"
    libdir = _cuda_lib_dir(nvcc)
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           f"-L{libdir}", f"-Xlinker=-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    for o in objs:
        os.remove(o)
    if verbose:
        print(f"built {out}")
    return out


if __name__ == "__main__":
    args = sys.argv[1:]
    defines = [a for a in args if a.startswith("-D")]
    outs = [a.split("=", 1)[1] for a in args if a.startswith("--out=")]
    if defines and not outs:
        raise SystemExit("a build with -D defines needs --out=PATH (the in-tree librdx.so is the default build)")
    build(force="--force" in args, defines=defines, out=outs[0] if outs else LIB, verbose=True)
