"""Builds libexact_topk.so in-tree for sm_103a (nvcc + g++, no CMake).

The CUDA translation unit and the host planner compile in parallel; the shared
library links the CUDA runtime dynamically so that it shares one runtime (and
its streams) with PyTorch in the same process.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIBRARY = os.path.join(BUILD_DIR, "libexact_topk.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["topk_kernels.cu", "exact_topk_api.cpp"]
HEADERS = ["etk_internal.h"]


def cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "exact_topk.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    t = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _run(cmd):
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("build step failed: " + " ".join(cmd))
    return res.stdout + res.stderr


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compiles the library if any input changed; returns its path."""
    if not force and not _stale():
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = "nvcc"
    inc = ["-I", INCLUDE, "-I", CSRC]
    obj_cu = os.path.join(BUILD_DIR, "topk_kernels.o")
    obj_api = os.path.join(BUILD_DIR, "exact_topk_api.o")
    cu_cmd = [nvcc, *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "--expt-relaxed-constexpr", *inc, "-c", os.path.join(CSRC, "topk_kernels.cu"),
              "-o", obj_cu]
    if verbose_ptxas:
        cu_cmd.insert(1, "-Xptxas=-v")
    api_cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", *inc,
               "-I", os.path.join(home, "include"), "-c",
               os.path.join(CSRC, "exact_topk_api.cpp"), "-o", obj_api]
    with ThreadPoolExecutor(2) as ex:
        outs = list(ex.map(_run, [cu_cmd, api_cmd]))
    tmp = LIBRARY + f".tmp{os.getpid()}"
    libdir = os.path.join(home, "lib64")
    _run([nvcc, *ARCH_FLAGS, "-shared", "-cudart", "shared", obj_cu, obj_api, "-o", tmp,
          "-Xlinker", f"-rpath={libdir}"])
    os.replace(tmp, LIBRARY)
    if verbose_ptxas:
        sys.stdout.write(outs[0])
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="-v" in sys.argv))
