"""Builds the CUDA library ``libtbe_gb300.so`` in the package directory.

Every ``csrc/*.cu`` translation unit is compiled for sm_103a in parallel (nvcc), then linked
against the shared CUDA runtime, so the library shares the runtime (and thus the current
device and streams) with any other CUDA user in the process.

``build(checked=True)`` makes the debug flavour ``libtbe_gb300_checked.so`` (objects in
``_build_checked/``): the same sources with ``-DTBE_CHECKED=1``, whose kernels range-check the
indices they derive from data and count failures in ``TBE_STAT_CHECK_FAILED`` instead of
accessing out of bounds.  Same C-ABI; load it with ``load(path=CHECKED_LIB_PATH)``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libtbe_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
CHECKED_BUILD_DIR = os.path.join(PKG, "_build_checked")
CHECKED_LIB_PATH = os.path.join(PKG, "libtbe_gb300_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the TBE CUDA library cannot be built")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(checked: bool = False) -> bool:
    lib = CHECKED_LIB_PATH if checked else LIB_PATH
    if not os.path.exists(lib):
        return False
    newest = max(os.path.getmtime(p) for p in sources() + _headers() + [__file__])
    return os.path.getmtime(lib) >= newest


def build(force: bool = False, jobs: int | None = None, verbose: bool = False,
          checked: bool = False) -> str:
    """Compiles and links the library (the TBE_CHECKED flavour with ``checked``) unless it is
    up to date; returns its path."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    build_dir = CHECKED_BUILD_DIR if checked else BUILD_DIR
    flags = NVCC_FLAGS + (["-DTBE_CHECKED=1"] if checked else [])
    if not force and up_to_date(checked):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    srcs = sources()

    newest_header = max([os.path.getmtime(h) for h in _headers()] + [os.path.getmtime(__file__)])

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        if (not force and os.path.exists(obj)
                and os.path.getmtime(obj) >= max(os.path.getmtime(src), newest_header)):
            return obj
        cmd = [nvcc, *ARCH, *flags, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=jobs or min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
            "-Xlinker", f"-rpath,{_cuda_lib_dir(nvcc)}"]
    if verbose:
        print(" ".join(link), flush=True)
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv))
