"""Build libspecverify.so in-tree for sm_103a (GB300) with nvcc.

Each .cu under csrc/ compiles to its own object in parallel, then nvcc links
them into a shared library beside this file. Only the names the public header
declares are exported (-fvisibility=hidden plus explicit default visibility).
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libspecverify.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
# The debug variant: the same sources with device-side index checks compiled
# in (-DSV_DEVICE_CHECKS), built beside the product library.
DEBUG_LIB_PATH = os.path.join(PKG, "libspecverify_debug.so")
DEBUG_FLAGS = ["-DSV_DEVICE_CHECKS=1"]
SOURCES = ["row_stats.cu", "scan.cu", "sample.cu", "filter.cu", "hist.cu", "lmhead.cu", "sv_api.cu",
           "sv_static.cu", "philox.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"),
            shutil.which("nvcc") or ""]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found (set CUDA_HOME)")


def cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    files.append(os.path.join(INCLUDE, "spec_verify.h"))
    return files


def stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in _inputs())


def compile_flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
                   "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
                   *extra]


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile (if needed) and return the library path: the product library,
    or with debug=True the variant with device-side index checks."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    build_dir = os.path.join(BUILD_DIR, "debug") if debug else BUILD_DIR
    if debug:
        extra_flags = (*DEBUG_FLAGS, *extra_flags)
    if not force and not stale(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    objs = []

    def one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *compile_flags(extra_flags), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{p.stdout}\n{p.stderr}")
        return obj, p.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(one, SOURCES))
    for obj, log in results:
        objs.append(obj)
        if verbose and log:
            print(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "shared",
           "-Xlinker", f"-rpath,{cuda_lib_dir()}"]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
