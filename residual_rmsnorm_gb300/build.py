"""Build the CUDA library libtpar.so in-tree (residual_rmsnorm_gb300/_build).

Each translation unit is compiled by nvcc for sm_103a only, in parallel, then
linked into one shared library against the shared CUDA runtime (so a process
that already loaded PyTorch's libcudart.so.13 keeps a single runtime).
No fast-math: the NVFP4 scale arithmetic must round exactly as IEEE binary32.
"""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libtpar.so")
# The debug variant (-DTPAR_DEBUG: every kernel checks its computed indices
# and reports one out of range through the device error word) builds apart.
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libtpar_debug.so")
SOURCES = ["api.cu"] + [f"kernels_q{q}_{t}.cu" for q in range(4) for t in ("bf16", "fp16")] + [
    "kernels_stream_bf16.cu", "kernels_stream_fp16.cu", "kernels_small.cu", "kernels_grid.cu", "unfused.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtpar.so")


def cuda_lib_dir() -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))
    return os.path.join(root, "lib64")


def flags(debug: bool = False) -> list[str]:
    return ["-std=c++17", "-O3", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O2",
            "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-Xptxas", "-v"] + (["-DTPAR_DEBUG"] if debug else [])


def lib_path(debug: bool = False) -> str:
    return LIB_DEBUG if debug else LIB


def _needs_rebuild(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "tpar.h"), __file__]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link libtpar.so (libtpar_debug.so with ``debug``); returns
    its path. Raises on failure. Processes that build at the same time take
    turns (a file lock); the ones that wait find the library up to date."""
    lib = lib_path(debug)
    if not force and not _needs_rebuild(lib):
        return lib
    out_dir = os.path.dirname(lib)
    os.makedirs(out_dir, exist_ok=True)
    with open(os.path.join(out_dir, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and not _needs_rebuild(lib):
            return lib
        return _build_locked(verbose, debug)


def _build_locked(verbose: bool, debug: bool) -> str:
    cc = nvcc()
    out_dir = os.path.dirname(lib_path(debug))
    LIB_OUT = lib_path(debug)

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [cc, *flags(debug), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    with open(os.path.join(out_dir, "ptxas.log"), "w") as f:
        for _, log in results:
            f.write(log)
    tmp = LIB_OUT + f".tmp{os.getpid()}"
    link = [cc, "-shared", *ARCH, "-cudart", "shared", "-o", tmp, *[o for o, _ in results],
            "-Xlinker", f"-rpath,{cuda_lib_dir()}"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_OUT)
    for obj, _ in results:  # every build recompiles all units: keep only the library
        os.remove(obj)
    if verbose:
        print("built", LIB_OUT)
    return LIB_OUT


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv)
