"""Build libringattn.so in-tree with nvcc for sm_103a (GB300).

Each .cu file under csrc/ is compiled to an object in parallel, then linked
into online_softmax_merge_gb300/libringattn.so against the shared CUDA runtime.
Rebuilds only when a source or header is newer than the library. With --debug
(build(debug=True)) the same sources become libringattn_debug.so with the
kernels' index checks compiled in (-DRA_DEBUG); the binding loads that library
instead when the environment sets RA_DEBUG=1.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libringattn.so")
# the same sources with the kernels' index checks compiled in (-DRA_DEBUG)
DEBUG_BUILD_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB_PATH = os.path.join(HERE, "libringattn_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin/ on PATH)")


def cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=None,
          debug: bool = False) -> str:
    """Compile and link; returns the library path. debug=True builds
    libringattn_debug.so with the kernels' index checks (-DRA_DEBUG)."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = nvcc_path()
    os.makedirs(build_dir, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I", INCLUDE, "-I", CSRC] + (["-DRA_DEBUG"] if debug else []) + list(
                        extra_flags or [])

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, "-c", src, "-o", obj] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, "-shared", "-cudart", "shared", "-o", tmp] + ARCH + objs + [
        "-Xlinker", "-rpath," + cuda_lib_dir(nvcc)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))
