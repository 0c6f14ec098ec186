"""In-tree build of libw4a16.so for GB300 (sm_103a) with nvcc; no cmake, no torch extension."""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "libw4a16.so")
# the same library with every kernel's index checks compiled in (W4A16_DEBUG_BOUNDS)
DEBUG_LIB_PATH = os.path.join(PKG, "libw4a16_debug.so")

SOURCES = ["w4a16_api.cu", "repack.cu", "gemv.cu", "tc_gemm.cu", "act.cu", "w4a8.cu"]
HEADERS = [os.path.join(CSRC, "common.cuh"), os.path.join(CSRC, "internal.h"), os.path.join(INCLUDE, "w4a16.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libw4a16")


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile every CUDA source for sm_103a (in parallel) and link libw4a16.so in the package
    (debug_bounds: libw4a16_debug.so, the same sources with W4A16_DEBUG_BOUNDS)."""
    bdir = os.path.join(BUILD_DIR, "debug_bounds") if debug_bounds else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug_bounds else LIB_PATH
    defs = ["-DW4A16_DEBUG_BOUNDS"] if debug_bounds else []
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    objs = []
    jobs = []
    for src in SOURCES:
        srcp = os.path.join(CSRC, src)
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [srcp] + HEADERS):
            cmd = [cc] + ARCH + FLAGS + defs + (["-Xptxas", "-v"] if verbose else []) + ["-c", srcp, "-o", obj]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failures = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr)
            if r.returncode != 0:
                failures.append(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if failures:
        raise RuntimeError("libw4a16 compilation failed:\n" + "\n".join(failures))
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + ".tmp"
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("libw4a16 link failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
