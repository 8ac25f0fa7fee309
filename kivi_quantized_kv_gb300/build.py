"""Builds libkivi.so in-tree for sm_103a with nvcc (no CMake, no torch extension).

Each .cu file under csrc/ compiles to an object in parallel; the objects link
into kivi_quantized_kv_gb300/libkivi.so with the static CUDA runtime.
append.cu is additionally compiled with -fmad=false: its quantizer already
uses explicit round-to-nearest intrinsics, and this keeps any other fp32
expression there from being contracted.

build(debug_checks=True) makes libkivi_debug.so instead, with
-DKIVI_DEBUG_CHECKS=1: the kernels then check every arena address they derive
against the cache region and every input for inf / NaN, and record what they
find in the cache's error word (kivi_read_error) rather than trapping.  The
binding loads it when KIVI_DEBUG_CHECKS=1 is set in the environment.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libkivi.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_PATH_DEBUG = os.path.join(HERE, "libkivi_debug.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "--expt-relaxed-constexpr", "-I", INCLUDE]
PER_FILE = {"append.cu": ["-fmad=false"]}


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkivi.so")


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose_ptxas: bool = False, debug_checks: bool = False) -> str:
    """Compiles and links libkivi.so (libkivi_debug.so with debug_checks) if
    any source is newer than it."""
    lib_path = LIB_PATH_DEBUG if debug_checks else LIB_PATH
    build_dir = BUILD_DEBUG if debug_checks else BUILD
    if not force and not _stale(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nv = nvcc()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if debug_checks:
        extra.append("-DKIVI_DEBUG_CHECKS=1")

    def compile_one(src):
        obj = os.path.join(build_dir, src[:-3] + ".o")
        cmd = [nv, *ARCH, *COMMON, *PER_FILE.get(src, []), *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose_ptxas:
        for _, log in results:
            print(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nv, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose_ptxas="-v" in sys.argv, debug_checks="--debug-checks" in sys.argv))
