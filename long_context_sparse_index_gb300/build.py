"""Builds libdsa.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit under csrc/ is compiled in parallel to an object
in _build/, then linked (static CUDA runtime) into libdsa.so next to this
file.  Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdsa.so")
# measurement variant: the persistent indexer records one globaltimer trace
# record per work item (DSA_ITEM_TRACE) and the tcgen05 forward sums each warp
# role's cycles per pipeline segment (DSA_FWD_PROFILE); nothing else differs
BUILD_TRACE = os.path.join(HERE, "_build_trace")
LIB_TRACE = os.path.join(HERE, "libdsa_trace.so")
# the same item stamps without the indexer's SM-cycle counters, whose clock
# reads in the fold loop make the trace build spill more and run slower: its
# per-item times are the default build's
BUILD_STAMPS = os.path.join(HERE, "_build_stamps")
LIB_STAMPS = os.path.join(HERE, "libdsa_stamps.so")
# checking variant: range checks on gathered rows and shared-memory offsets
# that record a device status (DSA_ERR_INTERNAL) instead of trapping
# (DSA_DEBUG); the arithmetic and results are the default build's
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libdsa_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I", INCLUDE] + ARCH


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, trace: bool = False, debug: bool = False,
          stamps: bool = False) -> str:
    """Compile and link libdsa.so (or, with trace=True, the measurement
    variant libdsa_trace.so, with stamps=True its stamps-only form
    libdsa_stamps.so, or with debug=True the range-checking variant
    libdsa_debug.so); returns its path."""
    if trace + debug + stamps > 1:
        raise ValueError("build: the trace, stamps and debug variants are separate builds")
    lib, bdir = (LIB_TRACE, BUILD_TRACE) if trace else (LIB_STAMPS, BUILD_STAMPS) if stamps else \
        (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and not _stale(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    flags = NVCC_FLAGS + (["-DDSA_ITEM_TRACE=1", "-DDSA_FWD_PROFILE=1"] if trace or stamps else []) + \
        (["-DDSA_TRACE_STAMPS_ONLY=1"] if stamps else []) + (["-DDSA_DEBUG=1"] if debug else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
