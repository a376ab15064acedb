"""Builds libmoe_gb300.so in-tree with nvcc for sm_103a (no cmake, one -gencode).

Each .cu file compiles to an object in parallel, then one link step makes the
shared library at moe_expert_layer_route_gb300/lib/libmoe_gb300.so. A rebuild
happens only when a source or header is newer than the library.

build(timing=True) makes the diagnostic variant lib/libmoe_gb300_timing.so from the
same sources with MOE_STAGE_TIMING defined (the grouped GEMMs' stage timing; see
stage_timing.py); the shipped library never contains it.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIB_DIR, "libmoe_gb300.so")
TIMING_BUILD = os.path.join(HERE, "_build_timing")
TIMING_LIB = os.path.join(LIB_DIR, "libmoe_gb300_timing.so")

SOURCES = ["moe_api.cu", "route_dispatch.cu", "router.cu", "grouped_gemm.cu",
           "dispatch_noalloc.cu", "ep.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-cudart", "shared", "-Xcompiler", "-fPIC,-O3", "--expt-relaxed-constexpr",
         "-I", CSRC, "-I", INCLUDE]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")
    return cand


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(timing: bool = False) -> bool:
    lib = TIMING_LIB if timing else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(src: str, extra: list[str], build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, timing: bool = False) -> str:
    """Compile the CUDA library if needed; returns the path of the shared library
    (timing=True: the stage-timing diagnostic variant)."""
    lib = TIMING_LIB if timing else LIB
    build_dir = TIMING_BUILD if timing else BUILD
    if not force and up_to_date(timing):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if timing:
        extra.append("-DMOE_STAGE_TIMING")
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-Xlinker",
           "-rpath," + os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64"),
           "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True))
