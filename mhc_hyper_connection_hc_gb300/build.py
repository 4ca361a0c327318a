"""Build the CUDA library in-tree: mhc_hyper_connection_hc_gb300/_lib/libmhc_gb300.so.

One nvcc per translation unit (run in parallel), then one link.  The only
target is sm_103a (GB300): -gencode arch=compute_103a,code=sm_103a.

build(stamps=True) builds the phase-stamp variant instead, with -DHC_STAMPS, as
_lib/stamps/libmhc_gb300_stamps.so: the same library, whose cluster pre kernel also
writes %globaltimer stamps at phase boundaries into the workspace (see hc_internal.cuh).

build(bounds=True) builds the bounds-checked variant, with -DHC_DEBUG_BOUNDS, as
_lib/bounds/libmhc_gb300_bounds.so: the cluster, helper and wide kernels check each
global output store against its buffer's size and report a refused store in the status word instead
of performing it (see hc_internal.cuh).
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libmhc_gb300.so")
STAMPS_DIR = os.path.join(OUT_DIR, "stamps")
STAMPS_LIB = os.path.join(STAMPS_DIR, "libmhc_gb300_stamps.so")
BOUNDS_DIR = os.path.join(OUT_DIR, "bounds")
BOUNDS_LIB = os.path.join(BOUNDS_DIR, "libmhc_gb300_bounds.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "--expt-relaxed-constexpr", "-I" + INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps() + [__file__])


def build(force: bool = False, verbose: bool = False, extra_flags=(), stamps: bool = False,
          bounds: bool = False) -> str:
    if stamps and bounds:
        raise ValueError("build one variant at a time: stamps or bounds")
    lib, out_dir = (STAMPS_LIB, STAMPS_DIR) if stamps else (BOUNDS_LIB, BOUNDS_DIR) if bounds else (LIB, OUT_DIR)
    if stamps:
        extra_flags = list(extra_flags) + ["-DHC_STAMPS"]
    if bounds:
        extra_flags = list(extra_flags) + ["-DHC_DEBUG_BOUNDS"]
    if not force and not _stale(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + NVCC_FLAGS + list(extra_flags) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose=True, extra_flags=sys.argv[1:]))
