"""Build libwenc.so in-tree with nvcc for sm_103a (no CMake, no torch extension machinery).

    python -m transformer_encoder_gb300.build                 # incremental
    python -m transformer_encoder_gb300.build --force         # rebuild everything
    python -m transformer_encoder_gb300.build --bounds-check  # the index-checked library (below)

Each .cu under csrc/ compiles to an object in parallel; the objects link into
transformer_encoder_gb300/_lib/libwenc.so with the CUDA runtime linked statically, so the
library loads on a host without a GPU driver (the driver is resolved only when a CUDA
call needs it).

With bounds_check, the same sources compile with -DWENC_BOUNDS_CHECK into
_build_bounds/ and _lib/libwenc_bounds.so: every index check in the kernels is live (an access
whose index falls outside its buffer is skipped and recorded in the device error word, which
wenc_sync_status reports as WENC_ERR_CUDA with the check's site). The binding loads it instead of
libwenc.so when WENC_LIBRARY names it.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libwenc.so")
BUILD_BOUNDS = os.path.join(PKG, "_build_bounds")
LIB_BOUNDS = os.path.join(LIBDIR, "libwenc_bounds.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libwenc.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, extra, verbose: bool):
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, bounds_check: bool = False) -> str:
    """Compile csrc/*.cu and link libwenc.so (libwenc_bounds.so with bounds_check); returns the
    library path."""
    build_dir, lib_path = (BUILD_BOUNDS, LIB_BOUNDS) if bounds_check else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    hdrs = headers()
    jobs = []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        if force or ptxas_info or _stale(obj, [src, *hdrs]):
            jobs.append((src, obj))
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DWENC_BOUNDS_CHECK"] if bounds_check else [])
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            futs = {ex.submit(_compile, s, o, extra, verbose): s for s, o in jobs}
            for fu in cf.as_completed(futs):
                msg = fu.result()
                if ptxas_info and msg:
                    print(f"== {os.path.basename(futs[fu])}\n{msg}", flush=True)
    objs = [os.path.join(build_dir, os.path.basename(s)[:-3] + ".o") for s in sources()]
    if force or jobs or _stale(lib_path, objs):
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", lib_path, *objs, "-lpthread", "-ldl", "-lrt"]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib_path


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers / spills / smem per kernel")
    ap.add_argument("--bounds-check", action="store_true", help="build the index-checked libwenc_bounds.so")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_info=a.ptxas_info, bounds_check=a.bounds_check))


if __name__ == "__main__":
    sys.exit(main())
