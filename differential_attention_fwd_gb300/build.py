"""Build libdiffattn.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu file under csrc/ is compiled to an object in parallel, then linked
into differential_attention_fwd_gb300/libdiffattn.so.  Objects go to
_build/ at the repository root.  A rebuild happens only when a source or
header is newer than the library.

build(variant="waitprof") makes a second library, libdiffattn_waitprof.so,
from the same sources compiled with -DDIFFATTN_WAIT_PROFILE: its forward
kernel also counts the cycles each warp role spends waiting on barriers
(diffattn_wait_profile reads them).  It is a measurement build only; the
product is libdiffattn.so.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdiffattn.so")
VARIANTS = {
    None: (LIB, BUILD, []),
    "waitprof": (os.path.join(PKG, "libdiffattn_waitprof.so"), os.path.join(BUILD, "waitprof"),
                 ["-DDIFFATTN_WAIT_PROFILE"]),
}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdiffattn.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.h")) +
                               glob.glob(os.path.join(CSRC, "*.cuh")) +
                               glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          variant=None) -> str:
    """Compile and link; returns the library path."""
    lib, objdir, defines = VARIANTS[variant]
    if not force and up_to_date(lib):
        return lib
    cc = nvcc()
    os.makedirs(objdir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + defines

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose or ptxas_info:
        for obj, log in results:
            if log.strip():
                print(f"== {os.path.basename(obj)}\n{log}", file=sys.stderr)
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
