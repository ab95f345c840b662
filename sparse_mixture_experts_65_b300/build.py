"""Builds libmoe.so in-tree from csrc/*.cu for sm_103a (B300) with nvcc, and
its bounds-checked variant libmoe_check.so (the same sources with
-DMOE_CHECK=1: routing-derived indices are range-tested on the device and a
failure is reported as MOE_ERR_BOUNDS by moe_check_status).

Usage:  python -m sparse_mixture_experts_65_b300.build [-v] [--check]
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe.so")
BUILD_CHECK = os.path.join(PKG, "_build_check")
LIB_CHECK = os.path.join(PKG, "libmoe_check.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
SOURCES = ["router.cu", "route.cu", "route_tc.cu", "route_wide.cu", "gemm_tc.cu", "gemm_simt.cu", "combine.cu", "balance.cu", "quant.cu", "moe_api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3",
              "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(INCLUDE, "moe.h"))
    return hs


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=None, ptxas_verbose: bool = False,
          check: bool = False) -> str:
    """Compiles the library (check=True: the bounds-checked variant)."""
    bdir, lib = (BUILD_CHECK, LIB_CHECK) if check else (BUILD, LIB)
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    flags = list(NVCC_FLAGS) + list(extra_flags or []) + (["-DMOE_CHECK=1"] if check else [])
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    hdrs = _headers()
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        if ptxas_verbose or _stale(o, [s] + hdrs):
            jobs.append([cc, *ARCH, *flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_verbose:
                sys.stdout.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    objs = [os.path.join(bdir, s.replace(".cu", ".o")) for s in SOURCES]
    if _stale(lib, objs):
        cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", lib, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose:
            sys.stdout.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv,
                check="--check" in sys.argv))
