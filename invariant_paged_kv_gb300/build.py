"""Build libpa.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

    python -m invariant_paged_kv_gb300.build [--force] [-v]

Each .cu is compiled to an object in parallel, then linked into
``invariant_paged_kv_gb300/_lib/libpa.so`` with the CUDA runtime linked
statically. Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
BUILDDIR = os.path.join(ROOT, "_build", "pa")
LIB = os.path.join(LIBDIR, "libpa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}")
    if verbose and r.stdout.strip():
        print(r.stdout, flush=True)
    return r.stdout


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every kernel source for sm_103a and link libpa.so. Returns its path."""
    if not force and not ptxas_info and up_to_date():
        return LIB
    os.makedirs(BUILDDIR, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = []
    for src in sources():
        obj = os.path.join(BUILDDIR, os.path.basename(src)[:-3] + ".o")
        jobs.append((src, obj, [cc, "-c", src, "-o", obj] + ARCH + FLAGS + extra))
    outs = {}
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        futs = {ex.submit(_run, cmd, verbose): src for src, _, cmd in jobs}
        for f in cf.as_completed(futs):
            outs[futs[f]] = f.result()
    tmp = LIB + ".tmp"
    _run([cc, "-shared", "-o", tmp] + ARCH + [o for _, o, _ in jobs] +
         ["-cudart", "static", "-Xcompiler", "-fPIC"], verbose)
    os.replace(tmp, LIB)
    if ptxas_info:
        for src in sorted(outs):
            print(f"== {os.path.basename(src)}\n{outs[src]}")
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print -Xptxas -v per source")
    ap.add_argument("-v", "--verbose", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_info=a.ptxas_info))


if __name__ == "__main__":
    sys.exit(main())
