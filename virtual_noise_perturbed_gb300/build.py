"""Build ``libvn.so`` in-tree with nvcc for sm_103a (GB300).

Usage: ``python -m virtual_noise_perturbed_gb300.build [--force] [-v]``.

Each ``csrc/*.cu`` file is compiled in parallel to ``_build/*.o`` and the
objects are linked into ``virtual_noise_perturbed_gb300/libvn.so`` (CUDA
runtime linked statically; the driver API is reached through the runtime's
entry-point query, so no link against libcuda is needed). A rebuild happens
only when a source or header is newer than the library. Builds take a file lock,
so processes that start together (the ranks of one job, test workers) build
once: the others wait, then find the library current.
"""

from __future__ import annotations

import argparse
import concurrent.futures as cf
import fcntl
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libvn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libvn.so")


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) \
        + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return r


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile and link libvn.so unless it is current; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with open(os.path.join(BUILD, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and up_to_date():  # another process built it while this one waited
                return LIB
            _compile_and_link(verbose, extra_flags)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)
    return LIB


def _compile_and_link(verbose: bool, extra_flags) -> None:
    cc = nvcc()
    flags = CFLAGS + list(extra_flags or [])
    objs, cmds = [], []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmds.append([cc, *ARCH, *flags, "-c", src, "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=min(len(cmds), os.cpu_count() or 4)) as ex:
        list(ex.map(lambda c: _run(c, verbose), cmds))
    tmp = LIB + ".tmp"
    _run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"], verbose)
    os.replace(tmp, LIB)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers / spills per kernel")
    a = ap.parse_args(argv)
    extra = ["-Xptxas", "-v"] if a.ptxas_info else []
    print(build(force=a.force or a.ptxas_info, verbose=a.verbose or a.ptxas_info, extra_flags=extra))
    return 0


if __name__ == "__main__":
    sys.exit(main())
