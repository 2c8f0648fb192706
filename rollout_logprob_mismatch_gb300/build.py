"""Builds libtim.so in-tree with nvcc for sm_103a (GB300) only.

    python -m rollout_logprob_mismatch_gb300.build [--force] [--ptxas-verbose]

Translation units compile in parallel into ``_build/``; the shared library
links the CUDA runtime statically and no other CUDA library, so it loads on a
machine without a GPU (the CPU tests check its exported symbols).  The same
sources compiled with -DTIM_DEBUG give ``libtim_debug.so`` (``_build/debug/``),
whose kernels also check their indices, TMA coordinates and input contracts
and record the first violation (``tim_debug_violation``).
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libtim.so")
DEBUG_LIB = os.path.join(PKG, "libtim_debug.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          "--expt-relaxed-constexpr", "-Werror", "all-warnings", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libtim.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _build_one(lib: str, objdir: str, extra: list, force: bool, ptxas_verbose: bool, quiet: bool):
    """Starts the compiles of one library; returns a function that waits for
    them and links (so both libraries' compiles run at once)."""
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                     + glob.glob(os.path.join(INCLUDE, "*.h")))
    os.makedirs(objdir, exist_ok=True)
    exe = nvcc()
    procs = []
    objs = []
    for s in srcs:
        o = os.path.join(objdir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or ptxas_verbose or _stale(o, [s] + headers):
            cmd = [exe] + ARCH + CFLAGS + extra + (["-Xptxas", "-v"] if ptxas_verbose else []) + ["-c", s, "-o", o]
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))

    def finish() -> str:
        failed = []
        for cmd, p in procs:
            out, _ = p.communicate()
            text = out.decode(errors="replace")
            if p.returncode != 0:
                failed.append(" ".join(cmd) + "\n" + text)
            elif text.strip() and (ptxas_verbose or not quiet):
                sys.stderr.write(text)
        if failed:
            raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
        if force or _stale(lib, objs):
            tmp = lib + ".%d.tmp" % os.getpid()
            cmd = [exe] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + ["-lpthread", "-ldl", "-lrt"]
            r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
            if r.returncode != 0:
                raise RuntimeError("link failed:\n" + " ".join(cmd) + "\n" + r.stdout.decode(errors="replace"))
            os.replace(tmp, lib)
        return lib

    return finish


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True, debug: bool = True) -> str:
    """Builds libtim.so (and, unless debug=False, libtim_debug.so); returns
    the path of libtim.so."""
    release = _build_one(LIB, BUILD, [], force, ptxas_verbose, quiet)
    checked = _build_one(DEBUG_LIB, os.path.join(BUILD, "debug"), ["-DTIM_DEBUG"], force, False, quiet) \
        if debug else None
    path = release()
    if checked is not None:
        checked()
    return path


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, ptxas_verbose=a.ptxas_verbose, quiet=False))


if __name__ == "__main__":
    main()
