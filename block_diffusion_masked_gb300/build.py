"""Build libdfa.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel to an object file under
``_build/``, then linked into ``block_diffusion_masked_gb300/libdfa.so``.
Usage: ``python -m block_diffusion_masked_gb300.build [--verbose-ptxas]``.
"""

from __future__ import annotations

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
LIB = os.path.join(PKG, "libdfa.so")

SOURCES = ["fwd.cu", "fwd2.cu", "bwd2.cu", "aux.cu", "api.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose_ptxas=False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-cudart", "shared",
                "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(srcs, target):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in srcs)


def build(verbose_ptxas=False, force=False, quiet=True):
    """Compile (if out of date) and return the path of libdfa.so."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "dfa.h"))
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or verbose_ptxas or _stale([s] + headers, o):
            jobs.append([nvcc] + _flags(verbose_ptxas) + ["-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failed = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for cmd, r in ex.map(run, jobs):
            if r.returncode != 0:
                failed.append((cmd, r))
            elif not quiet or verbose_ptxas:
                sys.stderr.write(r.stdout + r.stderr)
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + r.stdout + r.stderr for c, r in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    if force or jobs or _stale(objs, LIB):
        tmp = LIB + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    v = "--verbose-ptxas" in sys.argv
    print(build(verbose_ptxas=v, force="--force" in sys.argv, quiet=False))
