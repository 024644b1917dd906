"""Build libfa_gb300.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` file compiles to an object in parallel; the objects link into
``exact_io_aware_28_gb300/libfa_gb300.so`` against the shared CUDA runtime.  No
cmake, no torch extension machinery: the library has a plain C ABI.

    python -m exact_io_aware_28_gb300.build [--verbose-ptxas]
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libfa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libfa_gb300.so")


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return r.returncode, r.stdout


def build(verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                    "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    cc = nvcc()
    cmds = []
    objs = []
    for s in srcs:
        obj = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
        objs.append(obj)
        cmds.append([cc] + flags + ["-c", s, "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=jobs or min(8, len(cmds))) as ex:
        results = list(ex.map(_run, cmds))
    failed = False
    for cmd, (rc, out) in zip(cmds, results):
        if out.strip() and (rc != 0 or verbose_ptxas):
            sys.stderr.write(out)
        if rc != 0:
            failed = True
            sys.stderr.write(f"FAILED: {' '.join(cmd)}\n")
    if failed:
        raise RuntimeError("nvcc failed; see the messages above")
    tmp = LIB + ".tmp"
    rc, out = _run([cc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs +
                   ["-Xlinker", "-rpath,/usr/local/cuda/lib64"])
    if rc != 0:
        sys.stderr.write(out)
        raise RuntimeError("link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose-ptxas", action="store_true")
    a = ap.parse_args()
    print(build(a.verbose_ptxas))
