"""Builds libdsa.so in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libdsa.so")
SOURCES = [os.path.join(CSRC, f) for f in ("dsa_api.cu", "dsa_diag.cu", "dsa_proj.cu", "dsa_policy.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("dsa_decode.cuh", "dsa_ptx.cuh", "dsa_tc.cuh", "dsa_internal.h")] + [
    os.path.join(ROOT, "include", h) for h in ("dsa.h", "dsa_diag.h", "dsa_proj.h", "dsa_policy.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdsa.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles libdsa.so if it is missing or older than its sources."""
    os.makedirs(LIBDIR, exist_ok=True)
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(p) for p in DEPS)
        if os.path.getmtime(LIB) >= newest:
            return LIB
    tag = f".tmp{os.getpid()}"
    base = [nvcc(), "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC"]
    if verbose:
        base.insert(1, "-Xptxas=-v")
    # one object per translation unit, compiled in parallel, then linked
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(LIBDIR, os.path.basename(src) + tag + ".o")
        cmd = base + ["-c", "-o", obj, src]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
        objs.append(obj)
    errors = []
    for cmd, p in procs:
        out, err = p.communicate()
        if p.returncode != 0:
            errors.append(f"nvcc failed ({' '.join(cmd)}):\n{err}")
        elif verbose:
            print(err)
    try:
        if errors:
            raise RuntimeError("\n".join(errors))
        tmp = LIB + tag
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc link failed ({' '.join(cmd)}):\n{res.stderr}")
        os.replace(tmp, LIB)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
