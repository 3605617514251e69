"""Builds libindexer_bwd.so in-tree with nvcc for sm_103a.

Each .cu translation unit compiles in parallel to an object, then nvcc links
the shared library (CUDA runtime linked statically, plain C ABI).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libindexer_bwd.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libindexer_bwd.so")


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    cc = nvcc()
    with tempfile.TemporaryDirectory(prefix="ibwd_build_") as tmp:
        procs = []
        objs = []
        for src in _sources():
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            cmd = [cc, *ARCH, *FLAGS, "-I", INCLUDE, "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
            objs.append(obj)
        errs = []
        for src, pr in procs:
            out, _ = pr.communicate()
            if pr.returncode != 0:
                errs.append(f"{src}:\n{out.decode(errors='replace')}")
            elif verbose and out:
                print(out.decode(errors="replace"))
        if errs:
            raise RuntimeError("nvcc failed:\n" + "\n".join(errs))
        tmp_lib = os.path.join(tmp, "libindexer_bwd.so")
        subprocess.check_call([cc, *ARCH, "-shared", *objs, "-o", tmp_lib])
        shutil.copyfile(tmp_lib, LIB + f".tmp{os.getpid()}")
        os.replace(LIB + f".tmp{os.getpid()}", LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
