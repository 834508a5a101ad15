"""In-tree build of the CUDA library (``libspecv.so``) for sm_103a.

One translation unit (``csrc/specv.cu``) compiled by nvcc with the CUDA
runtime linked statically; the result sits next to this file, where the
binding loads it.  Rebuilt when any source or the public header is newer.
"""
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libspecv.so")
SOURCES = sorted(glob.glob(os.path.join(PKG, "csrc", "*.cu")) + glob.glob(os.path.join(PKG, "csrc", "*.cuh")))
HEADER = os.path.join(ROOT, "include", "specv.h")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecv.so")


def needs_build():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in SOURCES + [HEADER])


def build(force=False, verbose=False):
    """Compile libspecv.so if missing or stale; return its path."""
    if not force and not needs_build():
        return LIB
    tmp = LIB + ".tmp"
    cmd = [
        nvcc_path(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
        "-o", tmp, os.path.join(PKG, "csrc", "specv.cu"),
    ]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
