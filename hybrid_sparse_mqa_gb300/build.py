"""Builds libdsv4attn.so (sm_103a) in the package directory with nvcc.

The library is the whole compute path; the Python binding only loads it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", "dsv4_attn.cu"), os.path.join(PKG, "csrc", "dsv4_kv_store.cu"),
           os.path.join(PKG, "csrc", "dsv4_topk.cu")]
DEPS = SOURCES + [os.path.join(PKG, "csrc", "dsv4_device.cuh"), os.path.join(PKG, "csrc", "dsv4_internal.h"),
                  os.path.join(ROOT, "include", "dsv4attn.h"), os.path.join(ROOT, "include", "dsv4kvstore.h"),
                  os.path.join(ROOT, "include", "dsv4topk.h")]
LIB = os.path.join(PKG, "libdsv4attn.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdsv4attn.so")


def needs_build():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(force=False, verbose=False):
    """Compile the library if it is missing or older than its sources."""
    if not force and not needs_build():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xptxas", "-v",
           "-I", os.path.join(ROOT, "include"), "-Xcompiler", "-fPIC", "-shared",
           *SOURCES, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}) building {LIB}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)
