"""Build libselscan.so in-tree for sm_103a with nvcc.

    python -m selective_state_space_157_b300.build [--verbose]

The library is built beside this file so that it travels with the source
tree; the Python binding loads it from here and nowhere else.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libselscan.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


# The backward pass's own sources, and the file that puts the library's one
# translation unit together; the forward, decode and conv1d kernels and their
# host code do not depend on them.
BACKWARD_ONLY = ("scan_bwd.cuh", "selscan_bwd.cu", "libselscan.cu")


def source_digest(backward: bool = False) -> str:
    """sha256 over the CUDA sources a kernel is built from (identifies the
    kernels a profile was taken on; the public header's comments do not change
    them). The forward, decode and conv1d kernels leave out the backward's
    own files; the backward kernel takes every source."""
    import hashlib
    h = hashlib.sha256()
    for p in sources():
        if p.endswith(".py") or p.endswith(".h"):
            continue
        if not backward and os.path.basename(p) in BACKWARD_ONLY:
            continue
        h.update(os.path.basename(p).encode())
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    cmd = [NVCC, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-cudart", "shared", "-I", INCLUDE, "-I", CSRC,
           "-o", LIB + ".tmp", os.path.join(CSRC, "libselscan.cu")]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if verbose:
        sys.stderr.write(r.stdout + r.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose="--verbose" in sys.argv)
    print(LIB)
