"""Build libselscan.so in-tree for sm_103a with nvcc.

    python -m selective_state_space_157_b300.build [--verbose] [--force]

Each ``csrc/*.cu`` file is one translation unit (the host entry points, and
one per kernel family), compiled to an object under ``_build/`` in parallel
and linked into a shared library beside this file, so that it travels with
the source tree; the Python binding loads it from here and nowhere else. An
object is rebuilt when its source or any file it includes is newer.
"""
from __future__ import annotations

import glob
import hashlib
import os
import re
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libselscan.so")
# The benchmark's arithmetic-peak probe, built beside the library but not in it.
PROBE_SRC = os.path.join(CSRC, "probe", "alu_peaks.cu")
PROBE_LIB = os.path.join(PKG, "libselscan_probe.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]

# The translation units each kernel family is compiled from (with the host
# code that plans its launches): the digest of their sources identifies the
# kernels a profile was taken on.
KERNEL_UNITS = {
    "fwd": ("selscan.cu", "fwd_fused_f32_onepass.cu", "fwd_fused_f32_chunked.cu", "fwd_fused_bf16_onepass.cu",
            "fwd_fused_bf16_chunked.cu", "fwd_plain.cu"),
    "step": ("selscan.cu", "step.cu"),
    "conv1d": ("selscan.cu", "conv1d.cu"),
    "bwd": ("selscan_bwd.cu",),
    "ssd": ("ssd.cu",),
}

_INCLUDE_RE = re.compile(r'^\s*#\s*include\s+"([^"]+)"', re.M)


def units():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def sources():
    """Every file the library is built from."""
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def includes(path, seen=None):
    """The file and every project file it includes, transitively."""
    seen = set() if seen is None else seen
    if path in seen or not os.path.exists(path):
        return seen
    seen.add(path)
    for name in _INCLUDE_RE.findall(open(path).read()):
        for d in (os.path.dirname(path), CSRC, INCLUDE):
            cand = os.path.join(d, name)
            if os.path.exists(cand):
                includes(cand, seen)
                break
    return seen


def source_digest(kernel: str = "fwd") -> str:
    """sha256 over the sources a kernel family is built from (its translation
    units and everything they include, except the public header, whose
    comments do not change the kernels)."""
    files = set()
    for u in KERNEL_UNITS[kernel]:
        files |= includes(os.path.join(CSRC, u))
    h = hashlib.sha256()
    for p in sorted(files):
        if os.path.dirname(p) == INCLUDE:
            continue
        h.update(os.path.basename(p).encode())
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def _obj(unit):
    return os.path.join(BUILD, os.path.basename(unit)[:-3] + ".o")


def _stale(unit) -> bool:
    o = _obj(unit)
    if not os.path.exists(o):
        return True
    t = os.path.getmtime(o)
    return any(os.path.getmtime(s) > t for s in includes(unit))


def up_to_date() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(PROBE_LIB):
        return False
    if os.path.getmtime(PROBE_SRC) > os.path.getmtime(PROBE_LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(not _stale(u) and os.path.getmtime(_obj(u)) <= t for u in units())


def build_probe() -> str:
    cmd = [NVCC, *ARCH, *FLAGS, "-shared", "-cudart", "shared", "-o", PROBE_LIB + ".tmp", PROBE_SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on the peak probe:\n" + r.stdout + r.stderr)
    os.replace(PROBE_LIB + ".tmp", PROBE_LIB)
    return PROBE_LIB


def _compile(unit, verbose):
    cmd = [NVCC, *ARCH, *FLAGS, "-c", "-o", _obj(unit) + ".tmp", unit]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(unit)}:\n" + r.stdout + r.stderr)
    os.replace(_obj(unit) + ".tmp", _obj(unit))
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    todo = [u for u in units() if force or _stale(u)]
    probe = force or not os.path.exists(PROBE_LIB) or os.path.getmtime(PROBE_SRC) > os.path.getmtime(PROBE_LIB)
    with ThreadPoolExecutor(max_workers=max(1, min(len(todo) + 1, os.cpu_count() or 4))) as pool:
        pf = pool.submit(build_probe) if probe else None
        logs = list(pool.map(lambda u: _compile(u, verbose), todo))
        if pf is not None:
            pf.result()
    if verbose:
        for log in logs:
            sys.stderr.write(log)
    cmd = [NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", LIB + ".tmp", *[_obj(u) for u in units()]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="--verbose" in sys.argv)
    print(LIB)
