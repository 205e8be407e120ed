"""The C ABI on the CPU: the library loads, exports every function the public
header declares, and rejects bad arguments before making any CUDA call (so
these run without a GPU)."""
import ctypes
import os
import re

import pytest

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import build as bld

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "selscan.h")

F32, BF16 = 0, 1


@pytest.fixture(scope="module")
def lib():
    bld.build()
    return ss.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(selscan_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("selscan_fwd", "selscan_step", "selscan_last_error", "selscan_check_device_error",
              "selscan_release_workspace", "selscan_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/selscan.h but not exported"


def test_version(lib):
    assert "sm_103a" in ss.version()


def fwd(lib, x=0x10000, delta=0x20000, A=0x30000, B=0x40000, C=0x50000, y=0x60000,
        Bsz=1, L=8, D=4, N=4, dtype=F32, sp=1, h0=None, hT=None):
    return lib.selscan_fwd(x, delta, A, B, C, y, Bsz, L, D, N, dtype, sp, h0, hT, None)


# Fake, well-separated device addresses: every call below must fail in the
# argument checks, which run before any CUDA call.
@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), ss.ERR_INVALID_ARG),
    (dict(Bsz=-1), ss.ERR_INVALID_ARG),
    (dict(L=-5), ss.ERR_INVALID_ARG),
    (dict(D=-2), ss.ERR_INVALID_ARG),
    (dict(N=0), ss.ERR_INVALID_ARG),
    (dict(N=65), ss.ERR_UNSUPPORTED),
    (dict(A=None), ss.ERR_INVALID_ARG),
    (dict(x=None), ss.ERR_INVALID_ARG),
    (dict(y=None), ss.ERR_INVALID_ARG),
    (dict(C=None), ss.ERR_INVALID_ARG),
    (dict(x=0x10002), ss.ERR_INVALID_ARG),                 # misaligned fp32
    (dict(y=0x40000 + 4), ss.ERR_INVALID_ARG),             # y overlaps B
    (dict(y=0x10000 + 4), ss.ERR_INVALID_ARG),             # y overlaps x partially
    (dict(hT=0x30000), ss.ERR_INVALID_ARG),                # hT overlaps A
    (dict(h0=0x70000, hT=0x70000 + 8), ss.ERR_INVALID_ARG),  # partial h0/hT overlap
    (dict(Bsz=1 << 40, L=1 << 30, D=1 << 20), ss.ERR_INVALID_ARG),  # size overflow
])
def test_fwd_argument_errors(lib, kw, code):
    assert fwd(lib, **kw) == code
    assert ss.last_error() != ""


def test_fwd_empty_problem_is_ok_without_cuda(lib):
    assert fwd(lib, Bsz=0) == ss.OK
    assert fwd(lib, D=0, A=None) == ss.OK
    assert ss.last_error() == ""


@pytest.mark.parametrize("kw,code", [
    (dict(N=0), ss.ERR_INVALID_ARG),
    (dict(N=100), ss.ERR_UNSUPPORTED),
    (dict(Bsz=-3), ss.ERR_INVALID_ARG),
    (dict(state=None), ss.ERR_INVALID_ARG),
    (dict(y=0x10000), ss.ERR_INVALID_ARG),                 # y overlaps state
    (dict(y=0x20000), ss.ERR_INVALID_ARG),                 # y overlaps x
    (dict(state=0x30000), ss.ERR_INVALID_ARG),             # state overlaps A
    (dict(x=0x20001), ss.ERR_INVALID_ARG),                 # misaligned
])
def test_step_argument_errors(lib, kw, code):
    a = dict(state=0x10000, x=0x20000, delta=0x28000, A=0x30000, B=0x40000, C=0x50000,
             y=0x60000, Bsz=2, D=4, N=16)
    a.update(kw)
    rc = lib.selscan_step(a["state"], a["x"], a["delta"], a["A"], a["B"], a["C"], a["y"],
                          a["Bsz"], a["D"], a["N"], None)
    assert rc == code


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(ss, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(ss, "_lib", None)
    with pytest.raises(ImportError):
        ss.lib()
