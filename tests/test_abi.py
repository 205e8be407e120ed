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


@pytest.mark.parametrize("withhold, wait_ms", [(-1, 0), (0, -1), (1, 2001)])
def test_fault_injection_hook_checks_its_arguments(lib, withhold, wait_ms):
    assert lib.selscan_test_fault_injection(withhold, wait_ms) == ss.ERR_INVALID_ARG


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


# ---- the extended, gated, conv1d and host-buffer entry points ---------------

def fwd_ex(lib, flags=1, Dskip=None, z=None, **kw):
    a = dict(x=0x10000, delta=0x20000, A=0x30000, B=0x40000, C=0x50000, y=0x60000,
             Bsz=1, L=8, D=4, N=4, dtype=F32, h0=None, hT=None)
    a.update(kw)
    return lib.selscan_fwd_ex(a["x"], a["delta"], a["A"], a["B"], a["C"], Dskip, z, a["y"], a["Bsz"], a["L"],
                              a["D"], a["N"], a["dtype"], flags, a["h0"], a["hT"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(flags=4), ss.ERR_INVALID_ARG),                       # unknown flag bit
    (dict(z=0x60000 + 4), ss.ERR_INVALID_ARG),                 # z overlaps y partially
    (dict(z=0x70000, hT=0x70000 + 8), ss.ERR_INVALID_ARG),     # hT overlaps z
    (dict(Dskip=0x60000), ss.ERR_INVALID_ARG),                 # y overlaps Dskip
    (dict(Dskip=0x70002), ss.ERR_INVALID_ARG),                 # misaligned Dskip
    (dict(z=0x70002), ss.ERR_INVALID_ARG),                     # misaligned z
    (dict(N=65), ss.ERR_UNSUPPORTED),
])
def test_fwd_ex_argument_errors(lib, kw, code):
    assert fwd_ex(lib, **kw) == code
    assert ss.last_error() != ""


def test_fwd_ex_empty_problem_is_ok_without_cuda(lib):
    assert fwd_ex(lib, flags=ss.FLAG_SOFTPLUS | ss.FLAG_ZOH, Bsz=0) == ss.OK


def test_gated_forward_shares_the_checks(lib):
    rc = lib.selscan_fwd_gated(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, None, 0x60000 + 4, 0x60000,
                               1, 8, 4, 4, F32, 1, None, None, None)
    assert rc == ss.ERR_INVALID_ARG


def test_step_ex_takes_zoh_only(lib):
    rc = lib.selscan_step_ex(0x10000, 0x20000, 0x28000, 0x30000, 0x40000, 0x50000, None, None, 0x60000,
                             2, 4, 16, ss.FLAG_SOFTPLUS, None)
    assert rc == ss.ERR_INVALID_ARG and "ZOH" in ss.last_error()
    rc = lib.selscan_step_ex(0x10000, 0x20000, 0x28000, 0x30000, 0x40000, 0x50000, None, 0x60000, 0x60000,
                             2, 4, 16, ss.FLAG_ZOH, None)
    assert rc == ss.ERR_INVALID_ARG                            # y overlaps z


def conv(lib, **kw):
    a = dict(x=0x10000, w=0x20000, bias=None, out=0x30000, Bsz=1, L=8, D=4, K=4, dtype=F32, silu=1,
             state_in=None, state_out=None)
    a.update(kw)
    return lib.selscan_conv1d(a["x"], a["w"], a["bias"], a["out"], a["Bsz"], a["L"], a["D"], a["K"],
                              a["dtype"], a["silu"], a["state_in"], a["state_out"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(K=0), ss.ERR_INVALID_ARG),
    (dict(K=9), ss.ERR_UNSUPPORTED),
    (dict(dtype=3), ss.ERR_INVALID_ARG),
    (dict(L=-1), ss.ERR_INVALID_ARG),
    (dict(w=None), ss.ERR_INVALID_ARG),
    (dict(out=0x10000 + 8), ss.ERR_INVALID_ARG),               # out overlaps x (no in-place)
    (dict(state_in=0x40000, state_out=0x40000), ss.ERR_INVALID_ARG),  # state_out is state_in
    (dict(state_out=0x20000), ss.ERR_INVALID_ARG),             # state_out overlaps w
    (dict(x=0x10002), ss.ERR_INVALID_ARG),                     # misaligned
    (dict(Bsz=70000), ss.ERR_UNSUPPORTED),                     # grid limit
])
def test_conv1d_argument_errors(lib, kw, code):
    assert conv(lib, **kw) == code
    assert ss.last_error() != ""


def test_conv1d_empty_problem_is_ok_without_cuda(lib):
    assert conv(lib, Bsz=0) == ss.OK
    assert conv(lib, D=0) == ss.OK


@pytest.mark.parametrize("kw,code", [
    (dict(K=0), ss.ERR_INVALID_ARG),
    (dict(K=9), ss.ERR_UNSUPPORTED),
    (dict(state=None), ss.ERR_INVALID_ARG),                    # K > 1 needs the state
    (dict(out=0x10000), ss.ERR_INVALID_ARG),                   # out overlaps the state
    (dict(x=0x20001), ss.ERR_INVALID_ARG),
])
def test_conv1d_step_argument_errors(lib, kw, code):
    a = dict(state=0x10000, x=0x20000, w=0x30000, bias=None, out=0x40000, Bsz=2, D=4, K=4, silu=1)
    a.update(kw)
    rc = lib.selscan_conv1d_step(a["state"], a["x"], a["w"], a["bias"], a["out"], a["Bsz"], a["D"], a["K"],
                                 a["silu"], None)
    assert rc == code


@pytest.mark.parametrize("entry", ["selscan_fwd_host", "selscan_fwd_noalloc"])
def test_host_and_noalloc_forward_share_the_checks(lib, entry):
    f = getattr(lib, entry)
    assert f(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 1, 8, 4, 4, 9, 1, None, None, None) \
        == ss.ERR_INVALID_ARG                                  # bad dtype
    assert f(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x10000 + 4, 1, 8, 4, 4, F32, 1, None, None, None) \
        == ss.ERR_INVALID_ARG                                  # y overlaps x partially
    assert f(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 0, 8, 4, 4, F32, 1, None, None, None) == ss.OK


def bwd(lib, **kw):
    a = dict(x=0x10000, delta=0x20000, A=0x30000, B=0x40000, C=0x50000, h0=None, dy=0x60000, dhT=None,
             dx=0x70000, ddelta=0x80000, dA=0x90000, dB=0xA0000, dC=0xB0000, dh0=None,
             Bsz=1, L=8, D=4, N=16, sp=1)
    a.update(kw)
    return lib.selscan_bwd(a["x"], a["delta"], a["A"], a["B"], a["C"], a["h0"], a["dy"], a["dhT"], a["dx"],
                           a["ddelta"], a["dA"], a["dB"], a["dC"], a["dh0"], a["Bsz"], a["L"], a["D"], a["N"],
                           a["sp"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(N=0), ss.ERR_INVALID_ARG),
    (dict(N=33), ss.ERR_UNSUPPORTED),                          # lane groups end at one warp
    (dict(Bsz=70000), ss.ERR_UNSUPPORTED),                     # grid limit
    (dict(L=-1), ss.ERR_INVALID_ARG),
    (dict(dA=None), ss.ERR_INVALID_ARG),
    (dict(dy=None), ss.ERR_INVALID_ARG),
    (dict(x=0x10002), ss.ERR_INVALID_ARG),                     # misaligned
    (dict(dx=0x10000 + 4), ss.ERR_INVALID_ARG),                # dx overlaps x
    (dict(dB=0x70000 + 8), ss.ERR_INVALID_ARG),                # dB overlaps dx
    (dict(dh0=0xC0000, h0=0xC0000), ss.ERR_INVALID_ARG),       # dh0 overlaps h0
    (dict(dA=0x60000), ss.ERR_INVALID_ARG),                    # dA overlaps dy
    (dict(L=1 << 40, D=1 << 30), ss.ERR_INVALID_ARG),          # size overflow
])
def test_bwd_argument_errors(lib, kw, code):
    assert bwd(lib, **kw) == code
    assert ss.last_error() != ""


def test_bwd_empty_channel_count_is_ok_without_cuda(lib):
    assert bwd(lib, D=0, A=None, dA=None) == ss.OK


def bwd_gated(lib, **kw):
    a = dict(x=0x10000, delta=0x20000, A=0x30000, B=0x40000, C=0x50000, Dskip=0xD0000, z=0xE0000, h0=None,
             dy=0x60000, dhT=None, dx=0x70000, ddelta=0x80000, dA=0x90000, dB=0xA0000, dC=0xB0000,
             dDskip=0xF0000, dz=0x100000, dh0=None, Bsz=1, L=8, D=4, N=16, sp=1)
    a.update(kw)
    return lib.selscan_bwd_gated(*(a[k] for k in ("x", "delta", "A", "B", "C", "Dskip", "z", "h0", "dy", "dhT",
                                                   "dx", "ddelta", "dA", "dB", "dC", "dDskip", "dz", "dh0",
                                                   "Bsz", "L", "D", "N", "sp")), None)


@pytest.mark.parametrize("kw,code", [
    (dict(dDskip=None), ss.ERR_INVALID_ARG),                  # Dskip without its gradient
    (dict(Dskip=None), ss.ERR_INVALID_ARG),                   # dDskip without Dskip
    (dict(dz=None), ss.ERR_INVALID_ARG),                      # z without its gradient
    (dict(z=None), ss.ERR_INVALID_ARG),                       # dz without z
    (dict(z=0xE0002), ss.ERR_INVALID_ARG),                    # misaligned
    (dict(dz=0x70000 + 4), ss.ERR_INVALID_ARG),               # dz overlaps dx
    (dict(dDskip=0xD0000), ss.ERR_INVALID_ARG),               # dDskip overlaps Dskip
    (dict(dz=0xE0000 + 16), ss.ERR_INVALID_ARG),              # dz overlaps z
])
def test_bwd_gated_argument_errors(lib, kw, code):
    assert bwd_gated(lib, **kw) == code
    assert ss.last_error() != ""


def test_bwd_gated_empty_channel_count_is_ok_without_cuda(lib):
    assert bwd_gated(lib, D=0, A=None, dA=None) == ss.OK


def test_host_alloc_checks_its_arguments(lib):
    """The host allocator refuses an empty request and frees only its own
    blocks (no CUDA call is reached on these paths)."""
    assert lib.selscan_host_alloc(0) is None
    assert ss.last_error() != ""
    assert lib.selscan_host_free(ctypes.c_void_p(0x123000)) == ss.ERR_INVALID_ARG
    assert lib.selscan_host_free(None) == ss.OK


def ssd(lib, **kw):
    a = dict(x=16, dt=8, A=8, B=16, C=16, y=16, h0=None, hT=None, Bsz=1, L=4, H=2, P=64, N=128, dtype=0,
             softplus=1)
    a.update(kw)
    return lib.selscan_ssd_fwd(a["x"], a["dt"], a["A"], a["B"], a["C"], a["y"], a["h0"], a["hT"], a["Bsz"],
                               a["L"], a["H"], a["P"], a["N"], a["dtype"], a["softplus"], None)


@pytest.mark.parametrize("kw, code", [
    (dict(dtype=7), ss.ERR_INVALID_ARG), (dict(L=-1), ss.ERR_INVALID_ARG), (dict(P=0), ss.ERR_INVALID_ARG),
    (dict(N=32), ss.ERR_UNSUPPORTED), (dict(P=48), ss.ERR_UNSUPPORTED), (dict(x=None), ss.ERR_INVALID_ARG),
    (dict(A=None), ss.ERR_INVALID_ARG), (dict(y=12), ss.ERR_INVALID_ARG), (dict(x=24), ss.ERR_INVALID_ARG), (dict(Bsz=70000), ss.ERR_UNSUPPORTED),
])
def test_ssd_argument_errors(lib, kw, code):
    """Argument checks of selscan_ssd_fwd run before any CUDA call."""
    assert ssd(lib, **kw) == code


def test_ssd_empty_problem_is_ok_without_cuda(lib):
    assert ssd(lib, Bsz=0) == ss.OK and ssd(lib, H=0) == ss.OK
