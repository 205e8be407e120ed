"""ctypes wrapper around the fp64 CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it to check and time the CUDA path.
The library package never imports it, and it shares no code with it.

The oracle follows the simplified ``selective_scan`` loop of "Mamba:
Selective State Space Models" (youngju.dev, section 3.3) in double
precision; see the header of oracle.c for the exact statement.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-std=c99", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
           "-pthread", "-D_POSIX_C_SOURCE=200809L"]


def _compile(src: str, out: str) -> None:
    subprocess.run(["gcc", *_CFLAGS, "-o", out + ".tmp", src, "-lm"], check=True)
    os.replace(out + ".tmp", out)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (plain gcc, no fast-math,
    no FMA contraction, so every operation rounds as written)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SRC):
        _compile(SRC, _LIB)
    return _LIB


def _f32(a, shape, name):
    a = np.ascontiguousarray(a, dtype=np.float32)
    if tuple(a.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {a.shape}")
    return a


def _f64(a, shape, name):
    a = np.ascontiguousarray(a, dtype=np.float64)
    if tuple(a.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {a.shape}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data


class Oracle:
    """One loaded copy of the oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        INT = ctypes.c_int
        lib.oracle_softplus.restype = ctypes.c_double
        lib.oracle_softplus.argtypes = [ctypes.c_double]
        lib.oracle_selscan_fwd.restype = INT
        lib.oracle_selscan_fwd.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, I64, INT, INT]
        lib.oracle_selscan_fwd_chains.restype = INT
        lib.oracle_selscan_fwd_chains.argtypes = [P, P, P, P, P, P, P, I64, P, P,
                                                  I64, I64, I64, I64, INT, INT]
        lib.oracle_selscan_step.restype = INT
        lib.oracle_selscan_step.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, I64]
        lib.oracle_selscan_fwd_gated.restype = INT
        lib.oracle_selscan_fwd_gated.argtypes = [P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, INT, INT, INT]
        lib.oracle_selscan_fwd_chains_gated.restype = INT
        lib.oracle_selscan_fwd_chains_gated.argtypes = [P, P, P, P, P, P, P, P, P, I64, P, P,
                                                        I64, I64, I64, I64, INT, INT, INT]
        lib.oracle_selscan_step_gated.restype = INT
        lib.oracle_selscan_step_gated.argtypes = [P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, INT]
        lib.oracle_conv1d.restype = INT
        lib.oracle_conv1d.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, INT]
        lib.oracle_ssd_fwd.restype = INT
        lib.oracle_ssd_fwd.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, I64, I64, INT]
        lib.oracle_selscan_bwd_gated.restype = INT
        lib.oracle_selscan_bwd_gated.argtypes = [P] * 18 + [I64, I64, I64, I64, INT]
        lib.oracle_selscan_bwd.restype = INT
        lib.oracle_selscan_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, INT]
        self._lib = lib
        self.path = path

    def softplus(self, u: float) -> float:
        """log(1 + e^u) in double."""
        return self._lib.oracle_softplus(float(u))

    def selscan_fwd(self, x, delta, A, B, C, delta_softplus=False, h0=None, nthreads=0,
                    Dskip=None, z=None, zoh=False):
        """Sequential selective scan in fp64.

        x, delta: (Bsz, L, D); A: (D, N); B, C: (Bsz, L, N); h0: (Bsz, D, N)
        or None. Inputs are taken as float32 (the exact values the GPU reads);
        h0 as float64 (fp32 states widen exactly). Dskip (D,) and z
        (Bsz, L, D) add the block's skip and gate: y = (y + Dskip x) silu(z).
        zoh: the zero-order-hold Bbar of section 2.2 instead of dl * B.
        Returns (y (Bsz, L, D) float64, hT (Bsz, D, N) float64).
        """
        x = np.asarray(x)
        Bsz, L, D = x.shape
        N = np.asarray(A).shape[1]
        x = _f32(x, (Bsz, L, D), "x")
        delta = _f32(delta, (Bsz, L, D), "delta")
        A = _f32(A, (D, N), "A")
        B = _f32(B, (Bsz, L, N), "B")
        C = _f32(C, (Bsz, L, N), "C")
        h0 = None if h0 is None else _f64(h0, (Bsz, D, N), "h0")
        Dskip = None if Dskip is None else _f32(Dskip, (D,), "Dskip")
        z = None if z is None else _f32(z, (Bsz, L, D), "z")
        y = np.zeros((Bsz, L, D), np.float64)
        hT = np.zeros((Bsz, D, N), np.float64)
        rc = self._lib.oracle_selscan_fwd_gated(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                                _ptr(Dskip), _ptr(z), _ptr(h0),
                                                _ptr(y), _ptr(hT), Bsz, L, D, N,
                                                int(bool(delta_softplus)), int(bool(zoh)), int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle_selscan_fwd failed")
        return y, hT

    def selscan_fwd_chains(self, x, delta, A, B, C, chains, delta_softplus=False, h0=None,
                           nthreads=0, Dskip=None, z=None, zoh=False):
        """The same scan for selected chains c = b * D + d only.
        Returns (y (nchains, L), hT (nchains, N)) in float64."""
        x = np.asarray(x)
        Bsz, L, D = x.shape
        N = np.asarray(A).shape[1]
        x = _f32(x, (Bsz, L, D), "x")
        delta = _f32(delta, (Bsz, L, D), "delta")
        A = _f32(A, (D, N), "A")
        B = _f32(B, (Bsz, L, N), "B")
        C = _f32(C, (Bsz, L, N), "C")
        h0 = None if h0 is None else _f64(h0, (Bsz, D, N), "h0")
        chains = np.ascontiguousarray(chains, dtype=np.int64)
        nc = chains.shape[0]
        y = np.zeros((nc, L), np.float64)
        hT = np.zeros((nc, N), np.float64)
        Dskip = None if Dskip is None else _f32(Dskip, (D,), "Dskip")
        z = None if z is None else _f32(z, (Bsz, L, D), "z")
        rc = self._lib.oracle_selscan_fwd_chains_gated(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                                       _ptr(Dskip), _ptr(z), _ptr(h0), _ptr(chains), nc,
                                                       _ptr(y), _ptr(hT), Bsz, L, D, N,
                                                       int(bool(delta_softplus)), int(bool(zoh)),
                                                       int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle_selscan_fwd_chains failed")
        return y, hT

    def selscan_step(self, state, x, delta, A, B, C, chains=None, Dskip=None, z=None, zoh=False):
        """One decode step in place on a float64 state.

        state: (Bsz, D, N) float64, or (nchains, N) when ``chains`` is given;
        x, delta: (Bsz, D); A: (D, N); B, C: (Bsz, N). delta is used as given.
        Dskip (D,) and z (Bsz, D) add the block's skip and gate.
        Returns y: (Bsz, D) float64, or (nchains,) when ``chains`` is given.
        """
        if not (isinstance(state, np.ndarray) and state.dtype == np.float64
                and state.flags.c_contiguous):
            raise ValueError("state must be a C-contiguous float64 array (updated in place)")
        x = np.asarray(x)
        Bsz, D = x.shape
        N = np.asarray(A).shape[1]
        x = _f32(x, (Bsz, D), "x")
        delta = _f32(delta, (Bsz, D), "delta")
        A = _f32(A, (D, N), "A")
        B = _f32(B, (Bsz, N), "B")
        C = _f32(C, (Bsz, N), "C")
        if chains is None:
            if state.shape != (Bsz, D, N):
                raise ValueError("state shape")
            y = np.zeros((Bsz, D), np.float64)
            ch, nc = None, 0
        else:
            ch = np.ascontiguousarray(chains, dtype=np.int64)
            nc = ch.shape[0]
            if state.shape != (nc, N):
                raise ValueError("state shape")
            y = np.zeros((nc,), np.float64)
        Dskip = None if Dskip is None else _f32(Dskip, (D,), "Dskip")
        z = None if z is None else _f32(z, (Bsz, D), "z")
        rc = self._lib.oracle_selscan_step_gated(_ptr(state), _ptr(x), _ptr(delta), _ptr(A), _ptr(B),
                                                 _ptr(C), _ptr(Dskip), _ptr(z), _ptr(y), _ptr(ch), nc,
                                                 Bsz, D, N, int(bool(zoh)))
        if rc != 0:
            raise RuntimeError("oracle_selscan_step failed")
        return y


    def conv1d(self, x, w, bias=None, state_in=None, silu=True):
        """Causal depthwise convolution over L with K taps per channel, then
        SiLU (the MambaBlock's conv1d): x (Bsz, L, D), w (D, K), bias (D,) or
        None, state_in (Bsz, D, K-1) or None (zeros). Returns (out (Bsz, L, D)
        float64, state_out (Bsz, D, K-1) float32: the last K-1 inputs)."""
        x = np.asarray(x)
        Bsz, L, D = x.shape
        K = np.asarray(w).shape[1]
        x = _f32(x, (Bsz, L, D), "x")
        w = _f32(w, (D, K), "w")
        bias = None if bias is None else _f32(bias, (D,), "bias")
        state_in = None if state_in is None else _f32(state_in, (Bsz, D, K - 1), "state_in")
        out = np.zeros((Bsz, L, D), np.float64)
        st = np.zeros((Bsz, D, K - 1), np.float32)
        rc = self._lib.oracle_conv1d(_ptr(x), _ptr(w), _ptr(bias), _ptr(state_in), _ptr(out), _ptr(st),
                                     Bsz, L, D, K, int(bool(silu)))
        if rc != 0:
            raise RuntimeError("oracle_conv1d failed")
        return out, st


    def selscan_bwd(self, x, delta, A, B, C, gy, delta_softplus=False, h0=None, ghT=None, Dskip=None, z=None):
        """Gradients of a loss through the scan (dl * B form), by the plain
        reverse sweep over each chain's stored states.

        Shapes as selscan_fwd; gy (Bsz, L, D) = dLoss/dy, ghT (Bsz, D, N) =
        dLoss/dhT or None. Returns a dict of float64 arrays dx, ddelta
        (Bsz, L, D), dA (D, N), dB, dC (Bsz, L, N) and dh0 (Bsz, D, N).
        With Dskip (D,) and/or z (Bsz, L, D), y is the block's output
        (y + Dskip x) silu(z), gy its gradient, and the dict adds dDskip (D,)
        and/or dz (Bsz, L, D).
        """
        if Dskip is not None or z is not None:
            return self._selscan_bwd_gated(x, delta, A, B, C, gy, delta_softplus, h0, ghT, Dskip, z)
        x = np.asarray(x)
        Bsz, L, D = x.shape
        N = np.asarray(A).shape[1]
        x = _f32(x, (Bsz, L, D), "x")
        delta = _f32(delta, (Bsz, L, D), "delta")
        A = _f32(A, (D, N), "A")
        B = _f32(B, (Bsz, L, N), "B")
        C = _f32(C, (Bsz, L, N), "C")
        h0 = None if h0 is None else _f64(h0, (Bsz, D, N), "h0")
        gy = _f64(gy, (Bsz, L, D), "gy")
        ghT = None if ghT is None else _f64(ghT, (Bsz, D, N), "ghT")
        g = dict(dx=np.zeros((Bsz, L, D)), ddelta=np.zeros((Bsz, L, D)), dA=np.zeros((D, N)),
                 dB=np.zeros((Bsz, L, N)), dC=np.zeros((Bsz, L, N)), dh0=np.zeros((Bsz, D, N)))
        rc = self._lib.oracle_selscan_bwd(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(h0),
                                          _ptr(gy), _ptr(ghT), _ptr(g["dx"]), _ptr(g["ddelta"]),
                                          _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dh0"]),
                                          Bsz, L, D, N, int(bool(delta_softplus)))
        if rc != 0:
            raise RuntimeError("oracle_selscan_bwd failed")
        return g


    def _selscan_bwd_gated(self, x, delta, A, B, C, gy, delta_softplus, h0, ghT, Dskip, z):
        x = np.asarray(x)
        Bsz, L, D = x.shape
        N = np.asarray(A).shape[1]
        x = _f32(x, (Bsz, L, D), "x")
        delta = _f32(delta, (Bsz, L, D), "delta")
        A = _f32(A, (D, N), "A")
        B = _f32(B, (Bsz, L, N), "B")
        C = _f32(C, (Bsz, L, N), "C")
        h0 = None if h0 is None else _f64(h0, (Bsz, D, N), "h0")
        gy = _f64(gy, (Bsz, L, D), "gy")
        ghT = None if ghT is None else _f64(ghT, (Bsz, D, N), "ghT")
        Dskip = None if Dskip is None else _f32(Dskip, (D,), "Dskip")
        z = None if z is None else _f32(z, (Bsz, L, D), "z")
        g = dict(dx=np.zeros((Bsz, L, D)), ddelta=np.zeros((Bsz, L, D)), dA=np.zeros((D, N)),
                 dB=np.zeros((Bsz, L, N)), dC=np.zeros((Bsz, L, N)), dh0=np.zeros((Bsz, D, N)))
        if Dskip is not None:
            g["dDskip"] = np.zeros((D,))
        if z is not None:
            g["dz"] = np.zeros((Bsz, L, D))
        rc = self._lib.oracle_selscan_bwd_gated(
            _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(Dskip), _ptr(z), _ptr(h0), _ptr(gy), _ptr(ghT),
            _ptr(g["dx"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dh0"]),
            _ptr(g.get("dDskip")), _ptr(g.get("dz")), Bsz, L, D, N, int(bool(delta_softplus)))
        if rc != 0:
            raise RuntimeError("oracle_selscan_bwd_gated failed")
        return g

    def ssd_fwd(self, x, dt, A, B, C, dt_softplus=False, h0=None):
        """Mamba-2 SSD forward in fp64 (see oracle.c): x (Bsz, L, H, P),
        dt (Bsz, L, H), A (H,), B, C (Bsz, L, N), h0 (Bsz, H, N, P) or None.
        Returns (y (Bsz, L, H, P), hT (Bsz, H, N, P)) in float64."""
        x = np.asarray(x)
        Bsz, L, H, P = x.shape
        N = np.asarray(B).shape[2]
        x = _f32(x, (Bsz, L, H, P), "x")
        dt = _f32(dt, (Bsz, L, H), "dt")
        A = _f32(A, (H,), "A")
        B = _f32(B, (Bsz, L, N), "B")
        C = _f32(C, (Bsz, L, N), "C")
        h0 = None if h0 is None else _f64(h0, (Bsz, H, N, P), "h0")
        y = np.zeros((Bsz, L, H, P))
        hT = np.zeros((Bsz, H, N, P))
        rc = self._lib.oracle_ssd_fwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(h0), _ptr(y), _ptr(hT),
                                      Bsz, L, H, P, N, int(bool(dt_softplus)))
        if rc != 0:
            raise RuntimeError("oracle_ssd_fwd failed")
        return y, hT


def compile_variant(src: str, out: str) -> Oracle:
    """Build and load a copy of the oracle from another C source file
    (the mutation tests plant mistakes this way, on the CPU)."""
    _compile(src, out)
    return Oracle(out)


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def softplus(u):
    return default().softplus(u)


def selscan_fwd(*args, **kwargs):
    return default().selscan_fwd(*args, **kwargs)


def selscan_fwd_chains(*args, **kwargs):
    return default().selscan_fwd_chains(*args, **kwargs)


def selscan_step(*args, **kwargs):
    return default().selscan_step(*args, **kwargs)


def conv1d(*args, **kwargs):
    return default().conv1d(*args, **kwargs)


def selscan_bwd(*args, **kwargs):
    return default().selscan_bwd(*args, **kwargs)


def ssd_fwd(*args, **kwargs):
    return default().ssd_fwd(*args, **kwargs)
