"""The method's limiting cases on the GPU, against the fp64 oracle.

The limits are those of "3.1 LTI systems and input-dependent parameters"
(booiljung.github.io), section 0.4.2: a step size going to 0 keeps the state
(exp(0 * A) = 1 and the input term vanishes), and a step size going to
infinity with A < 0 resets it to the current input term. A = 0 turns the
state into a running sum. Softplus pre-activations far in either tail give
steps of e^-80 and 80. These are exactly the inputs where fp32 on the device
(ex2.approx with flush-to-zero, the packed softplus) departs furthest from
fp64.

Every case runs the forward scan on the TMA path and the plain-load path,
in one pass and chunked, for fp32 and bf16 I/O, and the decode step; every
output is compared element by element with the oracle. With delta = 0
exactly the final state must equal h0 bit for bit.

The bound. Steps of 1e4 make every state a sum of terms around 1e4 that
cancel to a much smaller result (and A = 0 turns a state into a running sum
of such terms), so no fp32 evaluation can hold |got - ref| / (1 + |ref|):
its rounding error scales with the terms, not with their sum. The error is
therefore measured against the magnitude of what was summed,
|got - ref| / (1 + M), with M the same scan run by the oracle on |x|, |B|,
|C| and |h0| (every decay is positive, so that scan adds the magnitudes of
the signed scan's terms) -- the forward-error bound of a floating-point sum.
The tolerances are the usual ones (1e-4 fp32, 2e-2 bf16). Where nothing
cancels (delta = 0, A = 0 with ordinary steps, softplus tails) the plain
metric must hold as well.
"""
import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import TOL, fwd_dev, oracle_fwd, scaled_err, to_dev, to_np

pytestmark = pytest.mark.gpu

PATHS = {
    "tma-onepass": {"SELSCAN_CHUNK": "0"},
    "tma-chunked": {"SELSCAN_CHUNK": "64"},
    "plain-onepass": {"SELSCAN_CHUNK": "0", "SELSCAN_NO_TMA": "1"},
    "plain-chunked": {"SELSCAN_CHUNK": "64", "SELSCAN_NO_TMA": "1"},
}
SOFTPLUS_TAILS = np.array([-80.0, -20.0, -5.0, 0.0, 5.0, 20.0, 80.0], np.float32)


def _set_delta(inp, delta_f32, softplus):
    """Replaces the step (or its pre-activation) of the inputs."""
    inp.delta_softplus = softplus
    inp.delta = W.to_bf16_bits(delta_f32) if inp.dtype == W.BF16 else delta_f32.astype(np.float32)
    return inp


def _case(name, dtype, seed=7):
    Bsz, L, D, N = 2, 300, 136, 16
    inp = W.fwd_inputs(Bsz, L, D, N, seed=seed, dtype=dtype, with_h0=True)
    g = np.random.default_rng(seed)
    if name == "delta_zero":
        _set_delta(inp, np.zeros((Bsz, L, D), np.float32), softplus=False)
    elif name == "delta_1e4":
        _set_delta(inp, np.full((Bsz, L, D), 1e4, np.float32), softplus=False)
    elif name == "A_zero":
        A = inp.A.copy()
        A[::3, :] = 0.0                     # whole channels with A = 0
        A[1::3, ::4] = 0.0                  # single states with A = 0
        inp.A = A
    elif name == "softplus_tails":
        _set_delta(inp, g.choice(SOFTPLUS_TAILS, size=(Bsz, L, D)).astype(np.float32), softplus=True)
    elif name == "mixed":
        steps = np.array([0.0, 1e-12, 1e-3, 0.05, 1.0, 1e4], np.float32)
        _set_delta(inp, g.choice(steps, size=(Bsz, L, D)).astype(np.float32), softplus=False)
        A = inp.A.copy()
        A[::5, :] = 0.0
        inp.A = A
    else:
        raise ValueError(name)
    return inp


CASES = ["delta_zero", "delta_1e4", "A_zero", "softplus_tails", "mixed"]
CANCELLING = {"delta_1e4", "mixed"}


def bounded_err(got, ref, mag) -> float:
    """max |got - ref| / (1 + M): the error against the magnitude of the terms."""
    got, ref, mag = (np.asarray(a, np.float64) for a in (got, ref, mag))
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(mag))))


def magnitudes(orc, inp):
    """The oracle's scan on |x|, |B|, |C|, |h0| (same steps and A): the sums
    of the magnitudes of the terms the signed scan adds, for y and hT."""
    h0 = None if inp.h0 is None else np.abs(inp.h0).astype(np.float64)
    return orc.selscan_fwd(np.abs(inp.f32("x")), inp.f32("delta"), inp.A, np.abs(inp.f32("B")),
                           np.abs(inp.f32("C")), inp.delta_softplus, h0)


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("case", CASES)
def test_forward_limits(orc, monkeypatch, case, dtype, path):
    for k, v in PATHS[path].items():
        monkeypatch.setenv(k, v)
    inp = _case(case, dtype)
    x, dl, A, B, C, h0 = fwd_dev(inp)
    y, hT = ss.selscan_fwd(x, dl, A, B, C, inp.delta_softplus, h0, return_final_state=True)
    torch.cuda.synchronize()
    ss.check_device_error()
    yr, hr = oracle_fwd(orc, inp)
    assert torch.isfinite(y.float()).all() and torch.isfinite(hT).all()
    ym, hm = magnitudes(orc, inp)
    ey, eh = bounded_err(to_np(y), yr, ym), bounded_err(to_np(hT), hr, hm)
    assert ey <= TOL[dtype], f"y error {ey:.3e} against the terms' magnitude"
    assert eh <= TOL[W.F32], f"hT error {eh:.3e} against the terms' magnitude"
    if case not in CANCELLING:
        ey, eh = scaled_err(to_np(y), yr), scaled_err(to_np(hT), hr)
        assert ey <= TOL[dtype], f"y error {ey:.3e}"
        assert eh <= TOL[W.F32], f"hT error {eh:.3e}"
    if case == "delta_zero":
        assert torch.equal(hT, h0), "delta = 0 must leave the state exactly as it was"


def test_forward_limits_take_the_paths_they_name(monkeypatch):
    """The chunked cases really are chunked, and the TMA cases run one fused
    launch (after the kernel that clears a chunked plan's control words)."""
    for path, env in PATHS.items():
        for k in ("SELSCAN_CHUNK", "SELSCAN_NO_TMA"):
            monkeypatch.delenv(k, raising=False)
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        p = ss.fwd_plan(2, 300, 136, 16)
        assert (p["chunks"] > 1) == path.endswith("chunked"), path
        if path.startswith("tma"):
            assert p["launches"] == (2 if path.endswith("chunked") else 1), path


def _step_case(name, seed=3):
    Bsz, D, N = 4, 200, 16
    g = np.random.default_rng(seed)
    f = lambda *s: g.standard_normal(s).astype(np.float32)
    state, x, B, C = f(Bsz, D, N), f(Bsz, D), f(Bsz, N), f(Bsz, N)
    A = np.broadcast_to(-np.arange(1, N + 1, dtype=np.float32), (D, N)).copy()
    delta = np.abs(f(Bsz, D)) * np.float32(0.05)
    if name == "delta_zero":
        delta[:] = 0.0
    elif name == "delta_1e4":
        delta[:] = 1e4
    elif name == "A_zero":
        A[::3, :] = 0.0
        A[1::3, ::4] = 0.0
    elif name == "mixed":
        delta = g.choice(np.array([0.0, 1e-12, 1e-3, 0.05, 1.0, 1e4], np.float32), size=(Bsz, D))
        A[::5, :] = 0.0
    return state, x, delta.astype(np.float32), A, B, C


@pytest.mark.parametrize("case", ["delta_zero", "delta_1e4", "A_zero", "mixed"])
def test_decode_step_limits(orc, case):
    state, x, delta, A, B, C = _step_case(case)
    sd = to_dev(state)
    y = ss.selscan_step(sd, to_dev(x), to_dev(delta), to_dev(A), to_dev(B), to_dev(C))
    torch.cuda.synchronize()
    st_ref = np.ascontiguousarray(state, dtype=np.float64)
    y_ref = orc.selscan_step(st_ref, x, delta, A, B, C)
    st_mag = np.abs(state).astype(np.float64)
    y_mag = orc.selscan_step(st_mag, np.abs(x), delta, A, np.abs(B), np.abs(C))
    assert bounded_err(to_np(y), y_ref, y_mag) <= TOL[W.F32]
    assert bounded_err(to_np(sd), st_ref, st_mag) <= TOL[W.F32]
    if case not in CANCELLING:
        assert scaled_err(to_np(y), y_ref) <= TOL[W.F32]
        assert scaled_err(to_np(sd), st_ref) <= TOL[W.F32]
    if case == "delta_zero":
        assert torch.equal(sd, to_dev(state)), "delta = 0 must leave the state exactly as it was"


# ---------------------------------------------------------------- in place on the fused path

def _fused_chunked_inputs(dtype, seed):
    # D a multiple of 8: rows meet TMA's 16-byte rule for both dtypes.
    return W.fwd_inputs(2, 1000, 96, 16, seed=seed, dtype=dtype, with_h0=True)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("over", ["x", "delta"])
def test_in_place_output_on_the_fused_chunked_path(orc, monkeypatch, dtype, over):
    """y written over x or delta while later chunks' reductions read them."""
    monkeypatch.setenv("SELSCAN_CHUNK", "64")
    inp = _fused_chunked_inputs(dtype, seed=31 + (over == "delta"))
    p = ss.fwd_plan(2, 1000, 96, 16, bf16=dtype == W.BF16)
    assert p["chunks"] == 16 and p["launches"] == 2
    x, dl, A, B, C, h0 = fwd_dev(inp)
    target = x if over == "x" else dl
    ss.selscan_fwd(x, dl, A, B, C, True, h0, y=target)
    torch.cuda.synchronize()
    ss.check_device_error()
    yr, _ = oracle_fwd(orc, inp)
    assert scaled_err(to_np(target), yr) <= TOL[dtype]


def test_in_place_gated_output_over_z(orc, monkeypatch):
    monkeypatch.setenv("SELSCAN_CHUNK", "64")
    inp = _fused_chunked_inputs(W.F32, seed=35)
    Dskip, z = W.gate_inputs(2, 1000, 96, seed=35)
    x, dl, A, B, C, h0 = fwd_dev(inp)
    zd, Dd = to_dev(z), to_dev(Dskip)
    ss.selscan_fwd(x, dl, A, B, C, True, h0, y=zd, D_skip=Dd, z=zd)
    torch.cuda.synchronize()
    ss.check_device_error()
    yr, _ = orc.selscan_fwd(inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C"), True,
                            inp.h0.astype(np.float64), Dskip=Dskip, z=z)
    assert scaled_err(to_np(zd), yr) <= TOL[W.F32]


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("path", ["tma-chunked", "plain-chunked"])
def test_resume_in_place_on_chunked_paths(orc, monkeypatch, dtype, path):
    """hT written over h0 while every chunk's first pass may still read h0."""
    for k, v in PATHS[path].items():
        monkeypatch.setenv(k, v)
    inp = _fused_chunked_inputs(dtype, seed=41)
    x, dl, A, B, C, h0 = fwd_dev(inp)
    y, _ = ss.selscan_fwd(x, dl, A, B, C, True, h0, hT=h0)
    torch.cuda.synchronize()
    ss.check_device_error()
    yr, hr = oracle_fwd(orc, inp)
    assert scaled_err(to_np(y), yr) <= TOL[dtype]
    assert scaled_err(to_np(h0), hr) <= TOL[W.F32]
