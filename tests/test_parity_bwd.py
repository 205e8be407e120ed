"""selscan_bwd: the backward pass of the scan against the fp64 oracle's
reverse sweep, on the same fp32 inputs and upstream gradients. Covers one
and many 16-step chunks with ragged tails, one segment and many (the
sequence is cut into segments whose carries are composed in both
directions), channel counts that leave the last block partly empty, every
width of a chain (1, 2, 4 and 8 threads of four states: N = 1 to 4, 5 to 8,
9 to 16, 17 to 32), with and without softplus, h0 and dhT, the empty
sequence, the 130M-like layer at full size, and autograd through the
differentiable wrapper; and the block's skip and gate (selscan_bwd_gated,
against the oracle's gated reverse sweep: dD_skip and dz as well)."""
import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import TOL, scaled_err, to_dev, to_np

pytestmark = pytest.mark.gpu

NAMES = ("dx", "ddelta", "dA", "dB", "dC", "dh0")


def run(orc, Bsz, L, D, N, seed, softplus=True, with_h0=True, with_dhT=True, a_init="loguniform"):
    inp = W.fwd_inputs(Bsz, L, D, N, seed=seed, a_init=a_init, with_h0=with_h0, delta_softplus=softplus,
                       u_mean=-3.0 if softplus else 0.0)
    dy, dhT = W.bwd_grads(Bsz, L, D, N, seed=seed + 1, with_dhT=with_dhT)
    x, u = inp.f32("x"), inp.f32("delta")
    if not softplus:
        u = np.abs(u) * np.float32(0.3)       # a positive step size taken as given
    h0 = inp.h0
    got = ss.selscan_bwd(to_dev(x), to_dev(u), to_dev(inp.A), to_dev(inp.f32("B")), to_dev(inp.f32("C")),
                         to_dev(dy), softplus, h0=to_dev(h0), dhT=to_dev(dhT))
    torch.cuda.synchronize()
    ss.check_device_error()
    ref = orc.selscan_bwd(x, u, inp.A, inp.f32("B"), inp.f32("C"), dy, softplus,
                          h0=None if h0 is None else h0.astype(np.float64),
                          ghT=None if dhT is None else dhT.astype(np.float64))
    errs = {k: scaled_err(to_np(got[k]), ref[k]) for k in NAMES}
    assert max(errs.values()) <= TOL[W.F32], errs
    return got


@pytest.mark.parametrize("shape", [(1, 64, 16, 4), (2, 300, 96, 16), (2, 37, 20, 16), (1, 16, 5, 3)])
@pytest.mark.parametrize("softplus", [True, False])
def test_shapes(orc, shape, softplus):
    run(orc, *shape, seed=sum(shape) + softplus, softplus=softplus)


@pytest.mark.parametrize("shape", [(2, 50, 300, 1), (1, 45, 130, 2), (1, 70, 9, 32), (1, 41, 33, 5),
                                   (3, 1, 40, 16)])
def test_lane_group_widths_and_one_step(orc, shape):
    """One thread a chain (N = 1, 2: 128 chains a block), eight (N = 32: four
    chains a warp, two sums a lane left by the reduce-scatter), two with
    padded states (N = 5), and L = 1."""
    run(orc, *shape, seed=sum(shape))


def test_one_segment_when_channels_fill_the_gpu(orc):
    """Enough chains for every resident block: the whole sequence is one
    segment (the carries pass h0 and dhT through unchanged)."""
    run(orc, 4, 40, 4800, 16, seed=17)


def test_without_initial_state_or_final_gradient(orc):
    run(orc, 2, 100, 48, 16, seed=11, with_h0=False, with_dhT=False, a_init="arange")


def test_empty_sequence(orc):
    Bsz, D, N = 2, 24, 16
    dhT = torch.randn(Bsz, D, N, device="cuda")
    e = torch.empty(Bsz, 0, D, device="cuda")
    g = ss.selscan_bwd(e, e, -torch.rand(D, N, device="cuda"), torch.empty(Bsz, 0, N, device="cuda"),
                       torch.empty(Bsz, 0, N, device="cuda"), e, True, dhT=dhT)
    torch.cuda.synchronize()
    assert torch.equal(g["dh0"], dhT) and not g["dA"].any()


def test_state_gradients_are_reproducible(orc):
    """dx, ddelta and dh0 come from one lane each, in a fixed order."""
    inp = W.fwd_inputs(2, 200, 64, 16, seed=13, a_init="loguniform")
    dy, dhT = W.bwd_grads(2, 200, 64, 16, seed=14)
    args = [to_dev(inp.f32(k)) for k in ("x", "delta")] + [to_dev(inp.A)] + \
           [to_dev(inp.f32(k)) for k in ("B", "C")] + [to_dev(dy)]
    g1 = ss.selscan_bwd(*args, True, dhT=to_dev(dhT))
    g2 = ss.selscan_bwd(*args, True, dhT=to_dev(dhT))
    torch.cuda.synchronize()
    for k in ("dx", "ddelta", "dh0"):
        assert torch.equal(g1[k], g2[k])


def test_mamba130m_layer_full_size(orc):
    """The 130M-like layer (Bsz 2, L 2048, D 1536, N 16, softplus on), every
    output compared."""
    w = W.WORKLOADS[2]
    run(orc, w.Bsz, w.L, w.D, w.N, seed=w.seed, with_h0=False, a_init="arange")


def test_selective_scan_autograd(orc):
    """loss.backward() through the differentiable wrapper reaches the CUDA
    backward: its gradients equal the oracle's for the same upstream ones."""
    Bsz, L, D, N = 2, 100, 48, 16
    inp = W.fwd_inputs(Bsz, L, D, N, seed=31, a_init="loguniform", with_h0=True)
    wy, wh = W.bwd_grads(Bsz, L, D, N, seed=32)
    leaves = [to_dev(a).requires_grad_() for a in (inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"),
                                                   inp.f32("C"), inp.h0)]
    x, dl, A, B, C, h0 = leaves
    y, hT = ss.selective_scan(x, dl, A, B, C, True, h0=h0)
    ((y * to_dev(wy)).sum() + (hT * to_dev(wh)).sum()).backward()
    torch.cuda.synchronize()
    ref = orc.selscan_bwd(inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C"), wy, True,
                          h0=inp.h0.astype(np.float64), ghT=wh.astype(np.float64))
    for t, k in zip(leaves, NAMES):
        assert scaled_err(to_np(t.grad), ref[k]) <= TOL[W.F32], k


def run_gated(orc, Bsz, L, D, N, seed, skip=True, gate=True, a_init="loguniform", with_h0=True):
    inp = W.fwd_inputs(Bsz, L, D, N, seed=seed, a_init=a_init, with_h0=with_h0)
    dy, dhT = W.bwd_grads(Bsz, L, D, N, seed=seed + 1)
    Dskip, z = W.gate_inputs(Bsz, L, D, seed=seed + 2)
    x, u, h0 = inp.f32("x"), inp.f32("delta"), inp.h0
    got = ss.selscan_bwd(to_dev(x), to_dev(u), to_dev(inp.A), to_dev(inp.f32("B")), to_dev(inp.f32("C")),
                         to_dev(dy), True, h0=to_dev(h0), dhT=to_dev(dhT),
                         D_skip=to_dev(Dskip) if skip else None, z=to_dev(z) if gate else None)
    torch.cuda.synchronize()
    ss.check_device_error()
    ref = orc.selscan_bwd(x, u, inp.A, inp.f32("B"), inp.f32("C"), dy, True,
                          h0=None if h0 is None else h0.astype(np.float64), ghT=dhT.astype(np.float64),
                          Dskip=Dskip if skip else None, z=z if gate else None)
    names = list(NAMES) + (["dD_skip"] if skip else []) + (["dz"] if gate else [])
    errs = {k: scaled_err(to_np(got[k]), ref["dDskip" if k == "dD_skip" else k]) for k in names}
    assert max(errs.values()) <= TOL[W.F32], errs


@pytest.mark.parametrize("terms", ["both", "skip", "gate"])
@pytest.mark.parametrize("shape", [(2, 300, 96, 16), (1, 41, 33, 5), (1, 70, 9, 32), (2, 50, 300, 1)])
def test_gated_shapes(orc, shape, terms):
    """Each term alone and both, over chain widths of 1, 2, 4 and 8 threads,
    ragged chunks and partly empty blocks."""
    run_gated(orc, *shape, seed=sum(shape) + len(terms), skip=terms != "gate", gate=terms != "skip")


def test_gated_mamba130m_layer_full_size(orc):
    """The 130M-like layer with its skip and gate (Bsz 2, L 2048, D 1536,
    N 16), every output compared."""
    w = W.WORKLOADS[6]
    run_gated(orc, w.Bsz, w.L, w.D, w.N, seed=w.seed, a_init="arange", with_h0=False)


def test_gated_selective_scan_autograd(orc):
    """loss.backward() through the wrapper with D_skip and z reaches the gated
    CUDA backward; every gradient equals the oracle's."""
    Bsz, L, D, N = 2, 100, 48, 16
    inp = W.fwd_inputs(Bsz, L, D, N, seed=41, a_init="loguniform")
    wy, _ = W.bwd_grads(Bsz, L, D, N, seed=42)
    Dskip, z = W.gate_inputs(Bsz, L, D, seed=43)
    leaves = [to_dev(a).requires_grad_() for a in (inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"),
                                                   inp.f32("C"), Dskip, z)]
    x, dl, A, B, C, Dk, zz = leaves
    y, _ = ss.selective_scan(x, dl, A, B, C, True, D_skip=Dk, z=zz)
    (y * to_dev(wy)).sum().backward()
    torch.cuda.synchronize()
    ref = orc.selscan_bwd(inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C"), wy, True,
                          Dskip=Dskip, z=z)
    for t, k in zip(leaves, ("dx", "ddelta", "dA", "dB", "dC", "dDskip", "dz")):
        assert scaled_err(to_np(t.grad), ref[k]) <= TOL[W.F32], k


def test_back_to_back_calls_see_each_others_outputs(orc):
    """Calls launched back to back on one stream, each reading what the one
    before wrote (its kernels start early and wait in the kernel for the
    previous grid): the second call's x is the first call's dx."""
    Bsz, L, D, N = 2, 300, 96, 16
    inp = W.fwd_inputs(Bsz, L, D, N, seed=51, a_init="loguniform")
    dy, _ = W.bwd_grads(Bsz, L, D, N, seed=52, with_dhT=False)
    dev = [to_dev(inp.f32(k)) for k in ("x", "delta")] + [to_dev(inp.A)] + [to_dev(inp.f32(k)) for k in ("B", "C")]
    g1 = ss.selscan_bwd(*dev, to_dev(dy), True, want_dh0=False)
    g2 = ss.selscan_bwd(g1["dx"], *dev[1:], to_dev(dy), True, want_dh0=False)
    torch.cuda.synchronize()
    r1 = orc.selscan_bwd(inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C"), dy, True)
    x2 = to_np(g1["dx"]).astype(np.float32)
    r2 = orc.selscan_bwd(x2, inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C"), dy, True)
    for k in ("dx", "ddelta", "dA", "dB", "dC"):
        assert scaled_err(to_np(g2[k]), r2[k]) <= TOL[W.F32], k
    assert scaled_err(to_np(g1["dx"]), r1["dx"]) <= TOL[W.F32]
