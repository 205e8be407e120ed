"""The differentiable wrapper ``selective_scan`` on the CPU: its forward and
backward are routed to stand-ins built on the fp64 oracle, so what is tested
here is the wrapper's own plumbing (which saved tensor goes where, which
gradient is returned for which input, h0 and hT optional). The gradients are
compared with torch's autograd of the recurrence unrolled with tensor ops.
The CUDA path behind it is covered by the backward parity tests."""
import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W


def fake_fwd(orc):
    def f(x, delta, A, B, C, delta_softplus=False, h0=None, return_final_state=False, D_skip=None, z=None, **kw):
        n = lambda t: None if t is None else t.detach().numpy()
        y, hT = orc.selscan_fwd(x.detach().numpy(), delta.detach().numpy(), A.detach().numpy(),
                                B.detach().numpy(), C.detach().numpy(), delta_softplus,
                                h0=None if h0 is None else h0.detach().numpy().astype(np.float64),
                                Dskip=n(D_skip), z=n(z))
        return torch.from_numpy(y), torch.from_numpy(hT)
    return f


def fake_bwd(orc):
    def f(x, delta, A, B, C, dy, delta_softplus=False, h0=None, dhT=None, want_dh0=True, stream=None,
          check=False, D_skip=None, z=None):
        n = lambda t: None if t is None else t.detach().numpy().astype(np.float64)
        f32 = lambda t: None if t is None else t.detach().numpy()
        g = orc.selscan_bwd(x.detach().numpy(), delta.detach().numpy(), A.detach().numpy(),
                            B.detach().numpy(), C.detach().numpy(), n(dy), delta_softplus, h0=n(h0), ghT=n(dhT),
                            Dskip=f32(D_skip), z=f32(z))
        out = {("dD_skip" if k == "dDskip" else k): torch.from_numpy(v) for k, v in g.items()}
        if not want_dh0:
            del out["dh0"]
        return out
    return f


def unrolled(x, delta, A, B, C, h0, softplus):
    dl = torch.nn.functional.softplus(delta) if softplus else delta
    Bsz, L, D = x.shape
    h = h0 if h0 is not None else torch.zeros(Bsz, D, A.shape[1], dtype=x.dtype)
    ys = []
    for s in range(L):
        d = dl[:, s, :, None]
        h = torch.exp(d * A[None]) * h + d * B[:, s, None, :] * x[:, s, :, None]
        ys.append((h * C[:, s, None, :]).sum(-1))
    return torch.stack(ys, 1), h


@pytest.mark.parametrize("with_h0,use_hT,softplus", [(True, True, True), (False, False, True), (True, False, False)])
def test_selective_scan_gradients(orc, monkeypatch, with_h0, use_hT, softplus):
    monkeypatch.setattr(ss, "selscan_fwd", fake_fwd(orc))
    monkeypatch.setattr(ss, "selscan_bwd", fake_bwd(orc))
    Bsz, L, D, N = 2, 9, 3, 4
    inp = W.fwd_inputs(Bsz, L, D, N, seed=21, a_init="loguniform", with_h0=with_h0)
    wy = torch.from_numpy(W.normal(W.rng(22, 1), (Bsz, L, D))).double()
    wh = torch.from_numpy(W.normal(W.rng(22, 2), (Bsz, D, N))).double()
    u = inp.f32("delta") if softplus else np.abs(inp.f32("delta")) * np.float32(0.3)

    def leaves(dtype):
        ts = [torch.tensor(np.asarray(a, np.float64), dtype=dtype, requires_grad=True)
              for a in (inp.f32("x"), u, inp.A, inp.f32("B"), inp.f32("C"))]
        h0 = torch.tensor(inp.h0.astype(np.float64), dtype=dtype, requires_grad=True) if with_h0 else None
        return ts, h0

    (x, dl, A, B, C), h0 = leaves(torch.float32)
    y, hT = ss.selective_scan(x, dl, A, B, C, softplus, h0=h0)
    loss = (y * wy).sum() + ((hT * wh).sum() if use_hT else 0.0)
    loss.backward()

    (rx, rdl, rA, rB, rC), rh0 = leaves(torch.float64)
    ry, rhT = unrolled(rx, rdl, rA, rB, rC, rh0, softplus)
    rloss = (ry * wy).sum() + ((rhT * wh).sum() if use_hT else 0.0)
    rloss.backward()
    assert torch.allclose(y.double(), ry, rtol=1e-9, atol=1e-12)
    pairs = [(x, rx), (dl, rdl), (A, rA), (B, rB), (C, rC)] + ([(h0, rh0)] if with_h0 else [])
    for got, ref in pairs:
        assert got.grad.dtype == torch.float32        # the stand-in's fp64 gradients, cast by autograd
        assert torch.allclose(got.grad.double(), ref.grad, rtol=1e-6, atol=1e-7)


def test_smoke_backward_block_runs_on_stand_ins(orc, monkeypatch):
    """The backward block of the smoke check, with selscan_bwd routed to the
    oracle-backed stand-in (so its own code runs here, on the CPU)."""
    import numpy as np
    import __graft_entry__ as ge
    monkeypatch.setattr(ss, "selscan_bwd", fake_bwd(orc))
    err = lambda got, ref: float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref))))
    ge._smoke_backward(torch.device("cpu"), err)


def test_selective_scan_check_reaches_both_passes(orc, monkeypatch):
    """selective_scan(check=True) asks the forward and the backward call to
    wait for their kernels and report a timed-out wait."""
    seen = []
    fwd, bwd = fake_fwd(orc), fake_bwd(orc)

    def f(*a, check=False, **kw):
        seen.append(("fwd", check))
        return fwd(*a, **kw)

    def b(*a, check=False, **kw):
        seen.append(("bwd", check))
        return bwd(*a, **kw)

    monkeypatch.setattr(ss, "selscan_fwd", f)
    monkeypatch.setattr(ss, "selscan_bwd", b)
    inp = W.fwd_inputs(1, 5, 2, 4, seed=23, a_init="loguniform")
    x, dl, A, B, C = (torch.tensor(inp.f32(k) if k != "A" else inp.A, requires_grad=True)
                      for k in ("x", "delta", "A", "B", "C"))
    y, hT = ss.selective_scan(x, dl, A, B, C, True, check=True)
    y.sum().backward()
    assert seen == [("fwd", True), ("bwd", True)]


@pytest.mark.parametrize("skip,gate", [(True, True), (True, False), (False, True)])
def test_selective_scan_gated_gradients(orc, monkeypatch, skip, gate):
    """The block's skip and gate through the wrapper: D_skip and z reach the
    forward and the backward, and their gradients come back to them."""
    monkeypatch.setattr(ss, "selscan_fwd", fake_fwd(orc))
    monkeypatch.setattr(ss, "selscan_bwd", fake_bwd(orc))
    Bsz, L, D, N = 2, 7, 3, 4
    inp = W.fwd_inputs(Bsz, L, D, N, seed=31, a_init="loguniform")
    zz = W.normal(W.rng(32, 1), (Bsz, L, D))
    dsk = W.normal(W.rng(32, 2), (D,))
    wy = torch.from_numpy(W.normal(W.rng(32, 3), (Bsz, L, D))).double()

    def leaves(dtype):
        ts = [torch.tensor(np.asarray(a, np.float64), dtype=dtype, requires_grad=True)
              for a in (inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C"), dsk, zz)]
        return ts

    x, dl, A, B, C, Dk, z = leaves(torch.float32)
    y, _ = ss.selective_scan(x, dl, A, B, C, True, D_skip=Dk if skip else None, z=z if gate else None)
    (y * wy).sum().backward()

    rx, rdl, rA, rB, rC, rDk, rz = leaves(torch.float64)
    ry, _ = unrolled(rx, rdl, rA, rB, rC, None, True)
    if skip:
        ry = ry + rDk * rx
    if gate:
        ry = ry * torch.nn.functional.silu(rz)
    (ry * wy).sum().backward()
    assert torch.allclose(y.double(), ry, rtol=1e-9, atol=1e-12)
    pairs = [(x, rx), (dl, rdl), (A, rA), (B, rB), (C, rC)] + ([(Dk, rDk)] if skip else []) + \
        ([(z, rz)] if gate else [])
    for got, ref in pairs:
        assert torch.allclose(got.grad.double(), ref.grad, rtol=1e-6, atol=1e-7)
