"""selscan_fwd_gated / selscan_step_gated: the block's skip and SiLU gate fused
into the scan's read-out, y = (scan + Dskip[d] x) * silu(z), against the fp64
oracle's gated entry points. Covers the fused TMA kernel (16-byte rows,
softplus on), the plain-load kernels (softplus off, or rows that are not
multiples of 16 bytes), chunked and one-pass plans, both dtypes, each term
alone, in-place output over z, and the decode step."""
import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import TOL, fwd_dev, scaled_err, to_dev, to_np

pytestmark = pytest.mark.gpu


def run(orc, inp, Dskip, z, with_skip=True, with_gate=True, chunk=None, monkeypatch=None, y_is_z=False):
    if chunk is not None:
        monkeypatch.setenv("SELSCAN_CHUNK", str(chunk))
    x, dl, A, B, C, h0 = fwd_dev(inp)
    dD = to_dev(Dskip) if with_skip else None
    dz = to_dev(z, inp.dtype) if with_gate else None
    y_out = dz if y_is_z else None
    y, hT = ss.selscan_fwd(x, dl, A, B, C, inp.delta_softplus, h0, return_final_state=True,
                           D_skip=dD, z=dz, y=y_out)
    torch.cuda.synchronize()
    ss.check_device_error()
    zf = (W.bf16_bits_to_f32(z) if inp.dtype == W.BF16 else z) if with_gate else None
    yr, hr = orc.selscan_fwd(inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C"),
                             inp.delta_softplus, None if inp.h0 is None else inp.h0.astype(np.float64),
                             Dskip=Dskip if with_skip else None, z=zf)
    assert scaled_err(to_np(y), yr) <= TOL[inp.dtype]
    assert scaled_err(to_np(hT), hr) <= TOL[W.F32] * (20 if inp.dtype == W.BF16 else 1)
    return y


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("chunk", [0, 100])
@pytest.mark.parametrize("terms", ["both", "skip", "gate"])
def test_fused_path(orc, monkeypatch, dtype, chunk, terms):
    """16-byte rows and softplus: the gate runs in the fused kernel's read-out."""
    Bsz, L, D, N = 2, 333, 136, 16
    inp = W.fwd_inputs(Bsz, L, D, N, seed=chunk + len(terms), dtype=dtype, with_h0=True)
    Dskip, z = W.gate_inputs(Bsz, L, D, seed=chunk + 1, dtype=dtype)
    run(orc, inp, Dskip, z, with_skip=terms != "gate", with_gate=terms != "skip", chunk=chunk,
        monkeypatch=monkeypatch)


@pytest.mark.parametrize("shape", [(2, 200, 130, 16), (1, 150, 64, 8), (3, 97, 40, 4), (1, 120, 64, 32)])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_other_shapes(orc, shape, dtype):
    """Rows that are not 16-byte multiples (plain-load kernels), and N of 4,
    8 and 32 (several threads per chain)."""
    Bsz, L, D, N = shape
    inp = W.fwd_inputs(Bsz, L, D, N, seed=sum(shape), dtype=dtype, with_h0=True)
    Dskip, z = W.gate_inputs(Bsz, L, D, seed=sum(shape) + 1, dtype=dtype)
    run(orc, inp, Dskip, z)


def test_softplus_off_takes_plain_kernels(orc):
    inp = W.fwd_inputs(2, 150, 128, 16, seed=5, delta_softplus=False)
    inp.delta = np.abs(inp.delta) * np.float32(0.05)
    Dskip, z = W.gate_inputs(2, 150, 128, seed=6)
    run(orc, inp, Dskip, z)


def test_workload_mamba130m_gated(orc):
    """The 130M-like layer (Bsz=2 L=2048 D=1536 N=16) with the block's skip and
    gate, every output against the oracle."""
    inp = W.workload_inputs(2)
    Dskip, z = W.gate_inputs(2, 2048, 1536, seed=202)
    run(orc, inp, Dskip, z)


def test_output_written_over_z(orc):
    inp = W.fwd_inputs(2, 260, 128, 16, seed=8)
    Dskip, z = W.gate_inputs(2, 260, 128, seed=9)
    run(orc, inp, Dskip, z, y_is_z=True)


def test_gated_forward_rejects_partial_overlap():
    x = torch.randn(1, 8, 16, device="cuda")
    A = -torch.ones(16, 4, device="cuda")
    B = torch.randn(1, 8, 4, device="cuda")
    buf = torch.randn(2 * 8 * 16, device="cuda")
    z = buf[:128].view(1, 8, 16)
    y = buf[64:192].view(1, 8, 16)
    with pytest.raises(ss.SelscanError) as e:
        ss.selscan_fwd(x, x.clone(), A, B, B.clone(), True, z=z, y=y)
    assert e.value.code == ss.ERR_INVALID_ARG


@pytest.mark.parametrize("N", [3, 16, 64])
def test_gated_decode_step(orc, N):
    Bsz, D = 4, 77
    g = np.random.default_rng(N)
    st = g.standard_normal((Bsz, D, N)).astype(np.float32)
    x = g.standard_normal((Bsz, D)).astype(np.float32)
    dl = (g.random((Bsz, D)) * 0.2).astype(np.float32)
    A = (-(0.5 + g.random((D, N)) * 4)).astype(np.float32)
    B = g.standard_normal((Bsz, N)).astype(np.float32)
    C = g.standard_normal((Bsz, N)).astype(np.float32)
    Dskip, z = W.gate_inputs(Bsz, 1, D, seed=N, steps=True)
    s_dev = to_dev(st)
    y = ss.selscan_step(s_dev, to_dev(x), to_dev(dl), to_dev(A), to_dev(B), to_dev(C),
                        D_skip=to_dev(Dskip), z=to_dev(z))
    torch.cuda.synchronize()
    s_ref = st.astype(np.float64)
    y_ref = orc.selscan_step(s_ref, x, dl, A, B, C, Dskip=Dskip, z=z)
    assert scaled_err(to_np(y), y_ref) <= TOL[W.F32]
    assert scaled_err(to_np(s_dev), s_ref) <= TOL[W.F32]


def test_gated_steps_equal_gated_forward():
    Bsz, L, D, N = 2, 30, 64, 16
    inp = W.fwd_inputs(Bsz, L, D, N, seed=12, with_h0=True)
    Dskip, z = W.gate_inputs(Bsz, L, D, seed=13)
    g = to_dev
    dl = (np.maximum(inp.delta, 0) + np.log1p(np.exp(-np.abs(inp.delta.astype(np.float64))))).astype(np.float32)
    y_f, h_f = ss.selscan_fwd(g(inp.x), g(dl), g(inp.A), g(inp.B), g(inp.C), False, g(inp.h0),
                              return_final_state=True, D_skip=g(Dskip), z=g(z))
    s = g(inp.h0)
    ys = [ss.selscan_step(s, g(inp.x[:, t]), g(dl[:, t]), g(inp.A), g(inp.B[:, t]), g(inp.C[:, t]),
                          D_skip=g(Dskip), z=g(z[:, t])) for t in range(L)]
    torch.cuda.synchronize()
    assert scaled_err(to_np(torch.stack(ys, dim=1)), to_np(y_f)) < 1e-5
    assert scaled_err(to_np(s), to_np(h_f)) < 1e-5
