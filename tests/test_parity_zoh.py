"""The zero-order-hold discretisation (selscan_fwd_ex / selscan_step_ex with
SELSCAN_FLAG_ZOH): Bbar = dl * B * (e^w - 1)/w, w = dl * A, against the fp64
oracle's zoh option. Covers small |w| (the series branch), A = 0 (the limit),
large |w|, chunked and one-pass plans, both dtypes, the skip and gate
together with it, and the decode step."""
import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import TOL, fwd_dev, scaled_err, to_dev, to_np

pytestmark = pytest.mark.gpu


def check(orc, inp, gate=None):
    x, dl, A, B, C, h0 = fwd_dev(inp)
    kw = {}
    if gate is not None:
        kw = dict(D_skip=to_dev(gate[0]), z=to_dev(gate[1], inp.dtype))
    y, hT = ss.selscan_fwd(x, dl, A, B, C, inp.delta_softplus, h0, return_final_state=True, zoh=True, **kw)
    torch.cuda.synchronize()
    ss.check_device_error()
    zf = None
    if gate is not None:
        zf = W.bf16_bits_to_f32(gate[1]) if inp.dtype == W.BF16 else gate[1]
    yr, hr = orc.selscan_fwd(inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C"),
                             inp.delta_softplus, None if inp.h0 is None else inp.h0.astype(np.float64),
                             Dskip=None if gate is None else gate[0], z=zf, zoh=True)
    assert scaled_err(to_np(y), yr) <= TOL[inp.dtype]
    assert scaled_err(to_np(hT), hr) <= TOL[W.F32] * (20 if inp.dtype == W.BF16 else 1)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("chunk", [0, 64])
@pytest.mark.parametrize("u_mean", [-6.0, -3.0, 0.0])
def test_zoh_forward(orc, monkeypatch, dtype, chunk, u_mean):
    """u_mean -6 keeps most |dl * A| under 1/16 (series branch); 0 puts most
    above it."""
    monkeypatch.setenv("SELSCAN_CHUNK", str(chunk))
    inp = W.fwd_inputs(2, 300, 136, 16, seed=int(10 - u_mean) + chunk, dtype=dtype, u_mean=u_mean, with_h0=True)
    check(orc, inp)


def test_zoh_with_zero_entries_of_A(orc):
    inp = W.fwd_inputs(2, 200, 64, 16, seed=3, with_h0=True)
    inp.A[:, ::3] = 0.0
    check(orc, inp)


@pytest.mark.parametrize("N", [4, 12, 32, 64])
def test_zoh_state_sizes(orc, N):
    inp = W.fwd_inputs(1, 150, 96, N, seed=N, with_h0=True)
    check(orc, inp)


def test_zoh_with_skip_and_gate(orc):
    inp = W.fwd_inputs(2, 256, 128, 16, seed=21)
    check(orc, inp, gate=W.gate_inputs(2, 256, 128, seed=22))


def test_zoh_rejects_unknown_flags():
    x = torch.randn(1, 8, 16, device="cuda")
    A = -torch.ones(16, 4, device="cuda")
    B = torch.randn(1, 8, 4, device="cuda")
    y = torch.empty_like(x)
    rc = ss.lib().selscan_fwd_ex(x.data_ptr(), x.data_ptr(), A.data_ptr(), B.data_ptr(), B.data_ptr(),
                                 None, None, y.data_ptr(), 1, 8, 16, 4, 0, 4, None, None,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == ss.ERR_INVALID_ARG


@pytest.mark.parametrize("N", [3, 16])
def test_zoh_decode_step(orc, N):
    Bsz, D = 4, 77
    g = np.random.default_rng(N + 50)
    st = g.standard_normal((Bsz, D, N)).astype(np.float32)
    x = g.standard_normal((Bsz, D)).astype(np.float32)
    dl = (g.random((Bsz, D)) * 0.3).astype(np.float32)
    A = (-(g.random((D, N)) * 4)).astype(np.float32)
    A[:, 0] = 0.0
    B = g.standard_normal((Bsz, N)).astype(np.float32)
    C = g.standard_normal((Bsz, N)).astype(np.float32)
    s_dev = to_dev(st)
    y = ss.selscan_step(s_dev, to_dev(x), to_dev(dl), to_dev(A), to_dev(B), to_dev(C), zoh=True)
    torch.cuda.synchronize()
    s_ref = st.astype(np.float64)
    y_ref = orc.selscan_step(s_ref, x, dl, A, B, C, zoh=True)
    assert scaled_err(to_np(y), y_ref) <= TOL[W.F32]
    assert scaled_err(to_np(s_dev), s_ref) <= TOL[W.F32]
