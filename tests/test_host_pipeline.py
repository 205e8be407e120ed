"""selscan_fwd_host: the forward scan from host buffers, with copies in,
scan and copies out pipelined over pieces of the sequence (each piece
starting from the device-resident final state of the one before). Results
against the fp64 oracle, for many pieces, a ragged last piece, both dtypes,
page-locked and pageable buffers, in-place output, and L = 0."""
import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import TOL, oracle_fwd, scaled_err

pytestmark = pytest.mark.gpu


def host(inp, pin):
    def t(a):
        if a is None:
            return None
        if a.dtype == np.uint16:     # bf16 bits
            h = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
        else:
            h = torch.from_numpy(np.ascontiguousarray(a))
        return h.pin_memory() if pin else h
    return [t(inp.x), t(inp.delta), t(inp.A), t(inp.B), t(inp.C), t(inp.h0)]


def as_np(t):
    return (t.float() if t.dtype == torch.bfloat16 else t).numpy().astype(np.float64)


@pytest.mark.parametrize("piece", [0, 50, 64])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("pin", [True, False])
def test_pieces_match_oracle(orc, monkeypatch, piece, dtype, pin):
    if piece:
        monkeypatch.setenv("SELSCAN_HOST_PIECE", str(piece))
    inp = W.fwd_inputs(3, 333, 136, 16, seed=piece + 5, dtype=dtype, with_h0=True)
    x, dl, A, B, C, h0 = host(inp, pin)
    y, hT = ss.selscan_fwd(x, dl, A, B, C, True, h0, return_final_state=True)
    assert y.device.type == "cpu" and hT.device.type == "cpu"
    yr, hr = oracle_fwd(orc, inp)
    assert scaled_err(as_np(y), yr) <= TOL[dtype]
    assert scaled_err(as_np(hT), hr) <= TOL[W.F32] * (20 if dtype == W.BF16 else 1)


def test_workload_mamba130m_from_host(orc):
    inp = W.workload_inputs(2)
    x, dl, A, B, C, _ = host(inp, True)
    y = ss.selscan_fwd(x, dl, A, B, C, True)
    yr, _ = oracle_fwd(orc, inp)
    assert scaled_err(as_np(y), yr) <= TOL[W.F32]


def test_no_state_in_or_out_and_in_place_output(orc, monkeypatch):
    monkeypatch.setenv("SELSCAN_HOST_PIECE", "40")
    inp = W.fwd_inputs(2, 170, 64, 8, seed=9)
    x, dl, A, B, C, _ = host(inp, True)
    yr, _ = oracle_fwd(orc, inp)
    y = ss.selscan_fwd(x, dl, A, B, C, True, y=x)       # y written over x, piece by piece
    assert y.data_ptr() == x.data_ptr()
    assert scaled_err(as_np(y), yr) <= TOL[W.F32]


def test_empty_sequence_from_host():
    h0 = torch.randn(2, 8, 4)
    x = torch.empty(2, 0, 8)
    B = torch.empty(2, 0, 4)
    A = -torch.ones(8, 4)
    y, hT = ss.selscan_fwd(x, x.clone(), A, B, B.clone(), True, h0, return_final_state=True)
    assert torch.equal(hT, h0) and y.shape == (2, 0, 8)
    _, hT0 = ss.selscan_fwd(x, x.clone(), A, B, B.clone(), True, None, return_final_state=True)
    assert torch.count_nonzero(hT0) == 0


def test_host_calls_behind_busy_device_are_deterministic():
    """Host calls issued while the current stream still has work queued wait
    for it, and two such calls give bit-identical outputs."""
    inp = W.fwd_inputs(1, 256, 128, 16, seed=3)
    x, dl, A, B, C, _ = host(inp, True)
    busy = torch.randn(4096, 4096, device="cuda")
    for _ in range(4):
        busy = busy @ busy.T / 4096.0
    y1 = ss.selscan_fwd(x, dl, A, B, C, True)
    y2 = ss.selscan_fwd(x, dl, A, B, C, True)
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("form", ["gated", "zoh", "gated_zoh"])
def test_gated_and_zoh_from_host(orc, monkeypatch, form):
    """selscan_fwd_host_ex: the block's skip and gate and the zero-order hold
    from host buffers, over several pieces, against the oracle."""
    monkeypatch.setenv("SELSCAN_HOST_PIECE", "64")
    inp = W.fwd_inputs(2, 300, 96, 16, seed=61, with_h0=True)
    x, dl, A, B, C, h0 = host(inp, True)
    gated, zoh = form != "zoh", form != "gated"
    Dskip, z = W.gate_inputs(2, 300, 96, seed=61)
    kw = {"D_skip": torch.from_numpy(Dskip).pin_memory(), "z": torch.from_numpy(z).pin_memory()} if gated else {}
    y, hT = ss.selscan_fwd(x, dl, A, B, C, True, h0, return_final_state=True, zoh=zoh, **kw)
    assert y.device.type == "cpu"
    yr, hr = orc.selscan_fwd(inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C"), True,
                             inp.h0.astype(np.float64), Dskip=Dskip if gated else None, z=z if gated else None,
                             zoh=zoh)
    assert scaled_err(as_np(y), yr) <= TOL[W.F32]
    assert scaled_err(as_np(hT), hr) <= TOL[W.F32]


def test_host_empty_round_trip_and_forward(orc):
    """Tensors from the library's page-locked host allocator: asynchronous
    copies both ways keep every byte, and the host-buffer forward reads and
    writes them like any pinned buffer."""
    t = ss.host_empty((257, 33))
    src = torch.randn(257, 33)
    t.copy_(src)
    d = t.to("cuda", non_blocking=True)
    back = ss.host_empty((257, 33))
    back.copy_(d, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    inp = W.fwd_inputs(2, 300, 64, 16, seed=71)
    host = [ss.host_empty(a.shape) for a in (inp.x, inp.delta, inp.A, inp.B, inp.C)]
    for h, a in zip(host, (inp.x, inp.delta, inp.A, inp.B, inp.C)):
        h.copy_(torch.from_numpy(a))
    y = ss.host_empty(inp.x.shape)
    ss.selscan_fwd(*host, True, y=y)
    yr, _ = orc.selscan_fwd(inp.x, inp.delta, inp.A, inp.B, inp.C, True)
    assert scaled_err(y.numpy(), yr) <= TOL[W.F32]
