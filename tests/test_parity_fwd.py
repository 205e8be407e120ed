"""selscan_fwd (through the C ABI) against the fp64 oracle.

Metric: max |y_gpu - y_ref| / (1 + |y_ref|); fp32 paths must stay within
1e-4, bf16 input/output paths within 2e-2 (the oracle reads the same
bf16-rounded inputs and keeps full precision). The same metric applies to
the final state hT.
"""
import os

import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import TOL, fwd_dev, oracle_fwd, scaled_err, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture
def env(monkeypatch):
    """Set plan-forcing environment variables for one test only."""
    def set_(**kw):
        for k, v in kw.items():
            monkeypatch.setenv(k, str(v))
    return set_


def check(orc, inp, *, want_hT=True, tol=None, h0_dev=None):
    x, dl, A, B, C, h0 = fwd_dev(inp)
    y, hT = ss.selscan_fwd(x, dl, A, B, C, delta_softplus=inp.delta_softplus, h0=h0,
                           return_final_state=True)
    torch.cuda.synchronize()
    yr, hr = oracle_fwd(orc, inp)
    tol = tol or TOL[inp.dtype]
    ey, eh = scaled_err(to_np(y), yr), scaled_err(to_np(hT), hr)
    assert ey <= tol, f"y error {ey:.3e} > {tol}"
    assert eh <= TOL[W.F32] * (20 if inp.dtype == W.BF16 else 1), f"hT error {eh:.3e}"
    return ey, eh


# ---------------------------------------------------------------- workloads

def test_workload_tiny_all_outputs(orc):
    inp = W.workload_inputs(1)
    check(orc, inp)


def test_workload_mamba130m_fp32_all_outputs(orc):
    inp = W.workload_inputs(2)
    check(orc, inp)


def test_workload_mamba370m_bf16_all_outputs(orc):
    inp = W.workload_inputs(3)
    check(orc, inp)


def test_workload_long_all_outputs(orc):
    """L = 131072 at full size, in the launch configuration the benchmark uses
    (37 chunks): every output and the final state against the oracle over the
    whole workload (201 M outputs; the oracle runs on all host cores, and the
    error is taken slice by slice to bound host memory)."""
    inp = W.workload_inputs(4)
    x, dl, A, B, C, _ = fwd_dev(inp)
    y, hT = ss.selscan_fwd(x, dl, A, B, C, delta_softplus=True, return_final_state=True)
    torch.cuda.synchronize()
    del x, dl, B, C
    yr, hr = orc.selscan_fwd(inp.x, inp.delta, inp.A, inp.B, inp.C, True)
    yg = to_np(y)
    del y
    L = yg.shape[1]
    worst = 0.0
    for t in range(0, L, 8192):
        worst = max(worst, scaled_err(yg[:, t:t + 8192], yr[:, t:t + 8192]))
    assert worst <= TOL[W.F32], worst
    assert scaled_err(to_np(hT), hr) <= TOL[W.F32]


# ---------------------------------------------------------------- shapes

SHAPES = [
    (1, 1, 1, 1), (2, 7, 33, 3), (1, 129, 65, 16), (3, 300, 130, 5), (2, 64, 16, 8),
    (1, 1000, 40, 17), (2, 257, 7, 32), (1, 200, 3, 64), (1, 77, 128, 12), (4, 33, 257, 4),
    (1, 513, 300, 16), (2, 96, 129, 2), (1, 40, 5, 48), (1, 65, 9, 24),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_shapes(orc, shape, dtype):
    Bsz, L, D, N = shape
    seed = sum(shape) * 31 + (dtype == W.BF16)
    inp = W.fwd_inputs(Bsz, L, D, N, seed=seed, dtype=dtype, with_h0=(seed % 2 == 0))
    check(orc, inp)


@pytest.mark.parametrize("softplus", [True, False])
def test_softplus_flag(orc, softplus):
    inp = W.fwd_inputs(2, 150, 70, 16, seed=5, delta_softplus=softplus)
    if not softplus:
        inp.delta = np.abs(inp.delta) * np.float32(0.05)   # a plausible positive step
    check(orc, inp)


# ---------------------------------------------------------------- plans

@pytest.mark.parametrize("chunk", [0, 1, 16, 37, 64, 250, 1000])
def test_forced_chunk_lengths(orc, env, chunk):
    """Chunked parallel scan (carries composed as associative pairs) equals the
    sequential definition for any chunk length, including one per step."""
    env(SELSCAN_CHUNK=chunk)
    inp = W.fwd_inputs(2, 1000, 96, 16, seed=chunk + 3, with_h0=True)
    check(orc, inp)


@pytest.mark.parametrize("dtype,D", [(W.F32, 44), (W.BF16, 40)])
@pytest.mark.parametrize("offset", [0, 1])
def test_one_pass_output_any_alignment(orc, env, dtype, D, offset):
    """The one-pass fused kernel writes y wherever it starts: 16-byte aligned,
    or one element past a boundary (the inputs stay aligned, so the TMA path
    runs). The last warp of each channel tile is partly past D, and L ends in
    a partial stage."""
    L = 333
    env(SELSCAN_CHUNK=L)
    inp = W.fwd_inputs(3, L, D, 16, seed=70 + offset, dtype=dtype, with_h0=True)
    p = ss.fwd_plan(3, L, D, 16, bf16=dtype == W.BF16)
    assert p["chunks"] == 1 and p["launches"] == 1   # aligned rows: the fused kernel, one pass
    x, dl, A, B, C, h0 = fwd_dev(inp)
    buf = torch.full((x.numel() + offset,), float("nan"), device="cuda", dtype=x.dtype)
    y = buf[offset:].view(x.shape)
    assert (y.data_ptr() % 16 == 0) == (offset == 0)
    ss.selscan_fwd(x, dl, A, B, C, delta_softplus=True, h0=h0, y=y)
    torch.cuda.synchronize()
    yr, _ = oracle_fwd(orc, inp)
    assert scaled_err(to_np(y), yr) <= TOL[dtype]
    if offset:
        assert torch.isnan(buf[0])   # nothing written before y


@pytest.mark.parametrize("nsplit", [2, 4])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_threads_per_chain(orc, env, nsplit, dtype):
    env(SELSCAN_NSPLIT=nsplit, SELSCAN_CHUNK=90)
    inp = W.fwd_inputs(2, 333, 100, 16, seed=nsplit, dtype=dtype, with_h0=True)
    check(orc, inp)


@pytest.mark.parametrize("stages", [2, 3, 4, 8])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_ring_depths(orc, env, stages, dtype):
    """Any number of shared-memory buffers in flight per CTA (the ring the
    tiles arrive in) gives the same result, with chunk lengths that are and
    are not multiples of the 16-step tile, and a ragged last chunk."""
    env(SELSCAN_TMA_STAGES=stages, SELSCAN_CHUNK=16 * stages + 5)
    inp = W.fwd_inputs(2, 401, 136, 16, seed=stages, dtype=dtype, with_h0=True)
    check(orc, inp)


def test_chunked_matches_sequential_closely(env):
    inp = W.fwd_inputs(1, 4096, 256, 16, seed=77, with_h0=True)
    outs = []
    for chunk in (0, 128):
        env(SELSCAN_CHUNK=chunk)
        x, dl, A, B, C, h0 = fwd_dev(inp)
        outs.append(ss.selscan_fwd(x, dl, A, B, C, True, h0, return_final_state=True))
    torch.cuda.synchronize()
    assert scaled_err(to_np(outs[1][0]), to_np(outs[0][0])) < 2e-5
    assert scaled_err(to_np(outs[1][1]), to_np(outs[0][1])) < 2e-5


# ---------------------------------------------------------------- state handling

@pytest.mark.parametrize("cut", [1, 100, 511])
def test_split_and_resume(orc, cut):
    inp = W.fwd_inputs(2, 512, 80, 16, seed=cut, with_h0=True)
    x, dl, A, B, C, h0 = fwd_dev(inp)
    y1, h1 = ss.selscan_fwd(x[:, :cut].contiguous(), dl[:, :cut].contiguous(), A, B[:, :cut].contiguous(),
                            C[:, :cut].contiguous(), True, h0, return_final_state=True)
    y2, h2 = ss.selscan_fwd(x[:, cut:].contiguous(), dl[:, cut:].contiguous(), A, B[:, cut:].contiguous(),
                            C[:, cut:].contiguous(), True, h1, return_final_state=True)
    torch.cuda.synchronize()
    yr, hr = oracle_fwd(orc, inp)
    assert scaled_err(np.concatenate([to_np(y1), to_np(y2)], axis=1), yr) <= TOL[W.F32]
    assert scaled_err(to_np(h2), hr) <= TOL[W.F32]


def test_resume_in_place_h0_is_hT(orc):
    inp = W.fwd_inputs(1, 300, 64, 16, seed=9, with_h0=True)
    x, dl, A, B, C, h0 = fwd_dev(inp)
    y, hT = ss.selscan_fwd(x, dl, A, B, C, True, h0, hT=h0)
    torch.cuda.synchronize()
    yr, hr = oracle_fwd(orc, inp)
    assert hT.data_ptr() == h0.data_ptr()
    assert scaled_err(to_np(y), yr) <= TOL[W.F32] and scaled_err(to_np(h0), hr) <= TOL[W.F32]


def test_empty_sequence_copies_state():
    h0 = torch.randn(2, 5, 16, device="cuda")
    e = torch.empty(2, 0, 5, device="cuda")
    A = -torch.ones(5, 16, device="cuda")
    eb = torch.empty(2, 0, 16, device="cuda")
    y, hT = ss.selscan_fwd(e, e, A, eb, eb, True, h0, return_final_state=True)
    torch.cuda.synchronize()
    assert y.shape == (2, 0, 5) and torch.equal(hT, h0)
    _, hz = ss.selscan_fwd(e, e, A, eb, eb, True, None, return_final_state=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(hz) == 0


def test_empty_batch_and_channels():
    A = -torch.ones(0, 4, device="cuda")
    z = torch.empty(0, 10, 0, device="cuda")
    y = ss.selscan_fwd(z, z, A, torch.empty(0, 10, 4, device="cuda"), torch.empty(0, 10, 4, device="cuda"))
    assert y.shape == (0, 10, 0)


def test_in_place_output_over_x(orc):
    inp = W.fwd_inputs(2, 200, 50, 16, seed=21)
    x, dl, A, B, C, _ = fwd_dev(inp)
    ss.selscan_fwd(x, dl, A, B, C, True, y=x)
    torch.cuda.synchronize()
    yr, _ = oracle_fwd(orc, inp)
    assert scaled_err(to_np(x), yr) <= TOL[W.F32]


def test_unaligned_inputs_take_scalar_path(orc):
    """B and C starting 4 bytes past a 16-byte boundary cannot use vector loads."""
    inp = W.fwd_inputs(2, 100, 40, 16, seed=4)
    x, dl, A, _, _, _ = fwd_dev(inp)
    n = inp.B.size
    bb = torch.empty(n + 1, device="cuda"); bb[1:] = to_dev(inp.B).reshape(-1)
    cb = torch.empty(n + 1, device="cuda"); cb[1:] = to_dev(inp.C).reshape(-1)
    B = bb[1:].view(inp.B.shape); C = cb[1:].view(inp.C.shape)
    assert B.data_ptr() % 16 != 0
    y = ss.selscan_fwd(x, dl, A, B, C, True)
    torch.cuda.synchronize()
    yr, _ = oracle_fwd(orc, inp)
    assert scaled_err(to_np(y), yr) <= TOL[W.F32]


def test_side_stream_and_determinism():
    inp = W.fwd_inputs(2, 700, 200, 16, seed=12, with_h0=True)
    x, dl, A, B, C, h0 = fwd_dev(inp)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        y1 = ss.selscan_fwd(x, dl, A, B, C, True, h0)
        y2 = ss.selscan_fwd(x, dl, A, B, C, True, h0)
    s.synchronize()
    assert torch.equal(y1, y2)


def test_host_tensors_round_trip(orc):
    inp = W.fwd_inputs(1, 64, 32, 16, seed=2)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    y = ss.selscan_fwd(t(inp.x), t(inp.delta), t(inp.A), t(inp.B), t(inp.C), True)
    assert y.device.type == "cpu"
    yr, _ = oracle_fwd(orc, inp)
    assert scaled_err(y.double().numpy(), yr) <= TOL[W.F32]


# ---------------------------------------------------------------- errors

def test_invalid_arguments_raise():
    x = torch.randn(1, 8, 4, device="cuda")
    A = -torch.ones(4, 65, device="cuda")
    B = torch.randn(1, 8, 65, device="cuda")
    with pytest.raises(ss.SelscanError) as e:
        ss.selscan_fwd(x, x.clone(), A, B, B.clone())
    assert e.value.code == ss.ERR_UNSUPPORTED
    A = -torch.ones(4, 4, device="cuda")
    B = torch.randn(1, 8, 4, device="cuda")
    with pytest.raises(ss.SelscanError) as e:
        ss.selscan_fwd(x, x.clone(), A, B, B.clone(), y=B.view(1, 8, 4))   # y overlaps B
    assert e.value.code == ss.ERR_INVALID_ARG
    ss.check_device_error()


@pytest.mark.parametrize("shape", [(2, 300, 256, 16), (1, 129, 96, 8), (3, 70, 64, 32), (1, 50, 128, 64)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_plain_load_path(orc, env, shape, dtype):
    """The kernels that read global memory directly (used when TMA's
    alignment rules do not hold) give the same results as the TMA path."""
    env(SELSCAN_NO_TMA=1, SELSCAN_CHUNK=64)
    Bsz, L, D, N = shape
    inp = W.fwd_inputs(Bsz, L, D, N, seed=L + D, dtype=dtype, with_h0=True)
    check(orc, inp)


def test_device_fault_word_clear_after_normal_runs():
    inp = W.fwd_inputs(1, 256, 128, 16, seed=1)
    x, dl, A, B, C, _ = fwd_dev(inp)
    ss.selscan_fwd(x, dl, A, B, C, True)
    ss.check_device_error()


def test_plan_query_matches_launches():
    p1 = ss.fwd_plan(1, 64, 16, 4)
    assert p1 == {"chunks": 1, "chunk_len": 64, "launches": 1, "workspace_bytes": 0}
    p2 = ss.fwd_plan(2, 2048, 1536, 16)
    # chunked on the fused path: the control-word clear, then the fused kernel
    assert p2["chunks"] > 1 and p2["launches"] == 2 and p2["workspace_bytes"] > 0
    assert p2["chunks"] * p2["chunk_len"] >= 2048 > (p2["chunks"] - 1) * p2["chunk_len"]
    assert ss.fwd_plan(0, 10, 5, 4)["launches"] == 0
