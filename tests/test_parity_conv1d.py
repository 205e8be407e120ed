"""selscan_conv1d / selscan_conv1d_step: the causal depthwise convolution and
SiLU in front of the scan, against the fp64 oracle. Covers tap counts 1..8,
runs that split the sequence (the kernel's 64-step runs) and ragged tails,
ragged channel counts, both dtypes, with and without a carried state, the
state handed from one piece to the next, and the decode step."""
import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import TOL, scaled_err, to_dev, to_np

pytestmark = pytest.mark.gpu


def f32(x, dtype):
    return W.bf16_bits_to_f32(x) if dtype == W.BF16 else x


@pytest.mark.parametrize("K", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("with_state", [False, True])
def test_conv1d_matches_oracle(orc, K, dtype, with_state):
    Bsz, L, D = 3, 200, 300
    x, w, bias, state = W.conv_inputs(Bsz, L, D, K, seed=K + 10 * with_state, dtype=dtype, with_state=with_state)
    out, st = ss.conv1d(to_dev(x, dtype), to_dev(w), to_dev(bias), state_in=to_dev(state), return_state=True)
    torch.cuda.synchronize()
    ref, st_ref = orc.conv1d(f32(x, dtype), w, bias, state_in=state)
    assert scaled_err(to_np(out), ref) <= TOL[dtype]
    assert np.array_equal(to_np(st).astype(np.float32), st_ref)


@pytest.mark.parametrize("L", [1, 3, 15, 16, 17, 31, 32, 33, 63, 64, 65, 129])
@pytest.mark.parametrize("D", [70, 72])
@pytest.mark.parametrize("vec", ["1", "0"])
def test_conv1d_run_boundaries(orc, monkeypatch, L, D, vec):
    """Short segments of the streaming kernel (four channels per thread,
    D % 4 == 0) and runs of 64 (one channel per thread), ragged tails, and
    both kernels on the same D."""
    monkeypatch.setenv("SELSCAN_CONV_VEC", vec)
    x, w, bias, state = W.conv_inputs(2, L, D, 4, seed=L + D, with_state=True)
    out, st = ss.conv1d(to_dev(x), to_dev(w), to_dev(bias), state_in=to_dev(state), return_state=True)
    torch.cuda.synchronize()
    ref, st_ref = orc.conv1d(x, w, bias, state_in=state)
    assert scaled_err(to_np(out), ref) <= TOL[W.F32]
    assert np.array_equal(to_np(st).astype(np.float32), st_ref)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("K,Bsz,L,D", [(4, 2, 3000, 1032), (8, 1, 17761, 72), (2, 3, 997, 516)])
def test_conv1d_segments_longer_than_the_ring(orc, dtype, K, Bsz, L, D):
    """Sizes at which the streaming kernel's segments (sized for three CTAs
    per SM) run past its 16-slot ring, so slots are refilled in flight, with
    a ragged last segment and a ragged last group of channels."""
    x, w, bias, state = W.conv_inputs(Bsz, L, D, K, seed=L + K, dtype=dtype, with_state=True)
    out, st = ss.conv1d(to_dev(x, dtype), to_dev(w), to_dev(bias), state_in=to_dev(state), return_state=True)
    torch.cuda.synchronize()
    ref, st_ref = orc.conv1d(f32(x, dtype), w, bias, state_in=state)
    assert scaled_err(to_np(out), ref) <= TOL[dtype]
    assert np.array_equal(to_np(st).astype(np.float32), st_ref)


def test_conv1d_workload_full_size(orc):
    """The benchmark's conv1d workload (Bsz=2 L=2048 D=1536 K=4, fp32, SiLU,
    carried state), every output and the handed-over state."""
    w = W.WORKLOADS[8]
    x, wt, bias, state = W.conv_inputs(w.Bsz, w.L, w.D, w.conv_K, seed=w.seed, with_state=True)
    out, st = ss.conv1d(to_dev(x), to_dev(wt), to_dev(bias), state_in=to_dev(state), return_state=True)
    torch.cuda.synchronize()
    ref, st_ref = orc.conv1d(x, wt, bias, state_in=state)
    assert scaled_err(to_np(out), ref) <= TOL[W.F32]
    assert np.array_equal(to_np(st).astype(np.float32), st_ref)


def test_conv1d_without_silu_or_bias(orc):
    x, w, _, _ = W.conv_inputs(2, 100, 64, 4, seed=5)
    out = ss.conv1d(to_dev(x), to_dev(w), None, silu=False)
    torch.cuda.synchronize()
    ref, _ = orc.conv1d(x, w, None, silu=False)
    assert scaled_err(to_np(out), ref) <= TOL[W.F32]


def test_conv1d_pieces_and_decode_steps_equal_one_pass():
    """Two pieces chained through the state, and then token-by-token decode
    steps, give the one-pass outputs."""
    Bsz, L, D, K = 2, 150, 96, 4
    x, w, bias, _ = W.conv_inputs(Bsz, L + 10, D, K, seed=9)
    xd, wd, bd = to_dev(x), to_dev(w), to_dev(bias)
    full, st_full = ss.conv1d(xd[:, :L].contiguous(), wd, bd, return_state=True)
    a, sa = ss.conv1d(xd[:, :77].contiguous(), wd, bd, return_state=True)
    b_, sb = ss.conv1d(xd[:, 77:L].contiguous(), wd, bd, state_in=sa, return_state=True)
    torch.cuda.synchronize()
    assert scaled_err(to_np(torch.cat([a, b_], 1)), to_np(full)) < 1e-6
    assert torch.equal(sb, st_full)
    ref, _ = ss.conv1d(xd, wd, bd, return_state=True)
    st = st_full.clone()
    for t in range(L, L + 10):
        o = ss.conv1d_step(st, xd[:, t].contiguous(), wd, bd)
        assert scaled_err(to_np(o), to_np(ref[:, t])) < 1e-6


@pytest.mark.parametrize("K", [1, 4, 8])
def test_conv1d_step_matches_oracle(orc, K):
    Bsz, D = 5, 77
    x, w, bias, state = W.conv_inputs(Bsz, 1, D, K, seed=K + 30, with_state=True)
    st = to_dev(state) if K > 1 else torch.empty((Bsz, D, 0), device="cuda")
    out = ss.conv1d_step(st, to_dev(x[:, 0]), to_dev(w), to_dev(bias))
    torch.cuda.synchronize()
    ref, st_ref = orc.conv1d(x, w, bias, state_in=state)
    assert scaled_err(to_np(out), ref[:, 0]) <= TOL[W.F32]
    assert np.array_equal(to_np(st).astype(np.float32), st_ref)


def test_conv1d_rejects_in_place_and_bad_K():
    x = torch.randn(1, 10, 16, device="cuda")
    w = torch.randn(16, 4, device="cuda")
    with pytest.raises(ss.SelscanError) as e:
        ss.conv1d(x, w, out=x)
    assert e.value.code == ss.ERR_INVALID_ARG
    with pytest.raises(ss.SelscanError) as e:
        ss.conv1d(x, torch.randn(16, 9, device="cuda"))
    assert e.value.code == ss.ERR_UNSUPPORTED


def test_back_to_back_calls_see_each_others_outputs(orc):
    """The streaming kernel starts early and waits for the kernel before it:
    a second convolution over the first one's output, launched right after
    it, reads the finished output."""
    Bsz, L, D, K = 2, 3000, 1032, 4
    x, w, bias, _ = W.conv_inputs(Bsz, L, D, K, seed=81)
    o1 = ss.conv1d(to_dev(x), to_dev(w), to_dev(bias))
    o2 = ss.conv1d(o1, to_dev(w), to_dev(bias))
    torch.cuda.synchronize()
    r1, _ = orc.conv1d(x, w, bias)
    r2, _ = orc.conv1d(to_np(o1).astype(np.float32), w, bias)
    assert scaled_err(to_np(o1), r1) <= TOL[W.F32]
    assert scaled_err(to_np(o2), r2) <= TOL[W.F32]
