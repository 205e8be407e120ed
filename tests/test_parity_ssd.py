"""selscan_ssd_fwd (Mamba-2 SSD on the tensor cores, through the C ABI)
against the fp64 oracle's recurrence (oracle_ssd_fwd).

The products run on tcgen05 with fp16 operands and fp32 accumulators, so
every output is held to the bf16 bar, max |got - ref| / (1 + |ref|) <= 2e-2,
for either input dtype; the oracle reads exactly the values the GPU reads
(bf16-rounded inputs for bf16 I/O). The final state hT is checked the same
way. Shapes cover the pages' layer (section 5.2: 64 heads of headdim 64,
state size 128), both state sizes and every headdim the kernels take,
partial last chunks, one-step sequences, h0 and softplus on and off.
"""
import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import scaled_err, to_np

pytestmark = pytest.mark.gpu
TOL = 2e-2


def run_case(orc, Bsz, L, H, P, N, dtype, seed, h0=False, softplus=True):
    x, dt, A, B, C, hh = W.ssd_inputs(Bsz, L, H, P, N, seed=seed, with_h0=h0)
    if not softplus:   # the step is used as given: hand in a positive one
        dt = np.log1p(np.exp(dt.astype(np.float64))).astype(np.float32)
    if dtype == W.BF16:
        x, B, C = (W.bf16_bits_to_f32(W.to_bf16_bits(a)) for a in (x, B, C))
        tdt = torch.bfloat16
    else:
        tdt = torch.float32
    dev = lambda a, t=torch.float32: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().to(t)
    y, hT = ss.ssd_fwd(dev(x, tdt), dev(dt), dev(A), dev(B, tdt), dev(C, tdt), softplus,
                       h0=None if hh is None else dev(hh), return_final_state=True)
    torch.cuda.synchronize()
    ss.check_device_error()
    yr, hr = orc.ssd_fwd(x, dt, A, B, C, softplus, h0=None if hh is None else hh.astype(np.float64))
    ey, eh = scaled_err(to_np(y), yr), scaled_err(to_np(hT), hr)
    assert ey <= TOL, f"y error {ey:.3e}"
    assert eh <= TOL, f"hT error {eh:.3e}"
    return ey, eh


@pytest.mark.parametrize("h0", [False, True])
def test_pages_layer_bf16(orc, h0):
    """Batch 1, 1024 steps, 64 heads of headdim 64, state 128, bf16 I/O."""
    run_case(orc, 1, 1024, 64, 64, 128, W.BF16, seed=90 + h0, h0=h0)


@pytest.mark.parametrize("shape", [(2, 100, 3, 64, 128), (1, 1, 2, 64, 64), (2, 200, 2, 32, 64),
                                   (1, 129, 2, 128, 128), (3, 64, 1, 32, 128), (1, 63, 4, 64, 64),
                                   (1, 70, 5, 128, 64), (2, 65, 6, 32, 128), (1, 130, 9, 64, 128)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_shapes(orc, shape, dtype):
    """Every state size and headdim, partial last chunks, and head counts
    that leave the last group of heads (the state kernel takes several per
    CTA) partly empty."""
    Bsz, L, H, P, N = shape
    run_case(orc, Bsz, L, H, P, N, dtype, seed=sum(shape) + (dtype == W.BF16), h0=(L % 2 == 1))


@pytest.mark.parametrize("shape", [(1, 600, 3, 64, 128), (2, 2100, 2, 32, 64), (1, 8192, 2, 32, 64),
                                   (1, 8250, 1, 32, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_long_sequences(orc, shape):
    """Sequences of 10, 33, 128 and 129 chunks: the carry kernel folds each
    row's chunk states in batches of eight, so these take two to seventeen
    batches with ragged last ones; with h0, so the carries start from it."""
    run_case(orc, *shape, W.BF16, seed=sum(shape), h0=True)


def test_softplus_off(orc):
    run_case(orc, 1, 300, 2, 64, 128, W.F32, seed=95, h0=True, softplus=False)


def test_empty_sequence_copies_state():
    h0 = torch.randn(1, 2, 64, 32, device="cuda")
    x = torch.empty(1, 0, 2, 32, device="cuda")
    e = torch.empty(1, 0, 64, device="cuda")
    y, hT = ss.ssd_fwd(x, torch.empty(1, 0, 2, device="cuda"), -torch.ones(2, device="cuda"), e, e, True,
                       h0=h0, return_final_state=True)
    torch.cuda.synchronize()
    assert y.shape == (1, 0, 2, 32) and torch.equal(hT, h0)


def test_unsupported_sizes_are_refused():
    x = torch.zeros(1, 4, 1, 48, device="cuda")
    with pytest.raises(ss.SelscanError) as e:
        ss.ssd_fwd(x, torch.zeros(1, 4, 1, device="cuda"), -torch.ones(1, device="cuda"),
                   torch.zeros(1, 4, 64, device="cuda"), torch.zeros(1, 4, 64, device="cuda"))
    assert e.value.code == ss.ERR_UNSUPPORTED


# ---------------------------------------------------------------- limiting cases
# The limits of booiljung.github.io "3.1 LTI systems and input-dependent
# parameters", section 0.4.2, for the scalar decay of each head: a step of 0
# keeps the state (exp(0 A) = 1, no input), a large step resets it to the
# current input term, and A = 0 turns the state into a running sum. Where the
# sums cancel, the error is measured against the magnitude of what was
# summed (the oracle on |x|, |B|, |C|, |h0|), the forward-error bound of a
# floating-point sum, as for the selective scan's limits.

def _run_edge(orc, dt, A, seed, softplus, cancelling, Bsz=1, L=200, H=3, P=64, N=128):
    x, _, _, B, C, hh = W.ssd_inputs(Bsz, L, H, P, N, seed=seed, with_h0=True)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    y, hT = ss.ssd_fwd(dev(x), dev(dt), dev(A), dev(B), dev(C), softplus, h0=dev(hh), return_final_state=True,
                       check=True)
    yr, hr = orc.ssd_fwd(x, dt, A, B, C, softplus, h0=hh.astype(np.float64))
    if cancelling:
        ym, hm = orc.ssd_fwd(np.abs(x), dt, A, np.abs(B), np.abs(C), softplus, h0=np.abs(hh).astype(np.float64))
        ey = float(np.max(np.abs(to_np(y) - yr) / (1.0 + np.abs(ym))))
        eh = float(np.max(np.abs(to_np(hT) - hr) / (1.0 + np.abs(hm))))
    else:
        ey, eh = scaled_err(to_np(y), yr), scaled_err(to_np(hT), hr)
    assert ey <= TOL, f"y error {ey:.3e}"
    assert eh <= TOL, f"hT error {eh:.3e}"
    return hh, hT


def test_zero_step_keeps_the_state(orc):
    """dt = 0 with softplus off: no decay and no input, so hT equals h0 bit for
    bit and y is C h0 at every step."""
    H = 3
    A = -np.array([1.0, 4.0, 16.0], np.float32)
    hh, hT = _run_edge(orc, np.zeros((1, 200, H), np.float32), A, seed=101, softplus=False, cancelling=False)
    assert torch.equal(hT.cpu(), torch.from_numpy(hh)), "dt = 0 must leave the state exactly as it was"


def test_softplus_tails(orc):
    """Step pre-activations far in either tail: softplus gives steps of e^-80
    (the state is kept) and of 80 (the state resets to the current input).
    Steps of 80 make terms of thousands in the masked product that cancel to a
    much smaller y, so the bound is the magnitude one (a numpy emulation of
    the chunked form with fp16 operands gives the same 9.5e-2 plain error the
    kernel does, and 4e-12 in fp64)."""
    g = np.random.default_rng(102)
    dt = g.choice(np.array([-80.0, -20.0, -5.0, 0.0, 5.0, 20.0, 80.0], np.float32), size=(1, 200, 3))
    _run_edge(orc, dt.astype(np.float32), -np.array([1.0, 4.0, 16.0], np.float32), seed=102, softplus=True,
              cancelling=True)


def test_zero_decay_heads_and_mixed_steps(orc):
    """A = 0 on some heads (running sums over 512 steps) and steps mixed from
    0 to 20 with softplus off."""
    g = np.random.default_rng(103)
    dt = g.choice(np.array([0.0, 1e-3, 0.05, 1.0, 20.0], np.float32), size=(1, 512, 3))
    _run_edge(orc, dt.astype(np.float32), np.array([0.0, -2.0, 0.0], np.float32), seed=103, softplus=False,
              cancelling=True, L=512)


def test_back_to_back_calls_see_each_others_outputs(orc):
    """Two calls on one stream, the second reading the first's y as its x
    (its kernels start early and wait for the kernel before them)."""
    Bsz, L, H, P, N = 1, 200, 3, 64, 128
    x, dt, A, B, C, _ = W.ssd_inputs(Bsz, L, H, P, N, seed=61)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    y1 = ss.ssd_fwd(dev(x), dev(dt), dev(A), dev(B), dev(C), True)
    y2 = ss.ssd_fwd(y1, dev(dt), dev(A), dev(B), dev(C), True)
    torch.cuda.synchronize()
    ss.check_device_error()
    r2, _ = orc.ssd_fwd(to_np(y1).astype(np.float32), dt, A, B, C, True)
    assert scaled_err(to_np(y2), r2) <= TOL
