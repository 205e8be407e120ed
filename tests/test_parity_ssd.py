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
                                   (1, 129, 2, 128, 128), (3, 64, 1, 32, 128), (1, 63, 4, 64, 64)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_shapes(orc, shape, dtype):
    Bsz, L, H, P, N = shape
    run_case(orc, Bsz, L, H, P, N, dtype, seed=sum(shape) + (dtype == W.BF16), h0=(L % 2 == 1))


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
