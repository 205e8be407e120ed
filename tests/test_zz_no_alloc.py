"""selscan_fwd_noalloc: the forward scan for callers that cannot allocate
device memory (another allocator owns it all, or they may not pay for an
allocation). It must give the results of selscan_fwd while using only the
library's fixed scratch array, and refuse problems that need more scratch
than that array holds, before launching anything.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import TOL, fwd_dev, scaled_err, to_np

pytestmark = pytest.mark.gpu


def c_abi_noalloc(x, dl, A, B, C, y, h0, hT, bf16=False):
    """Calls the entry point through the C ABI directly."""
    Bsz, L, D = x.shape
    N = A.shape[1]
    p = lambda t: None if t is None else t.data_ptr()
    return ss.lib().selscan_fwd_noalloc(p(x), p(dl), p(A), p(B), p(C), p(y), Bsz, L, D, N,
                                        1 if bf16 else 0, 1, p(h0), p(hT),
                                        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_matches_selscan_fwd_on_two_calls_in_a_row(dtype):
    Bsz, L, D, N = 2, 1500, 192, 16
    plan = ss.fwd_plan(Bsz, L, D, N, bf16=dtype == W.BF16)
    assert plan["chunks"] > 1, "the problem must be chunked so that the scratch array is used"
    inp = W.fwd_inputs(Bsz, L, D, N, seed=11, dtype=dtype, with_h0=True)
    x, dl, A, B, C, h0 = fwd_dev(inp)
    y_ref, h_ref = ss.selscan_fwd(x, dl, A, B, C, True, h0, return_final_state=True)
    torch.cuda.synchronize()
    for _ in range(2):
        y = torch.full_like(y_ref, float("nan"))
        hT = torch.full_like(h_ref, float("nan"))
        assert c_abi_noalloc(x, dl, A, B, C, y, h0, hT, bf16=dtype == W.BF16) == ss.OK, ss.last_error()
        torch.cuda.synchronize()
        # The same plan and kernels as selscan_fwd, each chain's arithmetic in
        # the same order: the results are identical, not merely close.
        assert torch.equal(y, y_ref)
        assert torch.equal(hT, h_ref)
    ss.check_device_error()


def test_in_place_resume_stages_the_state_in_the_scratch(orc):
    """hT written over h0 on a chunked problem: the final state passes through
    the scratch array (no allocation) and matches the oracle."""
    Bsz, L, D, N = 2, 1500, 192, 16
    inp = W.fwd_inputs(Bsz, L, D, N, seed=13, with_h0=True)
    x, dl, A, B, C, h0 = fwd_dev(inp)
    y = torch.empty_like(x)
    for _ in range(2):
        h = h0.clone()
        assert c_abi_noalloc(x, dl, A, B, C, y, h, h) == ss.OK, ss.last_error()
        torch.cuda.synchronize()
        yr, hr = orc.selscan_fwd(inp.x, inp.delta, inp.A, inp.B, inp.C, True, inp.h0.astype(np.float64))
        assert scaled_err(to_np(y), yr) <= TOL[W.F32]
        assert scaled_err(to_np(h), hr) <= TOL[W.F32]
    ss.check_device_error()


def test_refuses_a_problem_beyond_the_scratch(monkeypatch):
    monkeypatch.setenv("SELSCAN_CHUNK", "16")        # many chunks: a large carry workspace
    Bsz, L, D, N = 1, 16384, 128, 16
    plan = ss.fwd_plan(Bsz, L, D, N)
    assert plan["workspace_bytes"] > ss.NOALLOC_SCRATCH_BYTES
    inp = W.fwd_inputs(Bsz, L, D, N, seed=2)
    x, dl, A, B, C, _ = fwd_dev(inp)
    y = torch.full_like(x, 7.0)
    rc = c_abi_noalloc(x, dl, A, B, C, y, None, None)
    assert rc == ss.ERR_UNSUPPORTED and "scratch" in ss.last_error()
    torch.cuda.synchronize()
    assert bool(torch.all(y == 7.0)), "nothing may be written when the call is refused"
