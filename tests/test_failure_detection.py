"""Failure detection on the GPU without a fault: every wait inside the
kernels is bounded. Here the chunked forward path never announces its
composed chunk carries (a flag that nothing sets; selscan_test_fault_injection),
so the correction passes of later chunks run their wait to a short limit; the kernel
must end, the host must read SELSCAN_ERR_TIMEOUT with fault code 2 on the
stream the kernel ran on (and on no other), and the context must stay usable
for a correct call right after."""
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import TOL, fwd_dev, oracle_fwd, scaled_err, to_np

pytestmark = pytest.mark.gpu


def test_withheld_carries_end_in_timeout_status(orc, monkeypatch):
    inp = W.fwd_inputs(2, 512, 256, 16, seed=21, with_h0=True)
    x, dl, A, B, C, h0 = fwd_dev(inp)
    monkeypatch.setenv("SELSCAN_CHUNK", "64")            # 8 chunks: corrections of chunks 1..7 wait
    assert ss.fwd_plan(2, 512, 256, 16)["chunks"] == 8
    other = torch.cuda.Stream()
    ss.check_device_error(other)
    assert ss.lib().selscan_test_fault_injection(1, 20) == ss.OK
    try:
        ss.selscan_fwd(x, dl, A, B, C, True, h0, return_final_state=True)
        torch.cuda.synchronize()
    finally:
        assert ss.lib().selscan_test_fault_injection(0, 0) == ss.OK
    ss.check_device_error(other)                          # another stream sees no fault
    with pytest.raises(ss.SelscanError) as e:
        ss.check_device_error()
    assert e.value.code == ss.ERR_TIMEOUT
    assert "fault code 2" in str(e.value)
    ss.check_device_error()                               # the word was cleared

    # The same process and context compute correctly right after.
    y, hT = ss.selscan_fwd(x, dl, A, B, C, True, h0, return_final_state=True)
    torch.cuda.synchronize()
    ss.check_device_error()
    yr, hr = oracle_fwd(orc, inp)
    assert scaled_err(to_np(y), yr) <= TOL[W.F32]
    assert scaled_err(to_np(hT), hr) <= TOL[W.F32]


def test_timeout_hook_is_inert_on_one_chunk(orc, monkeypatch):
    """With a single chunk nothing waits on a flag: the hook changes nothing."""
    monkeypatch.setenv("SELSCAN_CHUNK", "0")
    inp = W.fwd_inputs(1, 300, 128, 16, seed=22)
    x, dl, A, B, C, _ = fwd_dev(inp)
    assert ss.lib().selscan_test_fault_injection(1, 20) == ss.OK
    try:
        y = ss.selscan_fwd(x, dl, A, B, C, True)
        torch.cuda.synchronize()
    finally:
        assert ss.lib().selscan_test_fault_injection(0, 0) == ss.OK
    ss.check_device_error()
    yr, _ = oracle_fwd(orc, inp)
    assert scaled_err(to_np(y), yr) <= TOL[W.F32]
