"""Shared helpers for the parity tests: host<->device conversion and the
error metric max |got - ref| / (1 + |ref|)."""
import numpy as np
import torch

from selective_state_space_157_b300 import workloads as W

TOL = {W.F32: 1e-4, W.BF16: 2e-2}


def to_dev(a: np.ndarray, dtype: str = W.F32, device="cuda"):
    """numpy fp32 array, or uint16 bf16 bit patterns, to a CUDA tensor."""
    if a is None:
        return None
    if dtype == W.BF16 and a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def to_np(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def scaled_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref))))


def fwd_dev(inp: W.FwdInputs, device="cuda"):
    """The device tensors of a forward call (x, delta, A, B, C, h0)."""
    dt = inp.dtype
    return (to_dev(inp.x, dt, device), to_dev(inp.delta, dt, device), to_dev(inp.A, W.F32, device),
            to_dev(inp.B, dt, device), to_dev(inp.C, dt, device),
            None if inp.h0 is None else to_dev(inp.h0, W.F32, device))


def oracle_fwd(orc, inp: W.FwdInputs, h0=None, nthreads=0):
    h = inp.h0 if h0 is None else h0
    return orc.selscan_fwd(inp.f32("x"), inp.f32("delta"), inp.A, inp.f32("B"), inp.f32("C"),
                           inp.delta_softplus, None if h is None else np.asarray(h, np.float64),
                           nthreads=nthreads)
