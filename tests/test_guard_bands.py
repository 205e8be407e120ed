"""Out-of-bounds writes: every output is placed inside a larger buffer whose
margins hold a canary pattern; after the call the margins must be unchanged
bit for bit and the outputs must match the oracle. Shapes cover ragged
channel tiles, ragged time tiles, chunked and one-pass plans, both dtypes,
the TMA path (rows a multiple of 16 bytes) and the plain-load path."""
import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import TOL, fwd_dev, oracle_fwd, scaled_err, to_dev, to_np

pytestmark = pytest.mark.gpu

MARGIN = 4096          # elements on each side
CANARY_F32 = -7.0e33


def guarded(shape, dtype):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * MARGIN,), CANARY_F32, dtype=dtype, device="cuda")
    return buf, buf[MARGIN:MARGIN + n].view(*shape)


def margins_intact(buf):
    ref = torch.full((MARGIN,), CANARY_F32, dtype=buf.dtype, device=buf.device)
    return torch.equal(buf[:MARGIN], ref) and torch.equal(buf[-MARGIN:], ref)


@pytest.mark.parametrize("D", [130, 136])
@pytest.mark.parametrize("chunk", [0, 100])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_forward_writes_stay_inside(orc, monkeypatch, D, chunk, dtype):
    monkeypatch.setenv("SELSCAN_CHUNK", str(chunk))
    Bsz, L, N = 3, 333, 16
    inp = W.fwd_inputs(Bsz, L, D, N, seed=D + chunk, dtype=dtype, with_h0=True)
    x, dl, A, B, C, h0 = fwd_dev(inp)
    ybuf, y = guarded((Bsz, L, D), x.dtype)
    hbuf, hT = guarded((Bsz, D, N), torch.float32)
    ss.selscan_fwd(x, dl, A, B, C, True, h0, y=y, hT=hT)
    torch.cuda.synchronize()
    ss.check_device_error()
    assert margins_intact(ybuf) and margins_intact(hbuf)
    yr, hr = oracle_fwd(orc, inp)
    assert scaled_err(to_np(y), yr) <= TOL[dtype]
    assert scaled_err(to_np(hT), hr) <= TOL[W.F32] * (20 if dtype == W.BF16 else 1)


@pytest.mark.parametrize("N", [3, 16, 64])
def test_step_writes_stay_inside(orc, N):
    Bsz, D = 5, 77
    g = np.random.default_rng(N)
    st = g.standard_normal((Bsz, D, N)).astype(np.float32)
    x = g.standard_normal((Bsz, D)).astype(np.float32)
    dl = (g.random((Bsz, D)) * 0.2).astype(np.float32)
    A = (-(0.5 + g.random((D, N)) * 4)).astype(np.float32)
    B = g.standard_normal((Bsz, N)).astype(np.float32)
    C = g.standard_normal((Bsz, N)).astype(np.float32)
    sbuf, s_dev = guarded((Bsz, D, N), torch.float32)
    s_dev.copy_(torch.from_numpy(st))
    ybuf, y = guarded((Bsz, D), torch.float32)
    ss.selscan_step(s_dev, to_dev(x), to_dev(dl), to_dev(A), to_dev(B), to_dev(C), y=y)
    torch.cuda.synchronize()
    assert margins_intact(sbuf) and margins_intact(ybuf)
    s_ref = st.astype(np.float64)
    y_ref = orc.selscan_step(s_ref, x, dl, A, B, C)
    assert scaled_err(to_np(y), y_ref) <= TOL[W.F32]
    assert scaled_err(to_np(s_dev), s_ref) <= TOL[W.F32]
