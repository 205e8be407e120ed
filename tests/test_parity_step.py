"""selscan_step (through the C ABI) against the fp64 oracle's decode step."""
import numpy as np
import pytest
import torch

import selective_state_space_157_b300 as ss
from selective_state_space_157_b300 import workloads as W
from tests.helpers import TOL, scaled_err, to_dev, to_np

pytestmark = pytest.mark.gpu


def rand_step(Bsz, D, N, seed):
    g = np.random.default_rng(seed)
    st = g.standard_normal((Bsz, D, N)).astype(np.float32)
    x = g.standard_normal((Bsz, D)).astype(np.float32)
    u = g.standard_normal((Bsz, D)) - 3.0
    dl = (np.maximum(u, 0) + np.log1p(np.exp(-np.abs(u)))).astype(np.float32)
    A = (-(0.5 + g.random((D, N)) * 8)).astype(np.float32)
    B = g.standard_normal((Bsz, N)).astype(np.float32)
    C = g.standard_normal((Bsz, N)).astype(np.float32)
    return st, x, dl, A, B, C


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 12, 16, 17, 20, 32, 48, 64])
def test_step_shapes(orc, N):
    Bsz, D = 3, 37
    st, x, dl, A, B, C = rand_step(Bsz, D, N, seed=N)
    s_dev = to_dev(st)
    y = ss.selscan_step(s_dev, to_dev(x), to_dev(dl), to_dev(A), to_dev(B), to_dev(C))
    torch.cuda.synchronize()
    s_ref = st.astype(np.float64)
    y_ref = orc.selscan_step(s_ref, x, dl, A, B, C)
    assert scaled_err(to_np(y), y_ref) <= TOL[W.F32]
    assert scaled_err(to_np(s_dev), s_ref) <= TOL[W.F32]


def test_steps_equal_forward_on_gpu(orc):
    """L decode steps reproduce one forward pass over L (delta post-softplus)."""
    Bsz, L, D, N = 2, 40, 64, 16
    inp = W.fwd_inputs(Bsz, L, D, N, seed=3, with_h0=True)
    g = lambda a: to_dev(a)
    dl = (np.maximum(inp.delta, 0) + np.log1p(np.exp(-np.abs(inp.delta.astype(np.float64))))).astype(np.float32)
    y_f, h_f = ss.selscan_fwd(g(inp.x), g(dl), g(inp.A), g(inp.B), g(inp.C), False, g(inp.h0),
                              return_final_state=True)
    s = g(inp.h0)
    ys = []
    for t in range(L):
        ys.append(ss.selscan_step(s, g(inp.x[:, t]), g(dl[:, t]), g(inp.A), g(inp.B[:, t]), g(inp.C[:, t])))
    torch.cuda.synchronize()
    y_s = torch.stack(ys, dim=1)
    assert scaled_err(to_np(y_s), to_np(y_f)) < 1e-5
    assert scaled_err(to_np(s), to_np(h_f)) < 1e-5
    y_r, h_r = orc.selscan_fwd(inp.x, dl, inp.A, inp.B, inp.C, False, inp.h0.astype(np.float64))
    assert scaled_err(to_np(y_s), y_r) <= TOL[W.F32]


def test_decode_workload_all_chains(orc):
    """Bsz=256, D=2560, N=16, 1024 consecutive steps on the full state in place:
    every step's output of all 655,360 chains, and the whole final state,
    against the oracle run step by step in fp64 (the chains split over host
    threads)."""
    from concurrent.futures import ThreadPoolExecutor
    w = W.WORKLOADS[5]
    st0 = W.decode_state(w)
    A = W.decode_A(w)
    s_dev = to_dev(st0)
    A_dev = to_dev(A)
    nchains = w.Bsz * w.D
    parts = np.array_split(np.arange(nchains, dtype=np.int64), 16)
    s_ref = [st0.reshape(-1, w.N)[p].astype(np.float64) for p in parts]
    worst = 0.0
    with ThreadPoolExecutor(len(parts)) as pool:
        for k in range(w.steps):
            x, dl, B, C = W.decode_step_inputs(w, k)
            y = ss.selscan_step(s_dev, to_dev(x), to_dev(dl), A_dev, to_dev(B), to_dev(C))
            y_ref = np.concatenate(list(pool.map(
                lambda i: orc.selscan_step(s_ref[i], x, dl, A, B, C, chains=parts[i]), range(len(parts)))))
            worst = max(worst, scaled_err(to_np(y).reshape(-1), y_ref))
    torch.cuda.synchronize()
    assert worst <= TOL[W.F32], worst
    assert scaled_err(to_np(s_dev).reshape(-1, w.N), np.concatenate(s_ref)) <= TOL[W.F32]
    assert torch.isfinite(s_dev).all()


def test_step_rejects_overlap():
    s = torch.randn(2, 4, 16, device="cuda")
    x = torch.randn(2, 4, device="cuda")
    A = -torch.ones(4, 16, device="cuda")
    B = torch.randn(2, 16, device="cuda")
    with pytest.raises(ss.SelscanError) as e:
        ss.selscan_step(s, x, x, A, B, B, y=x)
    assert e.value.code == ss.ERR_INVALID_ARG


@pytest.mark.parametrize("V", [1, 2, 4])
@pytest.mark.parametrize("N", [4, 8, 16, 32, 64])
def test_step_lane_widths(orc, monkeypatch, V, N):
    """Every states-per-lane choice of the vectorised step (4, 8 or 16 states
    per lane, narrowed where N is too small) gives the oracle's result."""
    monkeypatch.setenv("SELSCAN_STEP_V", str(V))
    Bsz, D = 5, 29
    st, x, dl, A, B, C = rand_step(Bsz, D, N, seed=100 + N + V)
    s_dev = to_dev(st)
    y = ss.selscan_step(s_dev, to_dev(x), to_dev(dl), to_dev(A), to_dev(B), to_dev(C))
    torch.cuda.synchronize()
    s_ref = st.astype(np.float64)
    y_ref = orc.selscan_step(s_ref, x, dl, A, B, C)
    assert scaled_err(to_np(y), y_ref) <= TOL[W.F32]
    assert scaled_err(to_np(s_dev), s_ref) <= TOL[W.F32]


def test_step_unaligned_state(orc):
    """A state that starts 4 bytes past a 16-byte boundary takes the one-thread-
    per-chain kernel and gives the same result."""
    Bsz, D, N = 2, 33, 16
    st, x, dl, A, B, C = rand_step(Bsz, D, N, seed=7)
    buf = torch.empty(Bsz * D * N + 1, device="cuda")
    s_dev = buf[1:].view(Bsz, D, N)
    s_dev.copy_(torch.from_numpy(st))
    y = ss.selscan_step(s_dev, to_dev(x), to_dev(dl), to_dev(A), to_dev(B), to_dev(C))
    torch.cuda.synchronize()
    s_ref = st.astype(np.float64)
    y_ref = orc.selscan_step(s_ref, x, dl, A, B, C)
    assert scaled_err(to_np(y), y_ref) <= TOL[W.F32]
    assert scaled_err(to_np(s_dev), s_ref) <= TOL[W.F32]
