"""The seeded input generator: determinism, shapes, distributions, bf16 encoding."""
import numpy as np
import torch

from selective_state_space_157_b300 import workloads as W


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(0)
    a = np.concatenate([g.standard_normal(100000).astype(np.float32) * 100,
                        # exact ties between two bf16 neighbours (round half to even)
                        (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
                        np.array([0.0, -0.0, 1e-40, -3.4e38, 3.3895e38], np.float32)])
    ours = W.to_bf16_bits(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = W.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(a).to(torch.bfloat16).float().numpy())


def test_deterministic_and_independent_streams():
    a = W.fwd_inputs(2, 33, 5, 4, seed=7)
    b = W.fwd_inputs(2, 33, 5, 4, seed=7)
    for k in ("x", "delta", "A", "B", "C"):
        assert np.array_equal(getattr(a, k), getattr(b, k))
    c = W.fwd_inputs(2, 33, 5, 4, seed=8)
    assert not np.array_equal(a.x, c.x)
    assert not np.array_equal(a.B, a.C)


def test_workload_shapes_and_distributions():
    w2 = W.WORKLOADS[2]
    i = W.workload_inputs(2)
    assert i.x.shape == (2, 2048, 1536) and i.B.shape == (2, 2048, 16) and i.A.shape == (1536, 16)
    assert i.x.dtype == np.float32 and i.delta_softplus
    assert abs(i.x.mean()) < 0.01 and abs(i.x.std() - 1) < 0.01
    assert abs(i.delta.mean() - w2.u_mean) < 0.01 and abs(i.delta.std() - 1) < 0.01
    assert np.array_equal(i.A[5], -np.arange(1, 17, dtype=np.float32))
    i1 = W.workload_inputs(1)
    assert i1.x.shape == (1, 64, 16) and i1.A.shape == (16, 4) and i1.h0 is None


def test_bf16_workload_A_range():
    A = W.make_A("loguniform", 64, 16, 103)
    assert A.dtype == np.float32 and np.all(A <= -1.0) and np.all(A >= -16.0)
    small = W.fwd_inputs(1, 8, 16, 16, seed=3, dtype=W.BF16)
    assert small.x.dtype == np.uint16 and small.f32("x").dtype == np.float32


def test_decode_inputs():
    w = W.WORKLOADS[5]
    x, dl, B, C = W.decode_step_inputs(w, 3)
    assert x.shape == (256, 2560) and dl.shape == (256, 2560) and B.shape == (256, 16)
    assert np.all(dl > 0)
    x2, _, _, _ = W.decode_step_inputs(w, 4)
    assert not np.array_equal(x, x2)


def test_backward_gradients_and_ssd_inputs():
    dy, dhT = W.bwd_grads(2, 50, 8, 4, seed=5)
    dy2, _ = W.bwd_grads(2, 50, 8, 4, seed=5, with_dhT=False)
    assert dy.shape == (2, 50, 8) and dhT.shape == (2, 8, 4) and np.array_equal(dy, dy2)
    assert dy.dtype == np.float32 and not np.array_equal(dy[0, :4, :4], dhT[0])
    w9 = W.WORKLOADS[9]
    assert w9.backward and (w9.Bsz, w9.L, w9.D, w9.N) == (2, 2048, 1536, 16)
    x, dt, A, B, C, h0 = W.ssd_inputs(1, 64, 8, 16, 32, seed=6, with_h0=True)
    assert x.shape == (1, 64, 8, 16) and dt.shape == (1, 64, 8) and A.shape == (8,)
    assert B.shape == C.shape == (1, 64, 32) and h0.shape == (1, 8, 32, 16)
    assert np.all(A <= -1.0) and np.all(A >= -16.0) and not np.array_equal(B, C)
    x2, *_ = W.ssd_inputs(1, 64, 8, 16, 32, seed=6)
    assert np.array_equal(x, x2)
