"""Pins on the fp64 oracle: each checks it against something other than itself.

The oracle restates the selective_scan loop of "Mamba: Selective State Space
Models" (youngju.dev, section 3.3). The pins below fix its result through
independent routes (brute-force unrolling, closed forms, special cases that
reduce to textbook formulas, invariants), so that a dropped term, a wrong sign
or index, or a transposed operand fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

from selective_state_space_157_b300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_inputs(Bsz, L, D, N, seed, softplus=True, h0=False, a_scale=1.0):
    g = np.random.default_rng(seed)
    x = g.standard_normal((Bsz, L, D)).astype(np.float32)
    u = (g.standard_normal((Bsz, L, D)) - 1.0).astype(np.float32)
    if not softplus:
        u = np.abs(u) * np.float32(0.3)
    # distinct, asymmetric A entries so a transposed A[n, d] would differ
    A = (-a_scale * (0.2 + g.random((D, N)))).astype(np.float32)
    B = g.standard_normal((Bsz, L, N)).astype(np.float32)
    C = g.standard_normal((Bsz, L, N)).astype(np.float32)
    hh = g.standard_normal((Bsz, D, N)) if h0 else None
    return x, u, A, B, C, hh


def sp(u):
    u = np.asarray(u, np.float64)
    return np.maximum(u, 0) + np.log1p(np.exp(-np.abs(u)))


def brute_force(x, delta, A, B, C, h0):
    """Unrolled form: y_t = sum_{s<=t} sum_n C_t[n] prod_{s<r<=t} exp(d_r A[n]) d_s B_s[n] x_s
    + sum_n C_t[n] prod_{r<=t} exp(d_r A[n]) h0[n]. Products taken literally."""
    x = x.astype(np.float64); delta = delta.astype(np.float64)
    A = A.astype(np.float64); B = B.astype(np.float64); C = C.astype(np.float64)
    Bsz, L, D = x.shape
    N = A.shape[1]
    y = np.zeros((Bsz, L, D))
    hT = np.zeros((Bsz, D, N))
    for b in range(Bsz):
        for d in range(D):
            E = np.exp(delta[b, :, d, None] * A[d][None, :])     # (L, N) per-step decay
            for t in range(L):
                tot = 0.0
                for s in range(t + 1):
                    decay = np.prod(E[s + 1:t + 1], axis=0)       # empty product = 1
                    tot += np.sum(C[b, t] * decay * delta[b, s, d] * B[b, s] * x[b, s, d])
                if h0 is not None:
                    tot += np.sum(C[b, t] * np.prod(E[:t + 1], axis=0) * h0[b, d])
                y[b, t, d] = tot
            st = np.zeros(N)
            for s in range(L):
                st += np.prod(E[s + 1:], axis=0) * delta[b, s, d] * B[b, s] * x[b, s, d]
            if h0 is not None:
                st += np.prod(E, axis=0) * h0[b, d]
            hT[b, d] = st
    return y, hT


def close(a, b, rtol, atol=0.0):
    np.testing.assert_allclose(a, b, rtol=rtol, atol=atol)


# ---------------------------------------------------------------- softplus

def test_softplus_values(orc):
    assert orc.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    for u in (-30.0, -5.0, -0.7, 0.3, 2.0, 19.0, 45.0):
        assert orc.softplus(u) - orc.softplus(-u) == pytest.approx(u, rel=1e-13, abs=1e-15)
        assert orc.softplus(u) == pytest.approx(math.log1p(math.exp(u)), rel=1e-14)
    assert orc.softplus(800.0) == 800.0                      # no overflow
    assert orc.softplus(-60.0) == pytest.approx(math.exp(-60.0), rel=1e-14)


# ---------------------------------------------------------------- golden

def test_hand_worked_cases(orc):
    g = json.load(open(os.path.join(HERE, "golden", "hand_worked.json")))
    for c in g["cases"]:
        arr = lambda k: np.array(c[k], np.float64)
        h0 = arr("h0") if "h0" in c else None
        y, hT = orc.selscan_fwd(arr("x"), arr("delta"), arr("A"), arr("B"), arr("C"),
                                delta_softplus=c["delta_softplus"], h0=h0)
        close(y, arr("y"), c["rtol"], c.get("atol", 0.0))
        close(hT, arr("hT"), c["rtol"], c.get("atol", 0.0))


# ---------------------------------------------------------------- P1 brute force

@pytest.mark.parametrize("Bsz,L,D,N,softplus,h0", [
    (1, 1, 1, 1, True, False),
    (2, 9, 3, 4, True, True),
    (1, 17, 2, 5, False, True),
    (2, 24, 3, 7, True, False),
])
def test_brute_force(orc, Bsz, L, D, N, softplus, h0):
    x, u, A, B, C, hh = rand_inputs(Bsz, L, D, N, seed=L * 7 + N, softplus=softplus, h0=h0)
    dl = sp(u) if softplus else u.astype(np.float64)
    yb, hb = brute_force(x, dl, A, B, C, hh)
    y, hT = orc.selscan_fwd(x, u, A, B, C, delta_softplus=softplus, h0=hh)
    scale = 1.0 + np.abs(yb)
    assert np.max(np.abs(y - yb) / scale) < 1e-12
    assert np.max(np.abs(hT - hb) / (1.0 + np.abs(hb))) < 1e-12


# ---------------------------------------------------------------- P2 A = 0

def test_A_zero_running_sum(orc):
    Bsz, L, D, N = 2, 40, 3, 6
    x, u, _, B, C, hh = rand_inputs(Bsz, L, D, N, seed=2, h0=True)
    A = np.zeros((D, N), np.float32)
    y, hT = orc.selscan_fwd(x, u, A, B, C, delta_softplus=True, h0=hh)
    dl = sp(u)
    # h_t = h0 + sum_{s<=t} delta_s B_s x_s
    contrib = dl[..., None] * B.astype(np.float64)[:, :, None, :] * x.astype(np.float64)[..., None]  # (Bsz,L,D,N)
    h = hh[:, None, :, :] + np.cumsum(contrib, axis=1)
    yr = np.einsum("bldn,bln->bld", h, C.astype(np.float64))
    close(y, yr, 1e-12, 1e-12)
    close(hT, h[:, -1], 1e-12, 1e-12)


# ---------------------------------------------------------------- P3 N = 1

def test_N1_scalar_recurrence(orc):
    """One state is the scalar recurrence h = a*h + b*x with a = exp(delta*A), b = delta*B."""
    Bsz, L, D = 2, 50, 4
    x, u, A, B, C, hh = rand_inputs(Bsz, L, D, 1, seed=3, h0=True)
    y, hT = orc.selscan_fwd(x, u, A, B, C, delta_softplus=True, h0=hh)
    for b in range(Bsz):
        for d in range(D):
            h = float(hh[b, d, 0])
            for t in range(L):
                dl = math.log1p(math.exp(float(u[b, t, d])))
                a = math.exp(dl * float(A[d, 0]))
                bb = dl * float(B[b, t, 0])
                h = a * h + bb * float(x[b, t, d])
                assert y[b, t, d] == pytest.approx(h * float(C[b, t, 0]), rel=1e-13, abs=1e-15)
            assert hT[b, d, 0] == pytest.approx(h, rel=1e-13, abs=1e-15)


# ---------------------------------------------------------------- P4 L = 1

def test_L1_closed_form(orc):
    Bsz, D, N = 3, 5, 8
    x, u, A, B, C, _ = rand_inputs(Bsz, 1, D, N, seed=4)
    y, hT = orc.selscan_fwd(x, u, A, B, C, delta_softplus=True)
    dl = sp(u)[:, 0, :]                                       # (Bsz, D)
    h = dl[..., None] * B[:, 0, None, :].astype(np.float64) * x[:, 0, :, None].astype(np.float64)
    close(hT, h, 1e-14)
    close(y[:, 0, :], np.einsum("bdn,bn->bd", h, C[:, 0].astype(np.float64)), 1e-13, 1e-15)


# ---------------------------------------------------------------- P5 LTI convolution

def test_lti_convolution_kernel(orc):
    """Delta, B, C constant over t: y = x * K with K_k = sum_n C[n] abar[n]^k delta B[n]
    (booiljung.github.io section 0.2.2, the convolution kernel of an LTI SSM)."""
    L, D, N = 64, 3, 5
    g = np.random.default_rng(5)
    x = g.standard_normal((1, L, D)).astype(np.float32)
    dl_d = (0.05 + g.random(D)).astype(np.float32)
    delta = np.broadcast_to(dl_d, (1, L, D)).copy()
    A = (-0.1 - g.random((D, N))).astype(np.float32)
    Bv = g.standard_normal(N).astype(np.float32)
    Cv = g.standard_normal(N).astype(np.float32)
    B = np.broadcast_to(Bv, (1, L, N)).copy()
    C = np.broadcast_to(Cv, (1, L, N)).copy()
    y, _ = orc.selscan_fwd(x, delta, A, B, C, delta_softplus=False)
    k = np.arange(L)
    for d in range(D):
        abar = np.exp(float(dl_d[d]) * A[d].astype(np.float64))          # (N,)
        K = np.sum(Cv.astype(np.float64)[None, :] * abar[None, :] ** k[:, None]
                   * float(dl_d[d]) * Bv.astype(np.float64)[None, :], axis=1)
        yc = np.convolve(x[0, :, d].astype(np.float64), K)[:L]
        close(y[0, :, d], yc, 1e-11, 1e-12)


# ---------------------------------------------------------------- P6 geometric

def test_geometric_closed_form(orc):
    L = 300
    xv, dv, Av, Bv = 0.7, 0.2, -0.3, 1.3
    x = np.full((1, L, 1), xv, np.float32)
    delta = np.full((1, L, 1), dv, np.float32)
    A = np.full((1, 1), Av, np.float32)
    B = np.full((1, L, 1), Bv, np.float32)
    C = np.ones((1, L, 1), np.float32)
    y, _ = orc.selscan_fwd(x, delta, A, B, C)
    a = math.exp(float(np.float32(dv)) * float(np.float32(Av)))
    b = float(np.float32(dv)) * float(np.float32(Bv)) * float(np.float32(xv))
    t = np.arange(L)
    close(y[0, :, 0], b * (1 - a ** (t + 1)) / (1 - a), 1e-12)


# ---------------------------------------------------------------- P7 delta -> 0

def test_delta_zero_persists_state(orc):
    Bsz, L, D, N = 2, 30, 3, 4
    x, _, A, B, C, hh = rand_inputs(Bsz, L, D, N, seed=7, h0=True)
    delta = np.zeros((Bsz, L, D), np.float32)
    y, hT = orc.selscan_fwd(x, delta, A, B, C, delta_softplus=False, h0=hh)
    assert np.array_equal(hT, hh)                                      # bit-exact
    yr = np.einsum("bdn,bln->bld", hh, C.astype(np.float64))
    close(y, yr, 1e-14, 1e-15)
    tiny = np.full((Bsz, L, D), 1e-12, np.float32)
    _, hT2 = orc.selscan_fwd(x, tiny, A, B, C, delta_softplus=False, h0=hh)
    assert np.max(np.abs(hT2 - hh)) < 1e-9


# ---------------------------------------------------------------- P8 delta -> inf

def test_large_delta_resets_state(orc):
    """A < 0 and a huge step: exp(delta*A) underflows to 0, so h_t = delta_t B_t x_t."""
    Bsz, L, D, N = 1, 12, 2, 3
    x, _, A, B, C, hh = rand_inputs(Bsz, L, D, N, seed=8, h0=True)
    delta = np.full((Bsz, L, D), 1e4, np.float32)
    y, hT = orc.selscan_fwd(x, delta, A, B, C, delta_softplus=False, h0=hh)
    h = 1e4 * B.astype(np.float64)[:, :, None, :] * x.astype(np.float64)[..., None]
    close(hT, h[:, -1], 1e-15)
    close(y, np.einsum("bldn,bln->bld", h, C.astype(np.float64)), 1e-14)


# ---------------------------------------------------------------- P9 chunked == sequential

@pytest.mark.parametrize("cuts", [(1,), (17,), (5, 40, 41), (10, 20, 30, 50, 63)])
def test_split_resume(orc, cuts):
    """Running [0, L1) then [L1, L) with the handed-over state equals one pass."""
    Bsz, L, D, N = 2, 64, 3, 5
    x, u, A, B, C, hh = rand_inputs(Bsz, L, D, N, seed=9, h0=True)
    y, hT = orc.selscan_fwd(x, u, A, B, C, delta_softplus=True, h0=hh)
    bounds = [0, *cuts, L]
    h = hh
    for a, b in zip(bounds[:-1], bounds[1:]):
        yi, h = orc.selscan_fwd(x[:, a:b], u[:, a:b], A, B[:, a:b], C[:, a:b], delta_softplus=True, h0=h)
        close(yi, y[:, a:b], 1e-13, 1e-14)
    close(h, hT, 1e-13, 1e-14)


def test_associative_chunk_composition(orc):
    """Parallel-scan form (booiljung.github.io section 3.1.5.2): each chunk reduced from a
    zero state to (prod abar, h_end) and composed with (a1,b1) o (a2,b2) = (a2 a1, a2 b1 + b2)
    gives the sequential state; the in-chunk outputs follow from a correction by the carry."""
    Bsz, L, D, N = 1, 96, 2, 4
    x, u, A, B, C, hh = rand_inputs(Bsz, L, D, N, seed=10, h0=True)
    y, hT = orc.selscan_fwd(x, u, A, B, C, delta_softplus=True, h0=hh)
    dl = sp(u)
    chunks = [(0, 30), (30, 31), (31, 80), (80, 96)]
    aggs = []
    for a, b in chunks:
        ylocal, hend = orc.selscan_fwd(x[:, a:b], u[:, a:b], A, B[:, a:b], C[:, a:b], delta_softplus=True)
        P = np.exp(A.astype(np.float64)[None] * dl[:, a:b].sum(axis=1)[..., None])  # (Bsz,D,N)
        aggs.append((P, hend, ylocal))
    carry = hh.copy()
    for (a, b), (P, hend, ylocal) in zip(chunks, aggs):
        # outputs: local outputs plus C_t . (prod_{s<=t} abar_s) carry
        cum = np.exp(A.astype(np.float64)[None, None] * np.cumsum(dl[:, a:b], axis=1)[..., None])
        corr = np.einsum("bldn,bdn,bln->bld", cum, carry, C[:, a:b].astype(np.float64))
        close(ylocal + corr, y[:, a:b], 1e-12, 1e-13)
        carry = P * carry + hend                                     # (a2 a1, a2 b1 + b2)
    close(carry, hT, 1e-12, 1e-13)


# ---------------------------------------------------------------- P10 step == fwd

def test_step_closed_form(orc):
    Bsz, D, N = 3, 4, 6
    g = np.random.default_rng(11)
    st = g.standard_normal((Bsz, D, N))
    x = g.standard_normal((Bsz, D)).astype(np.float32)
    dl = (0.05 + g.random((Bsz, D))).astype(np.float32)
    A = (-0.2 - g.random((D, N))).astype(np.float32)
    B = g.standard_normal((Bsz, N)).astype(np.float32)
    C = g.standard_normal((Bsz, N)).astype(np.float32)
    s = st.copy()
    y = orc.selscan_step(s, x, dl, A, B, C)
    ref = np.exp(dl.astype(np.float64)[..., None] * A.astype(np.float64)[None]) * st \
        + dl.astype(np.float64)[..., None] * B.astype(np.float64)[:, None, :] * x.astype(np.float64)[..., None]
    close(s, ref, 1e-14)
    close(y, np.einsum("bdn,bn->bd", ref, C.astype(np.float64)), 1e-13, 1e-15)


def test_steps_equal_forward(orc):
    Bsz, L, D, N = 2, 25, 3, 4
    x, u, A, B, C, hh = rand_inputs(Bsz, L, D, N, seed=12, h0=True)
    dl = sp(u).astype(np.float32)
    y, hT = orc.selscan_fwd(x, dl, A, B, C, delta_softplus=False, h0=hh)
    s = hh.copy()
    for t in range(L):
        yt = orc.selscan_step(s, x[:, t], dl[:, t], A, B[:, t], C[:, t])
        assert np.array_equal(yt, y[:, t])
    assert np.array_equal(s, hT)
    # chains subset of the step
    s2 = hh.reshape(Bsz * D, N)[[1, 4]].copy()
    for t in range(L):
        yt = orc.selscan_step(s2, x[:, t], dl[:, t], A, B[:, t], C[:, t], chains=[1, 4])
        assert np.array_equal(yt, y[:, t].reshape(-1)[[1, 4]])


# ---------------------------------------------------------------- P11 structure

def test_linearity_and_independence(orc):
    Bsz, L, D, N = 2, 20, 4, 3
    x1, u, A, B, C, h1 = rand_inputs(Bsz, L, D, N, seed=13, h0=True)
    x2, _, _, _, _, h2 = rand_inputs(Bsz, L, D, N, seed=14, h0=True)
    al, be = 0.75, -1.25
    y1, t1 = orc.selscan_fwd(x1, u, A, B, C, True, h1)
    y2, t2 = orc.selscan_fwd(x2, u, A, B, C, True, h2)
    x12 = (al * x1.astype(np.float64) + be * x2.astype(np.float64))
    # keep x exact in fp32: use multiples that are exact for these factors
    y12, t12 = orc.selscan_fwd(x12.astype(np.float32), u, A, B, C, True, al * h1 + be * h2)
    assert np.abs(x12.astype(np.float32) - x12).max() < 1e-6
    lin = al * y1 + be * y2
    # the fp32 rounding of x12 is the only perturbation; bound it loosely
    close(y12, lin, 1e-5, 1e-5)
    # scaling B or C by a power of two scales y exactly (no h0)
    y0, _ = orc.selscan_fwd(x1, u, A, B, C, True)
    yb, _ = orc.selscan_fwd(x1, u, A, B * 4, C, True)
    yc, _ = orc.selscan_fwd(x1, u, A, B, C * 0.5, True)
    assert np.array_equal(yb, 4 * y0) and np.array_equal(yc, 0.5 * y0)
    # permuting channels permutes outputs (A permuted with them)
    perm = np.array([2, 0, 3, 1])
    yp, tp = orc.selscan_fwd(x1[:, :, perm], u[:, :, perm], A[perm], B, C, True, h1[:, perm])
    y0h, t0h = orc.selscan_fwd(x1, u, A, B, C, True, h1)
    assert np.array_equal(yp, y0h[:, :, perm]) and np.array_equal(tp, t0h[:, perm])
    # chains are independent: changing channel 3 of batch 1 leaves every other chain alone
    x3 = x1.copy(); x3[1, :, 3] += 1.0
    y3, _ = orc.selscan_fwd(x3, u, A, B, C, True, h1)
    mask = np.ones_like(y3, bool); mask[1, :, 3] = False
    assert np.array_equal(y3[mask], y0h[mask]) and not np.array_equal(y3[1, :, 3], y0h[1, :, 3])


def test_threads_and_chain_subset_bit_identical(orc):
    Bsz, L, D, N = 3, 33, 5, 4
    x, u, A, B, C, hh = rand_inputs(Bsz, L, D, N, seed=15, h0=True)
    y1, h1 = orc.selscan_fwd(x, u, A, B, C, True, hh, nthreads=1)
    y4, h4 = orc.selscan_fwd(x, u, A, B, C, True, hh, nthreads=4)
    assert np.array_equal(y1, y4) and np.array_equal(h1, h4)
    chains = np.array([0, 7, 14, 3])
    yc, hc = orc.selscan_fwd_chains(x, u, A, B, C, chains, True, hh, nthreads=2)
    for i, c in enumerate(chains):
        b, d = divmod(int(c), D)
        assert np.array_equal(yc[i], y1[b, :, d]) and np.array_equal(hc[i], h1[b, d])


def test_empty_sequence(orc):
    hh = np.arange(2 * 3 * 4, dtype=np.float64).reshape(2, 3, 4)
    z = np.zeros((2, 0, 3), np.float32)
    y, hT = orc.selscan_fwd(z, z, np.zeros((3, 4), np.float32), np.zeros((2, 0, 4), np.float32),
                            np.zeros((2, 0, 4), np.float32), True, hh)
    assert y.shape == (2, 0, 3) and np.array_equal(hT, hh)


def test_workload_inputs_feed_oracle(orc):
    """The tiny workload runs end to end and its bf16 encoding round-trips."""
    i = W.workload_inputs(1)
    y, hT = orc.selscan_fwd(i.f32("x"), i.f32("delta"), i.A, i.f32("B"), i.f32("C"), True)
    assert y.shape == (1, 64, 16) and np.all(np.isfinite(y))


# ---- the block's skip and gate around the scan (section 3.4, MambaBlock) ----

def gate_inputs(Bsz, L, D, seed):
    g = np.random.default_rng(seed)
    Dskip = (0.5 + g.random(D)).astype(np.float32)
    z = (2.0 * g.standard_normal((Bsz, L, D))).astype(np.float32)
    return Dskip, z


def test_gate_with_zero_readout_is_skip_times_silu(orc):
    """C = 0 silences the scan: the block's output is Dskip[d] x silu(z), with
    silu(z) = z * sigmoid(z) from scipy's logistic function."""
    from scipy.special import expit
    x, u, A, B, C, _ = rand_inputs(2, 20, 5, 4, seed=31)
    Dskip, z = gate_inputs(2, 20, 5, seed=32)
    y, _ = orc.selscan_fwd(x, u, A, B, np.zeros_like(C), True, Dskip=Dskip, z=z)
    zz = z.astype(np.float64)
    ref = Dskip.astype(np.float64)[None, None, :] * x.astype(np.float64) * zz * expit(zz)
    assert np.allclose(y, ref, rtol=1e-14, atol=1e-15)


def test_skip_without_gate_adds_Dx_to_the_scan(orc):
    x, u, A, B, C, hh = rand_inputs(2, 30, 6, 4, seed=33, h0=True)
    Dskip, _ = gate_inputs(2, 30, 6, seed=34)
    y0, h0 = orc.selscan_fwd(x, u, A, B, C, True, hh)
    y1, h1 = orc.selscan_fwd(x, u, A, B, C, True, hh, Dskip=Dskip)
    assert np.array_equal(h0, h1)                      # the state does not see the skip
    assert np.allclose(y1, y0 + Dskip[None, None, :].astype(np.float64) * x, rtol=1e-14, atol=1e-14)


def test_gate_odd_part_is_identity(orc):
    """silu(z) - silu(-z) = z for every z, so gating with z and with -z differ
    by exactly (scan + skip) * z."""
    x, u, A, B, C, hh = rand_inputs(2, 25, 5, 3, seed=35, h0=True)
    Dskip, z = gate_inputs(2, 25, 5, seed=36)
    yp, _ = orc.selscan_fwd(x, u, A, B, C, True, hh, Dskip=Dskip, z=z)
    yn, _ = orc.selscan_fwd(x, u, A, B, C, True, hh, Dskip=Dskip, z=-z)
    ys, _ = orc.selscan_fwd(x, u, A, B, C, True, hh, Dskip=Dskip)
    assert np.allclose(yp - yn, ys * z.astype(np.float64), rtol=1e-12, atol=1e-12)


def test_gate_limits(orc):
    """silu(0) = 0 silences the block; silu(z) -> z for large z."""
    x, u, A, B, C, _ = rand_inputs(1, 12, 4, 4, seed=37)
    Dskip, _ = gate_inputs(1, 12, 4, seed=38)
    y0, _ = orc.selscan_fwd(x, u, A, B, C, True, Dskip=Dskip, z=np.zeros_like(x))
    assert np.array_equal(y0, np.zeros_like(y0))
    ys, _ = orc.selscan_fwd(x, u, A, B, C, True, Dskip=Dskip)
    y40, _ = orc.selscan_fwd(x, u, A, B, C, True, Dskip=Dskip, z=np.full_like(x, 40.0))
    assert np.allclose(y40, 40.0 * ys, rtol=1e-15, atol=0)


def test_gated_steps_equal_gated_forward(orc):
    Bsz, L, D, N = 2, 9, 4, 5
    x, u, A, B, C, hh = rand_inputs(Bsz, L, D, N, seed=39, softplus=False, h0=True)
    Dskip, z = gate_inputs(Bsz, L, D, seed=40)
    y, hT = orc.selscan_fwd(x, u, A, B, C, False, hh, Dskip=Dskip, z=z)
    st = hh.copy()
    for t in range(L):
        yt = orc.selscan_step(st, x[:, t], u[:, t], A, B[:, t], C[:, t], Dskip=Dskip, z=z[:, t])
        assert np.allclose(yt, y[:, t], rtol=1e-13, atol=1e-13)
    assert np.allclose(st, hT, rtol=1e-13, atol=1e-13)


# ---- zero-order-hold discretisation (section 2.2) ----------------------------

def test_zoh_is_the_exact_solution_for_held_inputs(orc):
    """With x, delta and B held over each step, the continuous system
    h' = A h + B x (diagonal A) moves from h to exp(dA) h + (exp(dA) - 1)/A B x.
    Each state is checked against scipy's matrix exponential of the augmented
    2x2 system [[A dl, B x dl], [0, 0]] applied to (h, 1)."""
    from scipy.linalg import expm
    Bsz, L, D, N = 1, 6, 3, 4
    x, u, A, B, C, hh = rand_inputs(Bsz, L, D, N, seed=41, softplus=False, h0=True)
    y, hT = orc.selscan_fwd(x, u, A, B, C, False, hh, zoh=True)
    h = hh.copy()
    for t in range(L):
        for d in range(D):
            dl = float(u[0, t, d])
            for n in range(N):
                M = np.array([[float(A[d, n]) * dl, float(B[0, t, n]) * float(x[0, t, d]) * dl], [0.0, 0.0]])
                h[0, d, n] = (expm(M) @ np.array([h[0, d, n], 1.0]))[0]
        assert np.allclose(y[0, t], (h[0] * C[0, t].astype(np.float64)[None, :]).sum(-1), rtol=1e-12, atol=1e-12)
    assert np.allclose(hT, h, rtol=1e-12, atol=1e-12)


def test_zoh_fixed_point_does_not_depend_on_delta(orc):
    """Held x and B: every step maps h to exp(dA) h + (exp(dA) - 1)/A B x, whose
    fixed point -B x / A is the continuous system's, for any step size."""
    D, N, L = 2, 3, 3000
    A = np.array([[-0.5, -1.0, -2.0], [-0.75, -1.5, -3.0]], np.float32)
    Bv = np.array([0.3, -0.7, 1.1], np.float32)
    for dl in (0.05, 0.5):
        x = np.full((1, L, D), 0.8, np.float32)
        u = np.full((1, L, D), dl, np.float32)
        B = np.tile(Bv, (1, L, 1)).astype(np.float32)
        _, hT = orc.selscan_fwd(x, u, A, B, np.zeros_like(B), False, zoh=True)
        star = -(Bv[None, :].astype(np.float64) * float(np.float32(0.8))) / A.astype(np.float64)
        assert np.allclose(hT[0], star, rtol=1e-9, atol=1e-12)


def test_zoh_limits(orc):
    """dl * A -> 0: the zero-order-hold Bbar tends to dl * B (the simplified
    form), exactly at A = 0; it stays below dl * B for A < 0."""
    x, u, A, B, C, hh = rand_inputs(2, 10, 3, 4, seed=43, softplus=False, h0=True)
    y0, h0_ = orc.selscan_fwd(x, u, np.zeros_like(A), B, C, False, hh)
    y1, h1 = orc.selscan_fwd(x, u, np.zeros_like(A), B, C, False, hh, zoh=True)
    assert np.array_equal(y0, y1) and np.array_equal(h0_, h1)
    tiny = (u * np.float32(1e-7)).astype(np.float32)
    ye, _ = orc.selscan_fwd(x, tiny, A, B, C, False, hh)
    yz, _ = orc.selscan_fwd(x, tiny, A, B, C, False, hh, zoh=True)
    assert np.allclose(yz, ye, rtol=1e-5, atol=1e-12)


def test_zoh_steps_equal_zoh_forward(orc):
    Bsz, L, D, N = 2, 8, 3, 5
    x, u, A, B, C, hh = rand_inputs(Bsz, L, D, N, seed=44, softplus=False, h0=True)
    y, hT = orc.selscan_fwd(x, u, A, B, C, False, hh, zoh=True)
    st = hh.copy()
    for t in range(L):
        yt = orc.selscan_step(st, x[:, t], u[:, t], A, B[:, t], C[:, t], zoh=True)
        assert np.allclose(yt, y[:, t], rtol=1e-13, atol=1e-13)
    assert np.allclose(st, hT, rtol=1e-13, atol=1e-13)


# ---- the causal depthwise convolution before the scan (section 3.4) ---------

def conv_inputs(Bsz, L, D, K, seed):
    g = np.random.default_rng(seed)
    x = g.standard_normal((Bsz, L, D)).astype(np.float32)
    w = g.standard_normal((D, K)).astype(np.float32)
    bias = g.standard_normal(D).astype(np.float32)
    return x, w, bias


def test_conv_is_a_fir_filter(orc):
    """Without SiLU each channel is numpy's full convolution with the taps in
    reverse order, cut to the first L outputs, plus the bias."""
    x, w, bias = conv_inputs(2, 37, 5, 4, seed=51)
    out, _ = orc.conv1d(x, w, bias, silu=False)
    for b in range(2):
        for d in range(5):
            ref = np.convolve(x[b, :, d].astype(np.float64), w[d, ::-1].astype(np.float64))[:37] + bias[d]
            assert np.allclose(out[b, :, d], ref, rtol=1e-14, atol=1e-14)


def test_conv_silu(orc):
    from scipy.special import expit
    x, w, bias = conv_inputs(1, 20, 3, 4, seed=52)
    lin, _ = orc.conv1d(x, w, bias, silu=False)
    out, _ = orc.conv1d(x, w, bias, silu=True)
    assert np.allclose(out, lin * expit(lin), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("K", [1, 2, 4, 7])
def test_conv_streams_through_its_state(orc, K):
    """Cutting the sequence anywhere and handing the last K-1 inputs over as
    the state gives the same outputs and the same final state; decode steps
    of one token each do too."""
    x, w, bias = conv_inputs(2, 30, 4, K, seed=53 + K)
    full, st_full = orc.conv1d(x, w, bias)
    a, st_a = orc.conv1d(x[:, :11], w, bias)
    b_, st_b = orc.conv1d(x[:, 11:], w, bias, state_in=st_a)
    assert np.array_equal(np.concatenate([a, b_], axis=1), full)
    assert np.array_equal(st_b, st_full)
    st = None
    for t in range(30):
        o, st = orc.conv1d(x[:, t:t + 1], w, bias, state_in=st)
        assert np.array_equal(o[:, 0], full[:, t])
    assert np.array_equal(st, st_full)
    if K > 1:
        assert np.array_equal(st_full, np.transpose(x[:, -(K - 1):], (0, 2, 1)))


def test_conv_single_tap_is_pointwise(orc):
    from scipy.special import expit
    x, w, bias = conv_inputs(1, 9, 3, 1, seed=58)
    out, st = orc.conv1d(x, w, bias)
    lin = x.astype(np.float64) * w[:, 0].astype(np.float64) + bias.astype(np.float64)
    assert np.allclose(out, lin * expit(lin), rtol=1e-14, atol=1e-15) and st.shape == (1, 3, 0)


# ---- the backward pass -------------------------------------------------------
# The pages give no gradient formulas (the hardware-aware design of
# booiljung.github.io "3.1 LTI ... Input-Dependent parameters", section
# 3.1.5.3, only says the backward pass recomputes the states). The oracle's
# reverse sweep is the chain rule on the recurrence; these pins fix it by
# numerical differentiation of the forward oracle, by automatic
# differentiation of an unrolled forward, and by homogeneity identities.

def _loss(orc, x, u, A, B, C, h0, gy, ghT, softplus):
    y, hT = orc.selscan_fwd(x, u, A, B, C, softplus, h0=h0)
    tot = float(np.sum(gy * y))
    if ghT is not None:
        tot += float(np.sum(ghT * hT))
    return tot


def _central(f, v, h):
    return (f(v + h) - f(v - h)) / (2 * h)


@pytest.mark.parametrize("softplus,h0", [(True, False), (True, True), (False, True)])
def test_bwd_matches_central_differences(orc, softplus, h0):
    """Every gradient entry against a Richardson-extrapolated central
    difference of the forward oracle's loss. The fp32 inputs are rounded to
    multiples of 2^-12, so every perturbed value v +- 2^-9, v +- 2^-10 is
    exact in fp32 and the differences are symmetric."""
    x, u, A, B, C, hh = rand_inputs(2, 5, 2, 3, seed=70 + 2 * softplus + h0, softplus=softplus, h0=h0)
    x, u, A, B, C = (np.round(v * 4096.0).astype(np.float32) / np.float32(4096.0) for v in (x, u, A, B, C))
    g = np.random.default_rng(71)
    gy = g.standard_normal(x.shape)
    ghT = g.standard_normal((2, 2, 3))
    grads = orc.selscan_bwd(x, u, A, B, C, gy, softplus, h0=hh, ghT=ghT)
    args = dict(x=x, u=u, A=A, B=B, C=C, h0=hh)
    names = dict(x="dx", u="ddelta", A="dA", B="dB", C="dC", h0="dh0")
    for key, gname in names.items():
        base = args[key]
        if base is None:
            continue
        num = np.zeros(base.shape)
        for idx in np.ndindex(base.shape):
            def f(v, key=key, idx=idx):
                a = {k: (None if w is None else w.copy()) for k, w in args.items()}
                a[key][idx] = v
                return _loss(orc, a["x"], a["u"], a["A"], a["B"], a["C"], a["h0"], gy, ghT, softplus)
            v0 = float(base[idx])
            d1, d2 = _central(f, v0, 2.0 ** -9), _central(f, v0, 2.0 ** -10)
            num[idx] = (4 * d2 - d1) / 3
        close(grads[gname], num, rtol=1e-9, atol=1e-10)


def _torch_grads(x, u, A, B, C, h0, gy, ghT, softplus):
    """Gradients by torch autograd (fp64, CPU) of the recurrence unrolled
    step by step with tensor ops."""
    import torch
    t = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)
    tx, tu, tA, tB, tC = t(x), t(u), t(A), t(B), t(C)
    th0 = t(h0) if h0 is not None else None
    Bsz, L, D = x.shape
    dl = torch.nn.functional.softplus(tu) if softplus else tu
    h = th0 if th0 is not None else torch.zeros(Bsz, D, A.shape[1], dtype=torch.float64)
    ys = []
    for s in range(L):
        d = dl[:, s, :, None]                                   # (Bsz, D, 1)
        h = torch.exp(d * tA[None]) * h + d * tB[:, s, None, :] * tx[:, s, :, None]
        ys.append((h * tC[:, s, None, :]).sum(-1))
    y = torch.stack(ys, 1)
    loss = (y * torch.from_numpy(gy)).sum() + (h * torch.from_numpy(ghT)).sum()
    loss.backward()
    out = dict(dx=tx.grad, ddelta=tu.grad, dA=tA.grad, dB=tB.grad, dC=tC.grad)
    if th0 is not None:
        out["dh0"] = th0.grad
    return {k: v.numpy() for k, v in out.items()}


@pytest.mark.parametrize("softplus", [True, False])
def test_bwd_matches_autograd(orc, softplus):
    x, u, A, B, C, hh = rand_inputs(2, 33, 3, 4, seed=72 + softplus, softplus=softplus, h0=True)
    g = np.random.default_rng(73)
    gy = g.standard_normal(x.shape)
    ghT = g.standard_normal(hh.shape)
    got = orc.selscan_bwd(x, u, A, B, C, gy, softplus, h0=hh, ghT=ghT)
    ref = _torch_grads(x, u, A, B, C, hh, gy, ghT, softplus)
    for k, v in ref.items():
        close(got[k], v, rtol=1e-11, atol=1e-12)


def test_bwd_homogeneity_identities(orc):
    """y and hT are linear in (x, h0) jointly, so by Euler's identity the loss
    equals sum dx*x + sum dh0*h0; y is linear in C, so sum gy*y = sum dC*C;
    with h0 = 0 everything is linear in B, so the loss equals sum dB*B."""
    x, u, A, B, C, hh = rand_inputs(2, 200, 8, 16, seed=74, h0=True)
    g = np.random.default_rng(75)
    gy = g.standard_normal(x.shape)
    ghT = g.standard_normal(hh.shape)
    y, hT = orc.selscan_fwd(x, u, A, B, C, True, h0=hh)
    gr = orc.selscan_bwd(x, u, A, B, C, gy, True, h0=hh, ghT=ghT)
    loss = np.sum(gy * y) + np.sum(ghT * hT)
    scale = np.sum(np.abs(gy * y)) + np.sum(np.abs(ghT * hT))
    assert abs(np.sum(gr["dx"] * x) + np.sum(gr["dh0"] * hh) - loss) <= 1e-12 * scale
    gr0 = orc.selscan_bwd(x, u, A, B, C, gy, True, h0=hh)   # no hT gradient
    assert abs(np.sum(gr0["dC"] * C) - np.sum(gy * y)) <= 1e-12 * np.sum(np.abs(gy * y))
    y0, hT0 = orc.selscan_fwd(x, u, A, B, C, True)          # h0 = 0
    gr1 = orc.selscan_bwd(x, u, A, B, C, gy, True, ghT=ghT)
    loss0 = np.sum(gy * y0) + np.sum(ghT * hT0)
    scale0 = np.sum(np.abs(gy * y0)) + np.sum(np.abs(ghT * hT0))
    assert abs(np.sum(gr1["dB"] * B) - loss0) <= 1e-12 * scale0


def test_bwd_empty_sequence_passes_the_state_gradient_through(orc):
    x, u, A, B, C, hh = rand_inputs(2, 0, 3, 4, seed=76, h0=True)
    ghT = np.random.default_rng(77).standard_normal(hh.shape)
    gr = orc.selscan_bwd(x, u, A, B, C, np.zeros(x.shape), True, h0=hh, ghT=ghT)
    assert np.array_equal(gr["dh0"], ghT) and not gr["dA"].any()


# ---- Mamba-2 SSD -------------------------------------------------------------
# The state-space-dual model of "Mamba: Selective State Space Models"
# (youngju.dev), section 4.1: a recurrence with a scalar decay per head, and
# its dual Y = (T * M) X with T the causal mask and M semiseparable.

def ssd_case(Bsz, L, H, P, N, seed, h0=True, softplus=True):
    x, dt, A, B, C, hh = W.ssd_inputs(Bsz, L, H, P, N, seed=seed, with_h0=h0)
    if not softplus:
        dt = np.abs(dt) * np.float32(0.1)
    return x, dt, A, B, C, hh


def test_ssd_headdim_one_is_the_selective_scan(orc):
    """With headdim 1 and one head per channel, the SSD recurrence is the
    selective scan with A[d, n] = A_head for every state n."""
    Bsz, L, H, N = 2, 40, 5, 6
    x, dt, A, B, C, hh = ssd_case(Bsz, L, H, 1, N, seed=80)
    y, hT = orc.ssd_fwd(x, dt, A, B, C, True, h0=hh)
    A_dn = np.repeat(A[:, None], N, axis=1)
    ys, hs = orc.selscan_fwd(x[..., 0], dt, A_dn, B, C, True, h0=hh[..., 0].astype(np.float64))
    close(y[..., 0], ys, rtol=1e-14, atol=1e-15)
    close(hT[..., 0], hs, rtol=1e-14, atol=1e-15)


def ssd_dual(x, dt, A, B, C, h0, softplus):
    """The attention view: for each (b, head), with cum_t = sum_{r<=t} dl_r A,
    M[t, s] = (C_t . B_s) dl_s exp(cum_t - cum_s) under the causal mask, y = M x
    (+ C_t exp(cum_t) h0); hT = sum_s exp(cum_{L-1} - cum_s) dl_s B_s x_s^T
    (+ exp(cum_{L-1}) h0)."""
    x = x.astype(np.float64); B = B.astype(np.float64); C = C.astype(np.float64)
    dl = sp(dt) if softplus else dt.astype(np.float64)
    Bsz, L, H, P = x.shape
    N = B.shape[2]
    y = np.zeros(x.shape); hT = np.zeros((Bsz, H, N, P))
    T = np.tril(np.ones((L, L)))
    for b in range(Bsz):
        G = C[b] @ B[b].T                                   # (L, L): C_t . B_s
        for hd in range(H):
            cum = np.cumsum(dl[b, :, hd] * np.float64(A[hd]))
            decay = np.exp(np.minimum(cum[:, None] - cum[None, :], 0.0))
            M = T * G * dl[b, None, :, hd] * decay
            y[b, :, hd] = M @ x[b, :, hd]
            w = np.exp(cum[-1] - cum) * dl[b, :, hd]
            hT[b, hd] = (B[b] * w[:, None]).T @ x[b, :, hd]
            if h0 is not None:
                y[b, :, hd] += (C[b] * np.exp(cum)[:, None]) @ h0[b, hd]
                hT[b, hd] += np.exp(cum[-1]) * h0[b, hd]
    return y, hT


@pytest.mark.parametrize("softplus,h0", [(True, True), (False, False)])
def test_ssd_dual_quadratic_form(orc, softplus, h0):
    x, dt, A, B, C, hh = ssd_case(2, 33, 3, 4, 5, seed=81 + h0, h0=h0, softplus=softplus)
    y, hT = orc.ssd_fwd(x, dt, A, B, C, softplus, h0=hh)
    yd, hd = ssd_dual(x, dt, A, B, C, None if hh is None else hh.astype(np.float64), softplus)
    close(y, yd, rtol=1e-11, atol=1e-12)
    close(hT, hd, rtol=1e-11, atol=1e-12)


def ssd_chunked(x, dt, A, B, C, h0, Q):
    """The chunked form: inside a chunk of Q steps the dual form, across
    chunks the state carried by its decay (the composition of section 4.1's
    recurrence over a chunk)."""
    x = x.astype(np.float64); B = B.astype(np.float64); C = C.astype(np.float64)
    dl = sp(dt)
    Bsz, L, H, P = x.shape
    N = B.shape[2]
    y = np.zeros(x.shape); hT = np.zeros((Bsz, H, N, P))
    for b in range(Bsz):
        for hd in range(H):
            st = np.zeros((N, P)) if h0 is None else h0[b, hd].copy()
            for c0 in range(0, L, Q):
                sl = slice(c0, min(L, c0 + Q))
                q = sl.stop - sl.start
                cum = np.cumsum(dl[b, sl, hd] * np.float64(A[hd]))
                decay = np.tril(np.exp(np.minimum(cum[:, None] - cum[None, :], 0.0)))
                M = (C[b, sl] @ B[b, sl].T) * dl[b, None, sl, hd] * decay
                y[b, sl, hd] = M @ x[b, sl, hd] + (C[b, sl] * np.exp(cum)[:, None]) @ st
                w = np.exp(cum[-1] - cum) * dl[b, sl, hd]
                st = np.exp(cum[-1]) * st + (B[b, sl] * w[:, None]).T @ x[b, sl, hd]
                assert q >= 1
            hT[b, hd] = st
    return y, hT


@pytest.mark.parametrize("Q", [1, 8, 16, 64])
def test_ssd_chunked_algorithm_equals_recurrence(orc, Q):
    x, dt, A, B, C, hh = ssd_case(1, 50, 2, 8, 16, seed=83)
    y, hT = orc.ssd_fwd(x, dt, A, B, C, True, h0=hh)
    yc, hc = ssd_chunked(x, dt, A, B, C, hh.astype(np.float64), Q)
    close(y, yc, rtol=1e-11, atol=1e-12)
    close(hT, hc, rtol=1e-11, atol=1e-12)


def test_ssd_heads_are_independent_and_linear(orc):
    x, dt, A, B, C, hh = ssd_case(1, 20, 4, 3, 5, seed=84)
    y, hT = orc.ssd_fwd(x, dt, A, B, C, True, h0=hh)
    perm = np.array([2, 0, 3, 1])
    yp, hp = orc.ssd_fwd(x[:, :, perm], dt[:, :, perm], A[perm], B, C, True, h0=hh[:, perm])
    assert np.array_equal(yp, y[:, :, perm]) and np.array_equal(hp, hT[:, perm])
    y2, h2 = orc.ssd_fwd(2 * x, dt, A, B, C, True, h0=2 * hh.astype(np.float64))
    close(y2, 2 * y, rtol=1e-14, atol=1e-15)
    close(h2, 2 * hT, rtol=1e-14, atol=1e-15)


# ---- the backward of the block's skip and gate ------------------------------

def _gated_case(seed, terms):
    x, u, A, B, C, hh = rand_inputs(2, 5, 2, 3, seed=seed, h0=True)
    g = np.random.default_rng(seed + 1)
    Dskip = (0.5 + g.random(2)).astype(np.float32) if terms != "gate" else None
    z = g.standard_normal(x.shape).astype(np.float32) if terms != "skip" else None
    q = lambda v: None if v is None else np.round(v * 4096.0).astype(np.float32) / np.float32(4096.0)
    return tuple(q(v) for v in (x, u, A, B, C)) + (hh, q(Dskip), q(z))


@pytest.mark.parametrize("terms", ["both", "skip", "gate"])
def test_bwd_gated_matches_central_differences(orc, terms):
    """Every gradient of a loss on the block's output (y + Dskip x) silu(z)
    against Richardson central differences of the gated forward oracle (inputs
    on a 2^-12 grid, so every perturbation is exact in fp32)."""
    x, u, A, B, C, hh, Dskip, z = _gated_case(90 + len(terms), terms)
    g = np.random.default_rng(91)
    gy = g.standard_normal(x.shape)
    ghT = g.standard_normal((2, 2, 3))
    grads = orc.selscan_bwd(x, u, A, B, C, gy, True, h0=hh, ghT=ghT, Dskip=Dskip, z=z)
    args = dict(x=x, u=u, A=A, B=B, C=C, h0=hh, Dskip=Dskip, z=z)
    names = dict(x="dx", u="ddelta", A="dA", B="dB", C="dC", h0="dh0", Dskip="dDskip", z="dz")

    def loss(a):
        y, hT = orc.selscan_fwd(a["x"], a["u"], a["A"], a["B"], a["C"], True, h0=a["h0"], Dskip=a["Dskip"],
                                z=a["z"])
        return float(np.sum(gy * y) + np.sum(ghT * hT))

    for key, gname in names.items():
        base = args[key]
        if base is None:
            assert gname not in grads
            continue
        num = np.zeros(base.shape)
        for idx in np.ndindex(base.shape):
            def f(v, key=key, idx=idx):
                a = {k: (None if w is None else w.copy()) for k, w in args.items()}
                a[key][idx] = v
                return loss(a)
            v0 = float(base[idx])
            d1, d2 = _central(f, v0, 2.0 ** -9), _central(f, v0, 2.0 ** -10)
            num[idx] = (4 * d2 - d1) / 3
        close(grads[gname], num, rtol=1e-9, atol=1e-10)


def test_bwd_gated_matches_autograd(orc):
    import torch
    x, u, A, B, C, hh = rand_inputs(2, 40, 3, 4, seed=94, h0=True)
    g = np.random.default_rng(95)
    Dskip = (0.5 + g.random(3)).astype(np.float32)
    z = g.standard_normal(x.shape).astype(np.float32)
    gy = g.standard_normal(x.shape)
    ghT = g.standard_normal(hh.shape)
    got = orc.selscan_bwd(x, u, A, B, C, gy, True, h0=hh, ghT=ghT, Dskip=Dskip, z=z)
    t = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)
    tx, tu, tA, tB, tC, th0, tD, tz = (t(v) for v in (x, u, A, B, C, hh, Dskip, z))
    dl = torch.nn.functional.softplus(tu)
    h = th0
    ys = []
    for s in range(x.shape[1]):
        d = dl[:, s, :, None]
        h = torch.exp(d * tA[None]) * h + d * tB[:, s, None, :] * tx[:, s, :, None]
        ys.append((h * tC[:, s, None, :]).sum(-1))
    y = (torch.stack(ys, 1) + tD * tx) * torch.nn.functional.silu(tz)
    ((y * torch.from_numpy(gy)).sum() + (h * torch.from_numpy(ghT)).sum()).backward()
    ref = dict(dx=tx.grad, ddelta=tu.grad, dA=tA.grad, dB=tB.grad, dC=tC.grad, dh0=th0.grad, dDskip=tD.grad,
               dz=tz.grad)
    for k, v in ref.items():
        close(got[k], v.numpy(), rtol=1e-11, atol=1e-12)
