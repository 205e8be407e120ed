"""Derives the polynomial behind the kernels' softplus (device_math.cuh).

softplus(u) = max(u, 0) + log1p(e) with e = exp(-|u|) in (0, 1]. log1p(e) is
evaluated as e * P(e), where P approximates log1p(e) / e on [0, 1] (a smooth
function falling from 1 to ln 2). P is fitted here by weighted least squares
on Chebyshev-spaced points, reweighting toward equal relative error (Lawson's
iteration for a minimax fit), rounded to fp32, and then checked by emulating
the kernel's fp32 fused-multiply-add Horner evaluation on a dense grid.

    python fit_log1p_poly.py [degree]      # prints coefficients and max error
"""
import sys

import numpy as np


def target(e):
    e = np.asarray(e, np.float64)
    return np.where(e == 0, 1.0, np.log1p(e) / np.where(e == 0, 1.0, e))


def fit(deg, iters=60):
    x = 0.5 - 0.5 * np.cos(np.linspace(0, np.pi, 4000))
    w = np.ones_like(x)
    V = np.vander(x, deg + 1, increasing=True)
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(V * w[:, None], target(x) * w, rcond=None)
        r = np.abs(V @ c - target(x)) / target(x)
        w = w * (r / r.max() + 1e-3) ** 0.5
        w /= w.max()
    return [float(np.float32(v)) for v in c]


def fp32_horner(c32, e):
    """fp32 Horner with one rounding per fused multiply-add, then e * P in fp32."""
    r = np.full(e.shape, c32[-1], np.float64)
    for ck in c32[-2::-1]:
        r = (r * e.astype(np.float64) + ck).astype(np.float32).astype(np.float64)
    return (r * e.astype(np.float64)).astype(np.float32).astype(np.float64)


def max_rel_error(c32):
    e = np.concatenate([np.float32(2.0) ** -np.arange(1, 40, 0.25, dtype=np.float32),
                        np.random.default_rng(0).random(400000).astype(np.float32),
                        np.linspace(0, 1, 100001, dtype=np.float32)])
    e = e[(e > 0) & (e <= 1)].astype(np.float32)
    exact = np.log1p(e.astype(np.float64))
    return float(np.max(np.abs(fp32_horner(c32, e) - exact) / exact))


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 8
    c = fit(deg)
    print("coefficients (c0..c%d):" % deg, ", ".join("%.9ef" % v for v in c))
    print("max relative error of e*P(e) vs log1p(e): %.3e" % max_rel_error(c))
