"""Fits the polynomial of softplus_poly.cuh: log2(1 + u) on [0, 1] as
u (c1 + c2 u + ... + cK u^(K-1)), so that u = 0 (a masked column) gives
exactly 0.

Method: minimax by Lawson's iteratively re-weighted least squares (each
pass multiplies the weights by the current absolute error, which drives the
weighted least-squares solution towards the equioscillating minimax one) on
4000 Chebyshev nodes of [0, 1].  The coefficients are then rounded to fp32
and the largest error of fp32 Horner evaluation is measured on a dense grid.

  python fit_softplus_poly.py [K]     (K = 6 is the degree the kernel uses)

prints the coefficients c1..cK (as the C literals to paste) and that error.
"""

import sys

import numpy as np


def fit(K=6, nodes=4000, passes=300):
    """Coefficients c1..cK (float64) of the weighted least-squares minimax fit."""
    t = 0.5 + 0.5 * np.cos(np.pi * (np.arange(nodes) + 0.5) / nodes)
    f = np.log2(1.0 + t)
    V = np.vander(t, K + 1, increasing=True)[:, 1:]      # t, t^2, ..., t^K: no constant term
    w = np.ones_like(t)
    for _ in range(passes):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(V * sw[:, None], f * sw, rcond=None)
        e = np.abs(V @ c - f)
        w = w * e
        w /= w.sum()
    return c


def horner_f32(c, u):
    """fp32 Horner evaluation in the kernel's order: u (c1 + u (c2 + ... + u cK))."""
    c32 = np.asarray(c, dtype=np.float32)
    u = np.asarray(u, dtype=np.float32)
    acc = np.full_like(u, c32[-1])
    for k in range(len(c32) - 2, -1, -1):
        acc = (acc * u + c32[k]).astype(np.float32)
    return (acc * u).astype(np.float32)


def max_error_f32(c, points=400001):
    u = np.linspace(0.0, 1.0, points).astype(np.float32)
    return float(np.abs(horner_f32(c, u).astype(np.float64) - np.log2(1.0 + u.astype(np.float64))).max())


if __name__ == "__main__":
    K = int(sys.argv[1]) if len(sys.argv) > 1 else 6
    c = fit(K)
    print("coefficients c1..c%d:" % K, ", ".join("%.16gf" % float(np.float32(x)) for x in c))
    print("largest error of fp32 Horner evaluation on [0, 1]: %.3e" % max_error_f32(c))
