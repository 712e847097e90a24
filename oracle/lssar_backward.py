"""Float64 NumPy oracle: gradients of the causal LSSAR / LSSA / softmax forward.

TEST INFRASTRUCTURE ONLY (tests, smoke check).  The notes on "Softplus
Attention with Re-weighting Boosts Length Extrapolation in Large Language
Models" train GPT-2 models with this attention (Experiments) and remark that
its element-wise structure carries over to the backward pass of a
FlashAttention-style kernel (Method, "element-wise" remark), but print no
gradient formula.  This module therefore takes the forward of
``lssar_oracle`` step by step, in the order of Key designs 1 and 2, and
applies the chain rule to each step in reverse:

  forward                                   backward (per head, row i)
  1 qh = q/max(|q|,eps), kh likewise        dq = (dqh - qh (qh.dqh)) / |q|   (|q| > eps)
  2 s = qh kh^T                             dqh = ds kh,  dkh = ds^T qh
  3 z = (ln d ln i) s                       ds = (ln d ln i) dz
  4 a = phi(z) * M'                         dz = phi'(z) da * M'
  5 A = a / sum_j a                         da = (dA - sum_j A dA) / sum_j a
  6 y = max(i A - O, 0), r = (y/max y)^p,   dr = (dR - sum_j R dR) / sum_j r
    R = r / sum_j r                         dA = i [i A - O > 0] p (y/max y)^(p-1) dr / max y
  7 out = R v                               dR = dout v^T,  dv = R^T dout

The row maximum in step 6 is a positive common factor of the row, which the
L1 normalisation cancels; its own derivative contributes
``sum_j dr_j r_j (-p / max y) = 0`` and is left out.  A degenerate row (every
``y`` zero, read as the uniform prefix mean) is constant in q and k, so its
``dA`` is zero; its ``dv`` is ``dout / i`` on each attended key.

Softmax mode: ``A = softmax(q k^T / sqrt(d) + M)`` on raw rows, with the
textbook derivative ``dz = A (dA - sum_j A dA)``; the softmax-normaliser
ablation applies step 6 on top of it.

Parity status: pinned by ``tests/test_oracle_backward.py`` against central
finite differences of the (separately pinned) forward oracle in every mode,
against PyTorch autograd of float64 scaled-dot-product attention in softmax
mode, and by invariants (sum of dv, radial components of dq and dk, constant
values).
"""

import math

import numpy as np

from .lssar_oracle import (MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW, MODE_SOFTMAX,
                           MODE_SOFTMAX_RW, NORM_EPS, Y_ZERO, bias_o, length_scale, sigmoid,
                           softplus)

_REWEIGHT = (MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW)


def _phi_and_slope(z, mode):
    """The nonnegative map of step 4 and its derivative dphi/dz."""
    if mode == MODE_SIGMOID_RW:
        sg = sigmoid(z)
        return sg, sg * (1.0 - sg)
    # softplus' = sigmoid
    return softplus(z), sigmoid(z)


def _norm_backward(x, dxh, eps=NORM_EPS):
    """Gradient through xh = x / max(|x|, eps), row by row."""
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    big = n > eps
    xh = x / np.maximum(n, eps)
    radial = np.sum(xh * dxh, axis=-1, keepdims=True)
    return np.where(big, (dxh - xh * radial) / np.maximum(n, eps), dxh / eps)


def _reweight_backward(A, dR, rows, p, o_rows):
    """Step 6 in reverse: dA from dR for the rows of one head.

    Returns (R, dA).  Row-maximum scaling as in the forward oracle.
    """
    o = bias_o(rows) if o_rows is None else np.broadcast_to(
        np.asarray(o_rows, dtype=np.float64), rows.shape)
    i = rows[:, None].astype(np.float64)
    causal = np.arange(1, A.shape[1] + 1)[None, :] <= rows[:, None]
    y = i * A - o[:, None]
    active = y > Y_ZERO                               # the forward's ReLU (residues of 0 are 0)
    y = np.where(active, y, 0.0)
    ymax = y.max(axis=1)
    R = causal / i
    dA = np.zeros_like(A)
    ok = ymax > 0.0
    if np.any(ok):
        t = y[ok] / ymax[ok, None]
        r = t ** int(p)
        rs = r.sum(axis=1, keepdims=True)
        Rk = r / rs
        R[ok] = Rk
        dr = (dR[ok] - np.sum(Rk * dR[ok], axis=1, keepdims=True)) / rs
        slope = int(p) * t ** (int(p) - 1) / ymax[ok, None]
        dA[ok] = i[ok] * active[ok] * slope * dr
    return R, dA


def head_backward(q, k, v, dout, mode, p=3, o_override=None):
    """dq, dk, dv of one head; q, k, v, dout are (L, d)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    L, d = q.shape
    rows = np.arange(1, L + 1, dtype=np.int64)
    causal = rows[None, :] <= rows[:, None]

    # forward, keeping the intermediates
    if mode in (MODE_SOFTMAX, MODE_SOFTMAX_RW):
        z = (q @ k.T) / math.sqrt(d)
        z = np.where(causal, z, -np.inf)
        e = np.exp(z - z.max(axis=1, keepdims=True))
        A = e / e.sum(axis=1, keepdims=True)
    elif mode in (MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW):
        nq = np.sqrt(np.sum(q * q, axis=1, keepdims=True))
        nk = np.sqrt(np.sum(k * k, axis=1, keepdims=True))
        qh = q / np.maximum(nq, NORM_EPS)
        kh = k / np.maximum(nk, NORM_EPS)
        c = length_scale(rows, d)[:, None]
        z = c * (qh @ kh.T)
        phi, slope = _phi_and_slope(z, mode)
        a = phi * causal
        s1 = a.sum(axis=1, keepdims=True)
        A = a / s1
    else:
        raise ValueError(f"unknown mode {mode}")

    # step 7 and step 6 in reverse
    dR = (dout @ v.T) * causal
    if mode in _REWEIGHT:
        R, dA = _reweight_backward(A, dR, rows, p, o_override)
    else:
        R, dA = A, dR
    dv = R.T @ dout

    # steps 5 to 1 in reverse
    if mode in (MODE_SOFTMAX, MODE_SOFTMAX_RW):
        dz = A * (dA - np.sum(A * dA, axis=1, keepdims=True))
        dq = dz @ k / math.sqrt(d)
        dk = dz.T @ q / math.sqrt(d)
    else:
        da = (dA - np.sum(A * dA, axis=1, keepdims=True)) / s1
        dz = slope * da * causal
        ds = c * dz
        dq = _norm_backward(q, ds @ kh)
        dk = _norm_backward(k, ds.T @ qh)
    return dq, dk, dv


def attention_backward(q, k, v, dout, mode, p=3, o_override=None):
    """Gradients (dq, dk, dv) of sum(dout * out) for [..., L, d] inputs."""
    q = np.asarray(q)
    if not (q.shape == np.shape(k) == np.shape(v) == np.shape(dout)):
        raise ValueError("q, k, v, dout must have the same shape")
    L, d = q.shape[-2], q.shape[-1]
    lead = q.shape[:-2]
    flat = [np.asarray(x, dtype=np.float64).reshape((-1, L, d)) for x in (q, k, v, dout)]
    grads = [np.empty_like(flat[0]) for _ in range(3)]
    for h in range(flat[0].shape[0]):
        g = head_backward(flat[0][h], flat[1][h], flat[2][h], flat[3][h], mode, p, o_override)
        for dst, src in zip(grads, g):
            dst[h] = src
    return tuple(x.reshape(lead + (L, d)) for x in grads)
