"""Float64 NumPy oracle: causal LSSAR, LSSA and softmax attention forward.

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU baseline).  It is slow,
plain and written to be checked by eye against the notes on "Softplus
Attention with Re-weighting Boosts Length Extrapolation in Large Language
Models" (papernotes.org, arXiv 2501.13428):

* Background: ``A = Softmax(QK^T/sqrt(d) + M)`` -- the softmax mode.
* Key design 1 (LSSA): ``Q_i <- Q_i/||Q_i||_2``, ``K_i <- K_i/||K_i||_2``,
  ``A = Softplus((log d . log N) (.) QK^T) (.) M'`` where row i of N is all
  ``i`` and ``M'`` is the 0/1 lower-triangular mask, then ``A_i <- A_i/||A_i||_1``.
* Key design 2 (re-weighting): ``A <- ReLU^p(A (.) N - O)``,
  ``A_i <- A_i/||A_i||_1``, with O all ones except rows 1-3 which are 0.
* Key design 3: the mask multiplies (0 replaces -inf) because Softplus is
  non-negative; it is applied after the Softplus.
* The attention output is ``A V``.
* Ablations (the notes' ablation table, 8K validation loss): re-weighting on
  a softmax normaliser, ``A = Softmax(QK^T/sqrt(d) + M)`` followed by Key
  design 2; and sigmoid + L1 + re-weighting, Key design 1 with Sigmoid in
  place of Softplus, followed by Key design 2.

Readings where the notes are silent (each is also listed in the design doc):
natural log; 1-based row index i (= number of attended tokens); the L2 norm
is clamped at 1e-12; ReLU^p is ``max(.,0)**p`` with integer p >= 1; O also
covers masked columns (they end at zero either way); a re-weighted row whose
every entry is zero (only an exactly uniform LSSA row, i >= 4) is 0/0 and is
read as the uniform prefix mean.

Rows are evaluated independently (every output row depends only on its own
scores), so long sequences are processed in row blocks; nothing else is
blocked, fused or reordered.

Parity status: every function here is pinned by ``tests/test_oracle.py``
(brute force, closed forms, limits and invariants).  No printed worked
example exists in the notes, so general LSSAR rows are pinned through those
properties only.
"""

import math

import numpy as np

MODE_SOFTMAX = 0
MODE_LSSA = 1
MODE_LSSAR = 2
MODE_SOFTMAX_RW = 3     # ablation: re-weighting on a softmax normaliser
MODE_SIGMOID_RW = 4     # ablation: sigmoid + L1 + re-weighting

NORM_EPS = 1e-12

# A re-weighting input y = i*A - O at or below this counts as zero.  In exact
# arithmetic a uniform LSSA row (the 0/0 case) has y = 0 on every entry; its
# float64 evaluation leaves residues of the order of i * 2^-53 of either sign,
# which the power p would otherwise turn into an arbitrary selection.
Y_ZERO = 1e-10


def softplus(x):
    """Softplus(x) = log(1 + e^x)  [Key design 1: Softplus replaces e^x].

    Evaluated as max(x, 0) + log1p(exp(-|x|)), which equals log(1+e^x)
    exactly in real arithmetic and never overflows.
    """
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def sigmoid(x):
    """1 / (1 + e^-x), the nonnegative map of the sigmoid ablation, evaluated
    without overflow for either sign of x."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def l2_normalize_rows(x, eps=NORM_EPS):
    """Q_i <- Q_i/||Q_i||_2 (same for K)  [Key design 1].

    The notes give no epsilon; the norm is clamped at ``eps`` so a zero row
    stays a zero row.
    """
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, eps)


def length_scale(i, d):
    """Row factor log d * log i of ``(log d . log N)``  [Key design 1].

    ``i`` is the 1-based row index, i.e. the number of tokens row i attends
    to (row i of N is all i).  Natural logarithm.
    """
    return math.log(d) * np.log(np.asarray(i, dtype=np.float64))


def bias_o(i):
    """Row value of the bias matrix O: 0 for rows 1, 2, 3, else 1  [Key design 2]."""
    return np.where(np.asarray(i) <= 3, 0.0, 1.0)


def _causal(rows, nk):
    """M' restricted to the given 1-based rows: 1 where j <= i, else 0."""
    j = np.arange(1, nk + 1, dtype=np.int64)[None, :]
    return j <= np.asarray(rows, dtype=np.int64)[:, None]


def lssa_rows(q_rows, k, rows, d, phi=None):
    """Rows of the LSSA matrix  [Key design 1].

    q_rows: raw queries of the requested rows, shape (n, d).
    k:      raw keys 1..max(rows), shape (>= max(rows), d).
    rows:   1-based row indices, shape (n,).
    phi:    the nonnegative map, Softplus by default (Sigmoid for the ablation).
    Returns A of shape (n, max(rows)): zero where j > i, rows summing to 1.
    """
    phi = softplus if phi is None else phi
    rows = np.asarray(rows, dtype=np.int64)
    nk = int(rows.max())
    qh = l2_normalize_rows(q_rows)
    kh = l2_normalize_rows(k[:nk])
    s = qh @ kh.T                                   # cosine scores, in [-1, 1]
    z = length_scale(rows, d)[:, None] * s          # (log d . log N) (.) QK^T
    a = phi(z) * _causal(rows, nk)                  # Softplus first, then the 0/1 mask M'
    return a / a.sum(axis=1, keepdims=True)         # L1 normalisation of each row


def reweight_rows(a, rows, p, o_rows=None):
    """Re-weighting  [Key design 2]: ``ReLU^p(A (.) N - O)`` then L1 per row.

    a:      LSSA rows from :func:`lssa_rows`, shape (n, nk).
    rows:   1-based row indices, shape (n,).
    p:      integer exponent >= 1.
    o_rows: optional per-row override of O (used only by tests, e.g. O = 0).

    ``y = max(i*a - O, 0)`` (values at or below ``Y_ZERO`` are rounding
    residues of 0) and the result is ``(y/max_j y)^p`` normalised:
    dividing by the row maximum first is a common factor that the L1
    normalisation cancels, and it keeps large p inside float64 range.  A row
    with ``max_j y == 0`` is degenerate (0/0) and is read as the uniform
    prefix mean over its i attended tokens.
    """
    rows = np.asarray(rows, dtype=np.int64)
    if o_rows is None:
        o = bias_o(rows)
    else:
        o = np.broadcast_to(np.asarray(o_rows, dtype=np.float64), rows.shape)
    y = rows[:, None] * a - o[:, None]
    y = np.where(y > Y_ZERO, y, 0.0)              # ReLU, with rounding residues of 0 taken as 0
    ymax = y.max(axis=1)
    out = _causal(rows, a.shape[1]) / rows[:, None].astype(np.float64)
    ok = ymax > 0.0
    if np.any(ok):
        r = (y[ok] / ymax[ok, None]) ** int(p)
        out[ok] = r / r.sum(axis=1, keepdims=True)
    return out


def softmax_rows(q_rows, k, rows, d):
    """Rows of ``Softmax(QK^T/sqrt(d) + M)`` with M the causal -inf mask  [Background].

    Raw (unnormalised) q and k, scale 1/sqrt(d).
    """
    rows = np.asarray(rows, dtype=np.int64)
    nk = int(rows.max())
    s = (q_rows @ k[:nk].T) / math.sqrt(d)
    s = np.where(_causal(rows, nk), s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=1, keepdims=True)


def attention_rows(q, k, v, rows, mode, p=3, o_override=None):
    """Output rows ``A V`` of one head for the given 1-based rows.

    q, k, v: (L, d) arrays of one head (any real dtype; used in float64).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    d = q.shape[-1]
    nk = int(rows.max())
    if mode in (MODE_SOFTMAX, MODE_SOFTMAX_RW):
        w = softmax_rows(q[rows - 1], k, rows, d)
    elif mode in (MODE_LSSA, MODE_LSSAR):
        w = lssa_rows(q[rows - 1], k, rows, d)
    elif mode == MODE_SIGMOID_RW:
        w = lssa_rows(q[rows - 1], k, rows, d, phi=sigmoid)
    else:
        raise ValueError(f"unknown mode {mode}")
    if mode in (MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW):
        w = reweight_rows(w, rows, p, o_override)
    return w @ v[:nk]


def attention_forward(q, k, v, mode, p=3, rows=None, o_override=None, block=256):
    """Causal attention forward of every head of [..., L, d] inputs.

    rows: None for all rows 1..L, else 1-based row indices evaluated in every
    head (the output then has shape [..., len(rows), d]).
    Rows are processed ``block`` at a time, each block independently.
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    if q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must have the same shape")
    L, d = q.shape[-2], q.shape[-1]
    lead = q.shape[:-2]
    all_rows = np.arange(1, L + 1) if rows is None else np.asarray(rows, dtype=np.int64)
    if all_rows.size and (all_rows.min() < 1 or all_rows.max() > L):
        raise ValueError("rows out of range")
    qf = q.reshape((-1, L, d))
    kf = k.reshape((-1, L, d))
    vf = v.reshape((-1, L, d))
    out = np.empty((qf.shape[0], all_rows.size, d), dtype=np.float64)
    for h in range(qf.shape[0]):
        for s0 in range(0, all_rows.size, block):
            r = all_rows[s0:s0 + block]
            out[h, s0:s0 + block] = attention_rows(qf[h], kf[h], vf[h], r, mode, p, o_override)
    return out.reshape(lead + (all_rows.size, d))
