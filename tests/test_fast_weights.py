"""The one-exponential LSSAR weights of the tensor-core kernel's weight pass,
checked on the CPU against the exact weights of the notes' formulas.

Key design 1 makes the first-stage weights Softplus(x) of the length-scaled
cosine scores; Key design 2 re-weights them as ReLU^p(i A - O).  In the
kernel's log2 units (z = log2(e) x, sp2(z) = log2(1 + 2^z)) a row's weights
are w_j = (max(sp2(z_j) - theta, 0) kappa)^p with theta = O S1 / i and
kappa = 1 / (sp2(m) - theta).  On rows where a bound from the row's
statistics allows it, the kernel replaces sp2(z) by z + 2^-|z| / ln 2.  These
tests restate that replacement and its bound in float64 and check:

* the two inequalities the bound rests on (for every u in [0, 1] and z < 0);
* on seeded iid and needle rows, that every row the bound admits has its
  weight sum changed by no more than the bound, and its output by no more
  than 2 R max|v|;
* that the check has teeth: with the wrong constant (u instead of u / ln 2)
  some admitted row breaks the bound.
"""

import math

import numpy as np
import pytest

from lssar_attn_fwd_gb300.inputs import bf16_bits_to_f64, make_qkv
from oracle import l2_normalize_rows

LN2 = math.log(2.0)
C = 0.5 / LN2             # u^2 / (2 ln 2) bounds the overestimate
FAST_BOUND = 2e-4         # largest admitted relative change of a row's weight sum


def admitted(theta, kappa, i, p):
    """The kernel's per-row test, in float64 (log2 domain as in the kernel)."""
    ys = np.minimum(1.0, (p - 1) * kappa * C)
    two_eta_k = 2.0 * C * 2.0 ** (-2.0 * (theta - 1.0))
    l_r = (np.log2(i * p * C * kappa) + two_eta_k + (p - 1) * np.log2(ys)
           - 2.0 * (theta + ys / kappa - 1.0))
    l_c = np.log2(i) + p * np.log2(C * kappa)
    bound = 2.0 ** l_r + 2.0 ** l_c
    ok = (theta >= 1.5) & (p >= 4) & (bound <= FAST_BOUND)
    return ok, bound


def row_terms(q, k, d):
    """z = log2(e) ln d ln i qh.kh for every causal (i, j) of one head."""
    L = q.shape[0]
    s = l2_normalize_rows(q) @ l2_normalize_rows(k).T
    i = np.arange(1, L + 1, dtype=np.float64)
    z = (math.log(d) * np.log(i) / LN2)[:, None] * s
    mask = np.arange(L)[None, :] < np.arange(1, L + 1)[:, None]
    return np.where(mask, z, -np.inf), mask, i


def weights(z, mask, i, p, c1=1.0 / LN2):
    sp2 = np.where(mask, np.logaddexp2(0.0, z), 0.0)
    theta = np.where(i <= 3, 0.0, 1.0) * sp2.sum(1) / i
    m = z.max(1)
    kappa = 1.0 / (np.logaddexp2(0.0, m) - theta)
    y = np.clip((sp2 - theta[:, None]) * kappa[:, None], 0.0, 1.0)
    zf = np.where(mask, z, 0.0)
    yf = np.clip((zf + c1 * 2.0 ** -np.abs(zf) - theta[:, None]) * kappa[:, None], 0.0, 1.0)
    w = np.where(mask, y ** p, 0.0)
    wf = np.where(mask, yf ** p, 0.0)
    return w, wf, theta, kappa


def test_gap_of_the_one_exponential_softplus():
    u = np.linspace(0.0, 1.0, 200001)
    gap = u / LN2 - np.log2(1.0 + u)
    assert gap.min() >= -1e-15
    assert (gap <= C * u * u + 1e-15).all()


def test_negative_columns_stay_below_the_threshold():
    z = -np.concatenate([np.linspace(0.0, 1.0, 10001)[1:], np.linspace(1.0, 120.0, 10001)])
    assert (z + 2.0 ** z / LN2 < 1.5).all()
    assert (np.logaddexp2(0.0, z) < 1.0).all()


CASES = [("iid", 2048, 64, 15), ("needle", 2048, 64, 15), ("iid", 1024, 128, 15), ("iid", 2048, 64, 64)]


def run_case(structure, L, d, p, c1=1.0 / LN2):
    qb, kb, vb = make_qkv(1, 2, L, d, seed=11, structure=structure)
    qf, kf, vf = (bf16_bits_to_f64(t)[0] for t in (qb, kb, vb))
    out = []
    for h in range(2):
        z, mask, i = row_terms(qf[h], kf[h], d)
        w, wf, theta, kappa = weights(z, mask, i, p, c1)
        ok, bound = admitted(theta, kappa, i, p)
        rel = np.abs(wf - w).sum(1) / w.sum(1)
        o = (w @ vf[h]) / w.sum(1)[:, None]
        of = (wf @ vf[h]) / wf.sum(1)[:, None]
        dout = np.abs(of - o).max(1)
        out.append((ok, bound, rel, dout, np.abs(vf[h]).max()))
    return out


@pytest.mark.parametrize("structure,L,d,p", CASES)
def test_admitted_rows_stay_within_the_bound(structure, L, d, p):
    for ok, bound, rel, dout, vmax in run_case(structure, L, d, p):
        assert ok.mean() > 0.3, ok.mean()
        assert (rel[ok] <= bound[ok]).all()
        assert (dout[ok] <= 2.0 * bound[ok] * vmax).all()


def test_wrong_constant_breaks_the_bound():
    broken = False
    for ok, bound, rel, dout, vmax in run_case("iid", 2048, 64, 15, c1=1.0):
        broken |= bool((rel[ok] > bound[ok]).any())
    assert broken


@pytest.mark.parametrize("p", [15, 40])
def test_backward_factor_stays_within_the_bound_at_p_minus_1(p):
    # The backward's row pass needs u = y^(p-1) as well as w = y^p: on rows
    # admitted at both p and p - 1, the sum of u over the row moves by at
    # most the bound at p - 1, relative to that sum (the same argument with
    # p - 1 in place of p; the row maximum has u = 1, so the sum is >= 1).
    qb, kb, vb = make_qkv(1, 2, 2048, 64, seed=12)
    qf, kf = (bf16_bits_to_f64(t)[0] for t in (qb, kb))
    for h in range(2):
        z, mask, i = row_terms(qf[h], kf[h], 64)
        _, _, theta, kappa = weights(z, mask, i, p)
        ok_p, _ = admitted(theta, kappa, i, p)
        ok_q, bound_q = admitted(theta, kappa, i, p - 1)
        ok = ok_p & ok_q
        u, uf, _, _ = weights(z, mask, i, p - 1)
        rel = np.abs(uf - u).sum(1) / u.sum(1)
        assert ok.mean() > 0.5, ok.mean()
        assert (rel[ok] <= bound_q[ok]).all()
