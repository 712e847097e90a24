"""Pins for the float64 backward oracle (CPU only).

The gradients are tied to things other than the backward code itself:
central finite differences of the forward oracle (pinned on its own in
test_oracle.py), PyTorch autograd of float64 scaled-dot-product attention for
the softmax mode, and invariants that follow from the forward's structure
(rows of the attention matrix sum to one; the L2 normalisation makes the
output blind to the length of q_i and k_j; constant values give a constant
output).  A dropped term (the derivative through the row sum of step 5 or the
threshold of step 6), a transposed product or a wrong slope fails the finite
differences.
"""

import numpy as np
import pytest

from oracle import (MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW, MODE_SOFTMAX, MODE_SOFTMAX_RW,
                    attention_forward)
from oracle.lssar_backward import attention_backward

ALL_MODES = (MODE_SOFTMAX, MODE_LSSA, MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW)
RW_MODES = (MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW)
NORMALISED = (MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW)


def inputs(L, d, seed, lead=(2,)):
    rng = np.random.default_rng(seed)
    shape = lead + (L, d)
    return [rng.standard_normal(shape) for _ in range(4)]


def loss(q, k, v, dout, mode, p, **kw):
    return float(np.sum(dout * attention_forward(q, k, v, mode, p, **kw)))


def finite_differences(q, k, v, dout, mode, p, h=1e-6, **kw):
    grads = []
    args = [q, k, v]
    for which in range(3):
        g = np.zeros_like(args[which])
        for idx in np.ndindex(*args[which].shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += h
            minus[which][idx] -= h
            g[idx] = (loss(*plus, dout, mode, p, **kw) - loss(*minus, dout, mode, p, **kw)) / (2 * h)
        grads.append(g)
    return grads


@pytest.mark.parametrize("mode,p", [(MODE_SOFTMAX, 1), (MODE_LSSA, 1)]
                         + [(m, p) for m in RW_MODES for p in (1, 2, 3, 15)])
def test_backward_matches_finite_differences(mode, p):
    # rows 1-3 (O = 0) and 4-7 (O = 1) of two heads; d = 8
    q, k, v, dout = inputs(7, 8, seed=100 + 7 * mode + p)
    got = attention_backward(q, k, v, dout, mode, p)
    ref = finite_differences(q, k, v, dout, mode, p)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        scale = max(1.0, float(np.abs(r).max()))
        err = float(np.abs(g - r).max())
        assert err <= 2e-6 * scale, f"{name}: max err {err:.3e} (scale {scale:.3e})"


def test_backward_o_override_finite_differences():
    q, k, v, dout = inputs(6, 4, seed=5)
    got = attention_backward(q, k, v, dout, MODE_LSSAR, 3, o_override=0.0)
    ref = finite_differences(q, k, v, dout, MODE_LSSAR, 3, o_override=0.0)
    for g, r in zip(got, ref):
        assert np.abs(g - r).max() <= 2e-6 * max(1.0, np.abs(r).max())


def test_softmax_backward_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    q, k, v, dout = inputs(33, 16, seed=9, lead=(2, 3))
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    out = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    out.backward(torch.tensor(dout, dtype=torch.float64))
    got = attention_backward(q, k, v, dout, MODE_SOFTMAX)
    for g, t in zip(got, (tq.grad, tk.grad, tv.grad)):
        np.testing.assert_allclose(g, t.numpy(), rtol=1e-10, atol=1e-11)


def test_p1_o0_reweighting_backward_equals_lssa():
    # ReLU^1(i A - 0) normalised is A itself, so the gradients coincide
    q, k, v, dout = inputs(40, 8, seed=3)
    a = attention_backward(q, k, v, dout, MODE_LSSAR, 1, o_override=0.0)
    b = attention_backward(q, k, v, dout, MODE_LSSA)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("mode", ALL_MODES)
def test_dv_column_sum_is_dout_sum(mode):
    # every row of the attention matrix sums to one: sum_j dv_j = sum_i dout_i
    q, k, v, dout = inputs(50, 8, seed=11 + mode)
    _, _, dv = attention_backward(q, k, v, dout, mode, 15)
    np.testing.assert_allclose(dv.sum(axis=-2), dout.sum(axis=-2), rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("mode", NORMALISED)
def test_gradients_orthogonal_to_rows(mode):
    # out is unchanged by q_i -> c q_i and k_j -> c k_j (c > 0)
    q, k, v, dout = inputs(30, 8, seed=21 + mode)
    dq, dk, _ = attention_backward(q, k, v, dout, mode, 3)
    np.testing.assert_allclose(np.sum(dq * q, axis=-1), 0.0, atol=1e-11)
    np.testing.assert_allclose(np.sum(dk * k, axis=-1), 0.0, atol=1e-11)


@pytest.mark.parametrize("mode", ALL_MODES)
def test_constant_values_give_zero_score_gradients(mode):
    q, k, v, dout = inputs(20, 8, seed=31 + mode)
    v[...] = np.arange(8, dtype=np.float64)
    dq, dk, _ = attention_backward(q, k, v, dout, mode, 3)
    assert np.abs(dq).max() < 1e-11 and np.abs(dk).max() < 1e-11


def test_row_one_gradient():
    # out_1 = v_1 whatever q_1 is: dq_1 = 0 and dv_1 collects dout_1
    q, k, v, dout = inputs(5, 8, seed=41, lead=())
    for mode in ALL_MODES:
        dq, dk, dv = attention_backward(q, k, v, dout, mode, 3)
        assert np.abs(dq[0]).max() < 1e-12
        fd = finite_differences(q[None], k[None], v[None], dout[None], mode, 3)
        np.testing.assert_allclose(dv, fd[2][0], atol=1e-6)


@pytest.mark.parametrize("L,d", [(12, 8), (64, 16), (160, 64)])
def test_degenerate_rows_have_no_score_gradient(L, d):
    # identical keys: every LSSA row is uniform, so LSSAR rows 4.. are the
    # constant prefix mean (the 0/0 reading) and contribute nothing to dq.
    # At the two larger sizes float64 leaves residues of order 1e-16 in
    # i A - 1, which must not count as a nonzero re-weighting input.
    rng = np.random.default_rng(7 + L)
    q = rng.standard_normal((L, d))
    k = np.tile(rng.standard_normal((1, d)), (L, 1))
    v = rng.standard_normal((L, d))
    dout = rng.standard_normal((L, d))
    dq, _, dv = attention_backward(q, k, v, dout, MODE_LSSAR, 3)
    assert np.abs(dq[3:]).max() == 0.0
    # uniform rows: dv_j = sum_{i >= j} dout_i / i
    ref = np.array([sum(dout[i] / (i + 1) for i in range(j, L)) for j in range(L)])
    np.testing.assert_allclose(dv, ref, rtol=1e-12, atol=1e-12)
    mean = np.cumsum(v, axis=0) / np.arange(1, L + 1)[:, None]
    np.testing.assert_allclose(attention_forward(q, k, v, MODE_LSSAR, 3), mean, atol=1e-12)
