"""GPU parity of the backward pass: gradients from the C ABI against the
float64 oracle's gradients on the same seeded bf16 inputs.

The training forward (lssar_attn_fwd_train) must give exactly the output of
lssar_attn_fwd and row statistics consistent with the oracle; the backward
(dq, dk, dv in bf16) must match the oracle's gradients element by element.

Tolerance: max abs error of each gradient tensor <= TOL * max|oracle gradient|
(+ a floor of 1e-3 for near-zero tensors).  The gradients go through the same
exponent p as the forward, so the score error of the forward's row constants
(fp16 normalised q, k in the score product) is amplified like the forward's
output error; the bf16 rounding of the gradients adds 2^-9 relative.
"""

import numpy as np
import pytest

from lssar_attn_fwd_gb300.inputs import (
    MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW, MODE_SOFTMAX, MODE_SOFTMAX_RW, bf16_bits_to_f64,
    make_dout, make_qkv)
from oracle import attention_forward
from oracle.lssar_backward import attention_backward

pytestmark = pytest.mark.gpu

RW_MODES = (MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW)


def tol(mode, p):
    return 5e-2 if (mode in RW_MODES and p >= 15) else 2e-2


@pytest.fixture(scope="module")
def torch_mod():
    import torch
    from lssar_attn_fwd_gb300 import api, build
    build.build()
    api.load_library()
    return torch


def to_dev(torch, bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def to_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_backward(torch, B, H, L, d, mode, p, seed, impl="simt"):
    from lssar_attn_fwd_gb300 import api
    qb, kb, vb = make_qkv(B, H, L, d, seed=seed)
    db = make_dout(B, H, L, d, seed=seed)
    q, k, v, dout = (to_dev(torch, t) for t in (qb, kb, vb, db))
    out, stats = api.lssar_attn_fwd_train(q, k, v, p=p, mode=mode)
    fn = api.lssar_attn_bwd_simt if impl == "simt" else api.lssar_attn_bwd
    dq, dk, dv = fn(q, k, v, dout, stats, p=p, mode=mode)
    torch.cuda.synchronize()
    assert api.device_error_word() == 0
    got = tuple(to_np(t) for t in (dq, dk, dv))
    ref = attention_backward(*(bf16_bits_to_f64(t) for t in (qb, kb, vb, db)), mode, p)
    return got, ref


def assert_close(got, ref, mode, p, what=""):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        scale = float(np.abs(r).max())
        err = float(np.abs(g - r).max())
        assert err <= tol(mode, p) * scale + 1e-3, f"{what} {name}: err {err:.3e} scale {scale:.3e}"


MODES = [(MODE_LSSAR, 3), (MODE_LSSAR, 15), (MODE_LSSAR, 1), (MODE_LSSA, 1), (MODE_SOFTMAX, 1),
         (MODE_SOFTMAX_RW, 3), (MODE_SOFTMAX_RW, 15), (MODE_SIGMOID_RW, 3), (MODE_SIGMOID_RW, 15)]


@pytest.mark.parametrize("mode,p", MODES)
def test_train_forward_output_and_stats(torch_mod, mode, p):
    from lssar_attn_fwd_gb300 import api
    torch = torch_mod
    B, H, L, d = 1, 2, 300, 64
    qb, kb, vb = make_qkv(B, H, L, d, seed=5)
    q, k, v = (to_dev(torch, t) for t in (qb, kb, vb))
    ref_out = api.lssar_attn_fwd(q, k, v, p=p, mode=mode)
    out, stats = api.lssar_attn_fwd_train(q, k, v, p=p, mode=mode)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)          # same kernel, same arithmetic
    st = stats.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(st))
    if mode != MODE_LSSA:
        assert np.all(st[..., 3] >= 1.0 - 1e-3)   # the row maximum has weight 1
    if mode in (MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW):
        # W = sum_j ((y_j / max y)^p) of the oracle's re-weighting, row by row
        from oracle.lssar_oracle import bias_o, lssa_rows, sigmoid, softmax_rows
        qf, kf = bf16_bits_to_f64(qb)[0, 0], bf16_bits_to_f64(kb)[0, 0]
        rows = np.arange(1, L + 1)
        if mode == MODE_SOFTMAX_RW:
            a = softmax_rows(qf, kf, rows, d)
        else:
            a = lssa_rows(qf, kf, rows, d, phi=sigmoid if mode == MODE_SIGMOID_RW else None)
        y = np.maximum(rows[:, None] * a - bias_o(rows)[:, None], 0.0)
        W = ((y / y.max(axis=1, keepdims=True)) ** p).sum(axis=1)
        np.testing.assert_allclose(st[0, 0, :, 3], W, rtol=5e-2 if p >= 15 else 1e-2)


@pytest.mark.parametrize("mode,p", MODES)
@pytest.mark.parametrize("d", [64, 128])
def test_backward_simt_parity(torch_mod, mode, p, d):
    got, ref = run_backward(torch_mod, 1, 2, 200, d, mode, p, seed=d + 10 * mode + p)
    assert_close(got, ref, mode, p, f"d={d}")


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 129])
def test_backward_simt_short_rows(torch_mod, L):
    for mode, p in [(MODE_LSSAR, 3), (MODE_SOFTMAX, 1), (MODE_SIGMOID_RW, 15)]:
        got, ref = run_backward(torch_mod, 2, 1, L, 64, mode, p, seed=L)
        assert_close(got, ref, mode, p, f"L={L}")


def test_backward_simt_uniform_rows(torch_mod):
    # identical keys: LSSAR rows >= 4 are the uniform prefix mean and pass no
    # gradient to q (the oracle's reading of the 0/0 row)
    from lssar_attn_fwd_gb300 import api
    torch = torch_mod
    B, H, L, d = 1, 1, 160, 64
    qb, kb, vb = make_qkv(B, H, L, d, seed=3)
    kb = np.broadcast_to(kb[:, :, :1], kb.shape).copy()
    db = make_dout(B, H, L, d, seed=3)
    q, k, v, dout = (to_dev(torch, t) for t in (qb, kb, vb, db))
    out, stats = api.lssar_attn_fwd_train(q, k, v, p=3, mode=MODE_LSSAR)
    dq, dk, dv = api.lssar_attn_bwd_simt(q, k, v, dout, stats, p=3, mode=MODE_LSSAR)
    torch.cuda.synchronize()
    st = stats.cpu().numpy()
    assert np.all(st[0, 0, 3:, 1] == 0.0) and np.all(st[0, 0, 3:, 2] == 1.0)
    np.testing.assert_array_equal(st[0, 0, 3:, 3], np.arange(4, L + 1, dtype=np.float32))
    ref = attention_backward(*(bf16_bits_to_f64(t) for t in (qb, kb, vb, db)), MODE_LSSAR, 3)
    assert np.abs(to_np(dq)[0, 0, 3:]).max() == 0.0
    assert_close((to_np(dq), to_np(dk), to_np(dv)), ref, MODE_LSSAR, 3)
