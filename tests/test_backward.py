"""GPU parity of the backward pass: gradients from the C ABI against the
float64 oracle's gradients on the same seeded bf16 inputs.

The training forward (lssar_attn_fwd_train) must give exactly the output of
lssar_attn_fwd and row statistics consistent with the oracle; the backward
(dq, dk, dv in bf16) must match the oracle's gradients element by element.

Tolerance, per gradient tensor, with TOL = 2e-2, or 5e-2 for p >= 15 in
the re-weighting modes (the forward's tolerance):
  elementwise   |got_ic - ref_ic| <= TOL (max_c' |ref_ic'| + 1e-2 G) + 2^-8 |ref_ic| + 1e-4
  aggregate     ||got - ref||_2 <= TOL ||ref||_2 + 1e-3 sqrt(n)
i.e. each element against its own row's largest gradient (a row's elements
are sums over the same weights and score gradients, and the kernel's errors
are relative to those), with a floor of 1 % of G, the largest entry of the
three gradients, for rows whose gradient cancels to near zero (a row of equal
keys has dq = 0 exactly, and the fp16 score gradients leave residues of about
2^-11 of their own size), plus 2^-8 for the bf16 rounding of
the result (1e-4: rounding residues where the exact gradient is 0).  Measured on this GPU, the largest error over all these cases is
0.017 of that scale (LSSAR p = 3: 0.014).  At p = 1 the re-weighting's ReLU has
a kink: a weight whose score lies within the score error of it may fall on
the other side, which moves that row by its whole contribution at the kink;
for p = 1 the elementwise bound is 3 TOL max |ref| (measured: 0.027 max |ref|).

Rows whose re-weighting is ill-conditioned at the precision of the fp16
score operands (well_conditioned_dout: a row's weights respond to a score
error with a gain of about p * kappa_i, and in a nearly uniform short row
that gain turns the fp16 rounding alone into a few per cent of its gradient)
get a zero upstream gradient on both sides.  The tests assert how many rows
that drops: at most 1 % of the rows (and one row in the smallest cases); the
seeded inputs here drop at most 2 rows of 256.
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


MAX_DROPPED = 0.01   # largest fraction of rows well_conditioned_dout may drop


def well_conditioned_dout(qb, kb, db, mode, p, limit=0.02):
    """Zero the upstream gradient of rows whose re-weighting is ill-conditioned
    at the precision of the fp16 normalised score operands, so that those
    rows drop out of every gradient (dq, dk and dv) on both sides.

    The score of q_i, k_j carries an fp16 rounding error of about
    2^-11 / sqrt(d), i.e. dx = ln d ln i 2^-11 / sqrt(d) in x.  The weight
    (y_ij)^p, y = i phi / S1 - O, then moves by the relative amount
    p (i phi'(x_ij) / S1_i) dx / y_ij; its average over the row's normalised
    weights R_ij is the row's expected relative error.  Rows where it exceeds
    `limit` are excluded.  Everything here comes from the oracle."""
    if mode not in (MODE_LSSAR, MODE_SIGMOID_RW):
        return db
    from oracle.lssar_oracle import bias_o, length_scale, l2_normalize_rows, sigmoid, softplus
    qf, kf = bf16_bits_to_f64(qb), bf16_bits_to_f64(kb)
    B, H, L, d = qf.shape
    rows = np.arange(1, L + 1)
    causal = rows[None, :] <= rows[:, None]
    dx = length_scale(rows, d) * 2.0 ** -11 / np.sqrt(d)
    out = db.copy()
    for b in range(B):
        for h in range(H):
            x = length_scale(rows, d)[:, None] * (l2_normalize_rows(qf[b, h]) @ l2_normalize_rows(kf[b, h]).T)
            sg = sigmoid(x)
            phi, slope = (sg, sg * (1.0 - sg)) if mode == MODE_SIGMOID_RW else (softplus(x), sg)
            phi, slope = phi * causal, slope * causal
            s1 = phi.sum(axis=1)
            y = np.maximum(rows[:, None] * phi / s1[:, None] - bias_o(rows)[:, None], 0.0)
            ymax = y.max(axis=1, keepdims=True)
            live = ymax[:, 0] > 0
            r = np.where(live[:, None], (y / np.where(live[:, None], ymax, 1.0)) ** p, 0.0)
            r /= np.maximum(r.sum(axis=1, keepdims=True), 1e-300)
            gain = np.where(y > 0, p * rows[:, None] * slope / s1[:, None] * dx[:, None] / np.maximum(y, 1e-300), 0.0)
            cond = (r * gain).sum(axis=1)
            out[b, h, cond > limit] = 0
    return out


def reference(qb, kb, vb, db, mode, p):
    return attention_backward(*(bf16_bits_to_f64(t) for t in (qb, kb, vb, db)), mode, p)


def run_backward(torch, B, H, L, d, mode, p, seed, impl="simt"):
    from lssar_attn_fwd_gb300 import api
    qb, kb, vb = make_qkv(B, H, L, d, seed=seed)
    d0 = make_dout(B, H, L, d, seed=seed)
    db = well_conditioned_dout(qb, kb, d0, mode, p)
    dropped = int((np.any(db != d0, axis=-1)).sum())
    rows = B * H * L
    print(f"well-conditioned rows: {rows - dropped} of {rows} kept (mode {mode}, p {p}, L {L}, d {d})")
    assert dropped <= max(1, MAX_DROPPED * rows), (dropped, rows)
    q, k, v, dout = (to_dev(torch, t) for t in (qb, kb, vb, db))
    out, stats = api.lssar_attn_fwd_train(q, k, v, p=p, mode=mode)
    fn = api.lssar_attn_bwd_simt if impl == "simt" else api.lssar_attn_bwd
    dq, dk, dv = fn(q, k, v, dout, stats, p=p, mode=mode)
    torch.cuda.synchronize()
    assert api.device_error_word() == 0
    got = tuple(to_np(t) for t in (dq, dk, dv))
    return got, reference(qb, kb, vb, db, mode, p)


def assert_close(got, ref, mode, p, what=""):
    t = tol(mode, p)
    kink = mode in RW_MODES and p == 1
    top_all = max(float(np.abs(r).max()) for r in ref)   # the problem's gradient scale
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        fro, nrm = float(np.linalg.norm(g - r)), float(np.linalg.norm(r))
        assert fro <= t * nrm + 1e-3 * np.sqrt(r.size), f"{what} {name}: ||err|| {fro:.3e} ||ref|| {nrm:.3e}"
        top = float(np.abs(r).max())
        if kink:
            bound = 3 * t * top + 1e-3 + 0.0 * r
        else:
            bound = t * (np.abs(r).max(axis=-1, keepdims=True) + 1e-2 * top_all) + 2.0 ** -8 * np.abs(r) + 1e-4
        excess = np.abs(g - r) - bound
        assert excess.max() <= 0.0, (f"{what} {name}: |err| {np.abs(g - r).flat[excess.argmax()]:.3e} "
                                     f"over the bound {bound.flat[excess.argmax()]:.3e}")


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
    ref = reference(qb, kb, vb, db, MODE_LSSAR, 3)
    assert np.abs(to_np(dq)[0, 0, 3:]).max() == 0.0
    assert_close((to_np(dq), to_np(dk), to_np(dv)), ref, MODE_LSSAR, 3)


# ---------------------------------------------------------------- tensor-core backward

@pytest.mark.parametrize("mode,p", MODES)
@pytest.mark.parametrize("d", [64, 128])
def test_backward_tc_parity(torch_mod, mode, p, d):
    # three 128-row tiles with a ragged tail
    got, ref = run_backward(torch_mod, 1, 2, 300, d, mode, p, seed=d + 10 * mode + p, impl="tc")
    assert_close(got, ref, mode, p, f"d={d}")


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 127, 128, 129, 257])
@pytest.mark.parametrize("d", [64, 128])
def test_backward_tc_lengths(torch_mod, L, d):
    for mode, p in [(MODE_LSSAR, 3), (MODE_LSSAR, 15), (MODE_SOFTMAX, 1), (MODE_LSSA, 1),
                    (MODE_SIGMOID_RW, 15), (MODE_SOFTMAX_RW, 2)]:
        got, ref = run_backward(torch_mod, 2, 1, L, d, mode, p, seed=L + d, impl="tc")
        assert_close(got, ref, mode, p, f"L={L} d={d} mode={mode} p={p}")


def test_backward_tc_many_items(torch_mod):
    # more work items (B*H*tiles = 480) than SMs: the dynamic schedule of both
    # passes; every element against the CUDA-core backward, two heads against
    # the oracle
    from lssar_attn_fwd_gb300 import api
    torch = torch_mod
    B, H, L, d, p = 2, 80, 300, 64, 15
    qb, kb, vb = make_qkv(B, H, L, d, seed=77)
    db = make_dout(B, H, L, d, seed=77)
    q, k, v, dout = (to_dev(torch, t) for t in (qb, kb, vb, db))
    _, stats = api.lssar_attn_fwd_train(q, k, v, p=p, mode=MODE_LSSAR)
    tc = api.lssar_attn_bwd(q, k, v, dout, stats, p=p, mode=MODE_LSSAR)
    si = api.lssar_attn_bwd_simt(q, k, v, dout, stats, p=p, mode=MODE_LSSAR)
    torch.cuda.synchronize()
    assert api.device_error_word() == 0
    for a, b in zip(tc, si):
        a, b = to_np(a), to_np(b)
        assert np.abs(a - b).max() <= 2e-2 * np.abs(b).max()
    for bb, hh in ((0, 0), (1, 79)):
        ref = reference(*(t[bb:bb + 1, hh:hh + 1] for t in (qb, kb, vb, db)), MODE_LSSAR, p)
        assert_close(tuple(to_np(t)[bb:bb + 1, hh:hh + 1] for t in tc), ref, MODE_LSSAR, p)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_tc_long_vs_simt(torch_mod, d):
    # nine key tiles and a ragged tail, every element against the CUDA-core path
    from lssar_attn_fwd_gb300 import api
    torch = torch_mod
    B, H, L = 1, 3, 1100
    for mode, p in [(MODE_LSSAR, 15), (MODE_SOFTMAX, 1), (MODE_SOFTMAX_RW, 3)]:
        qb, kb, vb = make_qkv(B, H, L, d, seed=d + mode)
        db = make_dout(B, H, L, d, seed=d + mode)
        q, k, v, dout = (to_dev(torch, t) for t in (qb, kb, vb, db))
        _, stats = api.lssar_attn_fwd_train(q, k, v, p=p, mode=mode)
        tc = api.lssar_attn_bwd(q, k, v, dout, stats, p=p, mode=mode)
        si = api.lssar_attn_bwd_simt(q, k, v, dout, stats, p=p, mode=mode)
        torch.cuda.synchronize()
        assert api.device_error_word() == 0
        for name, a, b in zip(("dq", "dk", "dv"), tc, si):
            a, b = to_np(a), to_np(b)
            assert np.abs(a - b).max() <= tol(mode, p) * np.abs(b).max(), (mode, name)


def test_backward_tc_uniform_rows(torch_mod):
    from lssar_attn_fwd_gb300 import api
    torch = torch_mod
    B, H, L, d = 1, 1, 300, 64
    qb, kb, vb = make_qkv(B, H, L, d, seed=3)
    kb = np.broadcast_to(kb[:, :, :1], kb.shape).copy()
    db = make_dout(B, H, L, d, seed=3)
    q, k, v, dout = (to_dev(torch, t) for t in (qb, kb, vb, db))
    _, stats = api.lssar_attn_fwd_train(q, k, v, p=15, mode=MODE_LSSAR)
    dq, dk, dv = api.lssar_attn_bwd(q, k, v, dout, stats, p=15, mode=MODE_LSSAR)
    torch.cuda.synchronize()
    assert api.device_error_word() == 0
    ref = reference(qb, kb, vb, db, MODE_LSSAR, 15)
    assert np.abs(to_np(dq)[0, 0, 3:]).max() == 0.0
    assert_close((to_np(dq), to_np(dk), to_np(dv)), ref, MODE_LSSAR, 15)


@pytest.mark.parametrize("mode", [MODE_LSSAR, MODE_SIGMOID_RW, MODE_SOFTMAX_RW])
@pytest.mark.parametrize("d", [64, 128])
def test_backward_tc_per_head_exponents(torch_mod, mode, d):
    # one exponent per head through the training forward and the backward:
    # every head's output and gradients against the oracle at its own p
    from lssar_attn_fwd_gb300 import api
    torch = torch_mod
    ps = [1, 3, 15, 7]
    B, H, L = 2, len(ps), 300
    qb, kb, vb = make_qkv(B, H, L, d, seed=21 + d + mode)
    d0 = make_dout(B, H, L, d, seed=21 + d + mode)
    db = d0.copy()
    for h, p in enumerate(ps):   # the well-conditioned rows of each head at its own p
        db[:, h:h + 1] = well_conditioned_dout(qb[:, h:h + 1], kb[:, h:h + 1], d0[:, h:h + 1], mode, p)
    dropped = int(np.any(db != d0, axis=-1).sum())
    assert dropped <= max(1, MAX_DROPPED * B * H * L), dropped
    q, k, v, dout = (to_dev(torch, t) for t in (qb, kb, vb, db))
    out, stats = api.lssar_attn_fwd_train_heads_p(q, k, v, ps, mode=mode)
    ref_out = api.lssar_attn_fwd_heads_p(q, k, v, ps, mode=mode)
    dq, dk, dv = api.lssar_attn_bwd_heads_p(q, k, v, dout, stats, ps, mode=mode)
    torch.cuda.synchronize()
    assert api.device_error_word() == 0
    assert torch.equal(out, ref_out)          # same kernel, same arithmetic as the inference entry
    got = tuple(to_np(t) for t in (dq, dk, dv))
    o = to_np(out)
    for h, p in enumerate(ps):
        sl = lambda t: t[:, h:h + 1]   # noqa: E731
        fwd = attention_forward(*(bf16_bits_to_f64(sl(t)) for t in (qb, kb, vb)), mode, p)
        assert np.abs(sl(o) - fwd).max() <= tol(mode, p), (h, p)
        ref = reference(*(sl(t) for t in (qb, kb, vb, db)), mode, p)
        assert_close(tuple(sl(g) for g in got), ref, mode, p, f"head {h} p={p}")


@pytest.mark.parametrize("p", [15, 40])
def test_backward_tc_one_exponential_weights(torch_mod, p, monkeypatch):
    # The row pass takes the forward's one-exponential weights (softplus as
    # z + 2^-|z| / ln 2) on warps (32 query rows) whose rows all meet the error
    # bound at p and at p - 1; LSSAR_EXACT_WEIGHTS=1 keeps log2(1 + 2^z)
    # everywhere.  With the same row statistics the two backward results are
    # bit-identical on every warp that the bound rejects, differ somewhere on
    # the admitted warps (a change of about 1e-6 of a weight flips the bf16
    # rounding of few dq elements), and both match the oracle's gradients
    # element by element.  The bound is recomputed here in float64 from the
    # saved statistics (theta = -beta / kappa), with a margin of 2x either
    # way around the kernel's float32 decision.  p = 40: generic power path.
    from test_fast_weights import FAST_BOUND, admitted
    from lssar_attn_fwd_gb300 import api
    torch = torch_mod
    B, H, L, d = 1, 2, 2048, 64
    qb, kb, vb = make_qkv(B, H, L, d, seed=31 + p)
    d0 = make_dout(B, H, L, d, seed=31 + p)
    db = well_conditioned_dout(qb, kb, d0, MODE_LSSAR, p)
    dropped = int(np.any(db != d0, axis=-1).sum())
    assert dropped <= max(1, MAX_DROPPED * B * H * L), dropped
    q, k, v, dout = (to_dev(torch, t) for t in (qb, kb, vb, db))
    monkeypatch.delenv("LSSAR_EXACT_WEIGHTS", raising=False)
    _, stats = api.lssar_attn_fwd_train(q, k, v, p=p, mode=MODE_LSSAR)
    fast = api.lssar_attn_bwd(q, k, v, dout, stats, p=p, mode=MODE_LSSAR)
    monkeypatch.setenv("LSSAR_EXACT_WEIGHTS", "1")
    exact = api.lssar_attn_bwd(q, k, v, dout, stats, p=p, mode=MODE_LSSAR)
    monkeypatch.delenv("LSSAR_EXACT_WEIGHTS")
    torch.cuda.synchronize()
    assert api.device_error_word() == 0
    got_f, got_e = tuple(to_np(t) for t in fast), tuple(to_np(t) for t in exact)
    st = stats.cpu().numpy().astype(np.float64)
    kap, bet = st[..., 1], st[..., 2]
    live = kap > 0
    theta = np.where(live, -bet / np.where(live, kap, 1.0), 0.0)
    i = np.arange(1, L + 1, dtype=np.float64)
    _, b_p = admitted(theta, np.where(live, kap, 1.0), i, p)
    _, b_q = admitted(theta, np.where(live, kap, 1.0), i, p - 1)
    bound = np.maximum(b_p, b_q)
    sure_out = ~live | (theta < 1.49) | (bound > 2.0 * FAST_BOUND)
    sure_in = live & (theta > 1.51) & (bound < 0.5 * FAST_BOUND)
    warp_out = np.repeat(sure_out.reshape(B, H, L // 32, 32).any(-1), 32, axis=-1)
    warp_in = np.repeat(sure_in.reshape(B, H, L // 32, 32).all(-1), 32, axis=-1)
    warp_in[..., :128] = False     # the first tile has only its diagonal tile: exact weights
    moved = np.any(got_f[0] != got_e[0], axis=-1)
    print(f"p {p}: warps admitted {warp_in.mean():.3f}, rejected {warp_out.mean():.3f}; "
          f"dq rows moved {moved.mean():.4f} (admitted warps: {moved[warp_in].mean():.4f})")
    assert warp_in.mean() > 0.3 and warp_out.mean() > 0.05
    assert not moved[warp_out].any()
    assert moved[warp_in].any()
    ref = reference(qb, kb, vb, db, MODE_LSSAR, p)
    assert_close(got_f, ref, MODE_LSSAR, p, "one-exponential")
    assert_close(got_e, ref, MODE_LSSAR, p, "exact")


@pytest.mark.parametrize("mode,p", [(MODE_LSSAR, 3), (MODE_LSSAR, 15), (MODE_SOFTMAX, 1), (MODE_SIGMOID_RW, 3)])
def test_backward_tc_zero_rows(torch_mod, mode, p):
    # All-zero query and key rows: the L2 normalisation max(|x|, 1e-12) takes
    # its floor there (zero scores: the query row is uniform, in LSSAR the
    # 0/0 prefix-mean row of the notes' re-weighting), and the fused
    # normalisation gradient of both passes takes its |x| <= 1e-12 branch.
    # In the normalised modes a zero key row's dk is its gradient with respect
    # to the normalised row times 1e12: those rows are checked against the
    # oracle each on its own scale, every other element with the usual bar.
    from lssar_attn_fwd_gb300 import api
    torch = torch_mod
    B, H, L, d = 1, 2, 300, 64
    zq, zk = [4, 76, 199], [9, 149]
    qb, kb, vb = make_qkv(B, H, L, d, seed=41 + mode)
    qb[:, :, zq] = 0           # bf16 +0.0 is the all-zero bit pattern
    kb[:, :, zk] = 0
    d0 = make_dout(B, H, L, d, seed=41 + mode)
    db = well_conditioned_dout(qb, kb, d0, mode, p)
    dropped = int(np.any(db != d0, axis=-1).sum())
    assert dropped <= max(1, MAX_DROPPED * B * H * L), dropped
    q, k, v, dout = (to_dev(torch, t) for t in (qb, kb, vb, db))
    out, stats = api.lssar_attn_fwd_train(q, k, v, p=p, mode=mode)
    grads = api.lssar_attn_bwd(q, k, v, dout, stats, p=p, mode=mode)
    torch.cuda.synchronize()
    assert api.device_error_word() == 0
    ref_out = attention_forward(*(bf16_bits_to_f64(t) for t in (qb, kb, vb)), mode, p)
    assert np.abs(to_np(out) - ref_out).max() <= tol(mode, p)
    got = [to_np(t) for t in grads]
    ref = list(reference(qb, kb, vb, db, mode, p))
    assert all(np.isfinite(g).all() for g in got)
    t = tol(mode, p)
    g_rows, r_rows = got[1][:, :, zk], ref[1][:, :, zk]
    scale = np.abs(r_rows).max(axis=-1, keepdims=True)
    assert (np.abs(g_rows - r_rows) <= t * scale + 2.0 ** -8 * np.abs(r_rows)).all()
    got[1][:, :, zk] = 0.0
    ref[1][:, :, zk] = 0.0
    if mode != MODE_SOFTMAX:
        # a zero query row reads as uniform (LSSA) or as the 0/0 row (LSSAR,
        # sigmoid re-weighting): its scores get no gradient, so neither does q
        assert np.abs(got[0][:, :, zq]).max() == 0.0
    assert_close(tuple(got), tuple(ref), mode, p, "zero rows")
