"""GPU parity: the tensor-core kernel (through the C ABI) against the float64
oracle on the same seeded bf16 inputs.

Tolerance (max abs error of the bf16 output against the float64 oracle):
2e-2 for LSSA, softmax and LSSAR with p <= 3; 5e-2 for p >= 15.  The
budget is dominated by the bf16 rounding of the output (up to 1.6e-2 for
|out| in [4, 8)), bf16 rounding of the weights fed to the tensor core, and
fp16 rounding of the normalised q, k in the score product.
"""

import numpy as np
import pytest

from lssar_attn_fwd_gb300.inputs import (
    MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW, MODE_SOFTMAX, MODE_SOFTMAX_RW, WORKLOADS,
    bf16_bits_to_f64, make_qkv, needle_targets)
from oracle import attention_forward

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


def run(torch, qb, kb, vb, p, mode, impl="tc"):
    from lssar_attn_fwd_gb300 import api
    q, k, v = (to_dev(torch, t) for t in (qb, kb, vb))
    fn = api.lssar_attn_fwd if impl == "tc" else api.lssar_attn_fwd_simt
    out = fn(q, k, v, p=p, mode=mode)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def check_error_word():
    from lssar_attn_fwd_gb300 import api
    assert api.device_error_word() == 0


MODES = [(MODE_LSSAR, 3), (MODE_LSSAR, 15), (MODE_LSSAR, 1), (MODE_LSSAR, 2), (MODE_LSSAR, 7),
         (MODE_LSSA, 1), (MODE_SOFTMAX, 1), (MODE_SOFTMAX_RW, 3), (MODE_SOFTMAX_RW, 15),
         (MODE_SOFTMAX_RW, 1), (MODE_SIGMOID_RW, 3), (MODE_SIGMOID_RW, 15), (MODE_SIGMOID_RW, 2)]


@pytest.mark.parametrize("mode,p", MODES)
def test_tiny_all_modes(torch_mod, mode, p):
    w = WORKLOADS["tiny"]
    qb, kb, vb = make_qkv(*w.shape, seed=0)
    got = run(torch_mod, qb, kb, vb, p, mode)
    ref = attention_forward(*(bf16_bits_to_f64(t) for t in (qb, kb, vb)), mode, p)
    err = np.abs(got - ref).max()
    assert err <= tol(mode, p), err
    check_error_word()


@pytest.mark.parametrize("L", [1, 2, 3, 5, 127, 129, 200, 255, 256, 257, 300, 513])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_lengths(torch_mod, L, d):
    qb, kb, vb = make_qkv(2, 2, L, d, seed=L + d)
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    for mode, p in [(MODE_LSSAR, 3), (MODE_LSSAR, 15), (MODE_LSSA, 1), (MODE_SOFTMAX, 1),
                    (MODE_SOFTMAX_RW, 15), (MODE_SIGMOID_RW, 3)]:
        got = run(torch_mod, qb, kb, vb, p, mode)
        ref = attention_forward(qf, kf, vf, mode, p)
        err = np.abs(got - ref).max()
        assert err <= tol(mode, p), (mode, p, err)
    check_error_word()


@pytest.mark.parametrize("d", [64, 128])
def test_multi_pair_full_check(torch_mod, d):
    # several Q-tile pairs per head, a ragged tail, more items than SMs
    B, H, L = 3, 60, 700
    qb, kb, vb = make_qkv(B, H, L, d, seed=d)
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    heads = [(0, 0), (1, 17), (2, 59)]
    for mode, p in [(MODE_LSSAR, 3), (MODE_LSSAR, 15), (MODE_SOFTMAX, 1), (MODE_LSSA, 1),
                    (MODE_SOFTMAX_RW, 3), (MODE_SIGMOID_RW, 15)]:
        got = run(torch_mod, qb, kb, vb, p, mode)
        for b, h in heads:
            ref = attention_forward(qf[b, h], kf[b, h], vf[b, h], mode, p)
            err = np.abs(got[b, h] - ref).max()
            assert err <= tol(mode, p), (mode, p, b, h, err)
    check_error_word()


def sample_rows(L, seed):
    rng = np.random.default_rng(seed)
    fixed = [1, 2, 3, 4, 5, 127, 128, 129, 256, 257, L // 2, L - 1, L]
    return np.unique(np.clip(np.concatenate([fixed, rng.integers(1, L + 1, 24)]), 1, L))


@pytest.mark.parametrize("name", ["gpt2", "extrap", "needle", "wide"])
def test_full_size_sampled_rows(torch_mod, name):
    w = WORKLOADS[name]
    qb, kb, vb = make_qkv(*w.shape, seed=0, structure=w.structure)
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    rows = sample_rows(w.L, seed=1)
    heads = [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 2)]
    for mode, p in w.runs:
        got = run(torch_mod, qb, kb, vb, p, mode)
        assert np.isfinite(got).all()
        for b, h in heads:
            ref = attention_forward(qf[b, h], kf[b, h], vf[b, h], mode, p, rows=rows)
            err = np.abs(got[b, h, rows - 1] - ref).max()
            assert err <= tol(mode, p), (name, mode, p, b, h, err)
    check_error_word()


def test_rows_sum_to_one_full_size(torch_mod):
    # V = ones: every mode ends in an L1 normalisation, so out == 1.
    w = WORKLOADS["extrap"]
    qb, kb, _ = make_qkv(*w.shape, seed=2)
    ones = np.full(w.shape, 0x3F80, dtype=np.uint16)   # bf16 1.0
    for mode, p in [(MODE_LSSAR, 15), (MODE_LSSAR, 3), (MODE_LSSA, 1), (MODE_SOFTMAX, 1),
                    (MODE_SOFTMAX_RW, 15), (MODE_SIGMOID_RW, 15)]:
        got = run(torch_mod, qb, kb, ones, p, mode)
        assert np.abs(got - 1.0).max() <= 1e-2, mode


def test_first_row_is_first_value(torch_mod):
    qb, kb, vb = make_qkv(2, 3, 384, 64, seed=5)
    vf = bf16_bits_to_f64(vb)
    for mode, p in [(MODE_LSSAR, 15), (MODE_LSSA, 1), (MODE_SOFTMAX, 1), (MODE_SOFTMAX_RW, 15),
                    (MODE_SIGMOID_RW, 3)]:
        got = run(torch_mod, qb, kb, vb, p, mode)
        np.testing.assert_array_equal(got[:, :, 0], vf[:, :, 0])


def test_identical_keys_give_prefix_mean(torch_mod):
    # Uniform scores: LSSA weights 1/i; LSSAR rows from 4 on are all-zero
    # (0/0) re-weighted rows, read as the uniform prefix mean.
    B, H, L, d = 1, 2, 600, 64
    qb, kb, vb = make_qkv(B, H, L, d, seed=6)
    kb = np.broadcast_to(kb[:, :, :1], kb.shape).copy()
    vf = bf16_bits_to_f64(vb)
    mean = np.cumsum(vf, axis=2) / np.arange(1, L + 1)[None, None, :, None]
    for mode, p in [(MODE_LSSA, 1), (MODE_LSSAR, 3), (MODE_LSSAR, 15), (MODE_SOFTMAX_RW, 15),
                    (MODE_SIGMOID_RW, 15)]:
        got = run(torch_mod, qb, kb, vb, p, mode)
        assert np.abs(got - mean).max() <= 2e-2, mode


def test_needle_large_p_is_argmax(torch_mod):
    # p = 64 (generic power path): the weight concentrates on the needle key.
    B, H, L, d = 1, 2, 1024, 64
    qb, kb, vb = make_qkv(B, H, L, d, seed=3, structure="needle")
    j = needle_targets(B, H, L, d, seed=3)
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    got = run(torch_mod, qb, kb, vb, 64, MODE_LSSAR)
    rows = sample_rows(L, seed=4)
    for h in range(H):
        ref = attention_forward(qf[0, h], kf[0, h], vf[0, h], MODE_LSSAR, 64, rows=rows)
        assert np.abs(got[0, h, rows - 1] - ref).max() <= 5e-2
    picked = np.take_along_axis(vf, (j - 1)[..., None].repeat(d, -1), axis=2)
    close = np.abs(got - picked).max(axis=-1) < 5e-2
    assert close[:, :, 64:].mean() > 0.95


@pytest.mark.parametrize("p", [200, 1024])
def test_largest_exponents(torch_mod, p):
    # up to the largest exponent the C ABI accepts (generic power path): on
    # the needle structure (one key clearly above the rest) the re-weighted
    # rows are well conditioned, and every sampled row must match the oracle;
    # the decode step must match the oracle's last row
    from lssar_attn_fwd_gb300 import api
    torch = torch_mod
    B, H, L, d = 1, 2, 1024, 64
    qb, kb, vb = make_qkv(B, H, L, d, seed=5, structure="needle")
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    got = run(torch, qb, kb, vb, p, MODE_LSSAR)
    rows = np.unique(np.concatenate([np.arange(1, 9), sample_rows(L, seed=6)]))
    q_last = to_dev(torch, np.ascontiguousarray(qb[:, :, -1]))
    dec = api.lssar_attn_decode(q_last, to_dev(torch, kb), to_dev(torch, vb), p=p, mode=MODE_LSSAR)
    torch.cuda.synchronize()
    dec = dec.float().cpu().numpy().astype(np.float64)
    for h in range(H):
        ref = attention_forward(qf[0, h], kf[0, h], vf[0, h], MODE_LSSAR, p, rows=rows)
        assert np.abs(got[0, h, rows - 1] - ref).max() <= tol(MODE_LSSAR, p), (p, h)
        assert np.abs(dec[0, h] - ref[-1]).max() <= tol(MODE_LSSAR, p), (p, h)
    check_error_word()


def test_tc_matches_simt_full_size(torch_mod):
    # Consistency between the two GPU implementations on every row (an extra
    # check beside the oracle parity above).
    w = WORKLOADS["gpt2"]
    qb, kb, vb = make_qkv(*w.shape, seed=7)
    for mode, p in w.runs:
        a = run(torch_mod, qb, kb, vb, p, mode, "tc")
        b = run(torch_mod, qb, kb, vb, p, mode, "simt")
        assert np.abs(a - b).max() <= 2 * tol(mode, p)


@pytest.mark.parametrize("name", ["extrap", "wide"])
def test_ablation_modes_full_size_sampled_rows(torch_mod, name):
    # The two ablation normalisers (notes' ablation table) at full size.
    w = WORKLOADS[name]
    qb, kb, vb = make_qkv(*w.shape, seed=10)
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    rows = sample_rows(w.L, seed=11)
    for mode in (MODE_SOFTMAX_RW, MODE_SIGMOID_RW):
        got = run(torch_mod, qb, kb, vb, 15, mode)
        assert np.isfinite(got).all()
        for b, h in [(0, 0), (w.B - 1, w.H - 1)]:
            ref = attention_forward(qf[b, h], kf[b, h], vf[b, h], mode, 15, rows=rows)
            err = np.abs(got[b, h, rows - 1] - ref).max()
            assert err <= tol(mode, 15), (name, mode, b, h, err)
    check_error_word()


@pytest.mark.parametrize("mode", [MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW])
@pytest.mark.parametrize("d", [64, 128])
def test_per_head_exponents(torch_mod, mode, d):
    # lssar_attn_fwd_heads_p: head h uses its own p; each head must match the
    # oracle at that p.
    torch = torch_mod
    from lssar_attn_fwd_gb300 import api
    B, H, L = 2, 5, 300
    ps = [1, 3, 15, 40, 2]
    qb, kb, vb = make_qkv(B, H, L, d, seed=12)
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    q, k, v = (to_dev(torch, t) for t in (qb, kb, vb))
    got = api.lssar_attn_fwd_heads_p(q, k, v, ps, mode=mode)
    torch.cuda.synchronize()
    got = got.float().cpu().numpy().astype(np.float64)
    for b in range(B):
        for h in range(H):
            ref = attention_forward(qf[b, h], kf[b, h], vf[b, h], mode, ps[h])
            err = np.abs(got[b, h] - ref).max()
            assert err <= tol(mode, ps[h]), (mode, d, b, h, ps[h], err)
    check_error_word()


def test_simt_matches_oracle(torch_mod):
    qb, kb, vb = make_qkv(1, 2, 300, 128, seed=8)
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    for mode, p in [(MODE_LSSAR, 3), (MODE_LSSAR, 15), (MODE_LSSA, 1), (MODE_SOFTMAX, 1),
                    (MODE_SOFTMAX_RW, 15), (MODE_SIGMOID_RW, 15)]:
        got = run(torch_mod, qb, kb, vb, p, mode, "simt")
        ref = attention_forward(qf, kf, vf, mode, p)
        assert np.abs(got - ref).max() <= tol(mode, p)


def test_nonzero_stream_and_preallocated_out(torch_mod):
    torch = torch_mod
    from lssar_attn_fwd_gb300 import api
    qb, kb, vb = make_qkv(1, 2, 256, 64, seed=9)
    q, k, v = (to_dev(torch, t) for t in (qb, kb, vb))
    out = torch.full_like(q, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        api.lssar_attn_fwd(q, k, v, p=3, mode=MODE_LSSAR, out=out)
    s.synchronize()
    ref = attention_forward(*(bf16_bits_to_f64(t) for t in (qb, kb, vb)), MODE_LSSAR, 3)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= 2e-2


def bf16_ulp(x):
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


@pytest.mark.parametrize("structure,p,min_moved,d", [("iid", 15, 0.5, 64), ("needle", 15, 0.0, 64),
                                                     ("iid", 64, 0.2, 64), ("iid", 15, 0.5, 128)])
def test_one_exponential_weights(torch_mod, structure, p, min_moved, d, monkeypatch):
    # LSSAR rows whose error bound holds take z + 2^-|z|/ln 2 for the softplus
    # in the weight pass; LSSAR_EXACT_WEIGHTS=1 keeps log2(1 + 2^z) on every row.
    # The row sums W = sum_j w_j saved by the training forward show which rows
    # took the one-exponential weights (W differs in its low bits) and bound
    # the change (at most 2e-4 of W); the outputs agree to within one bf16
    # rounding step, and both match the oracle on sampled rows.
    from lssar_attn_fwd_gb300 import api
    torch = torch_mod
    B, H, L = 1, 2, 8192
    qb, kb, vb = make_qkv(B, H, L, d, seed=5, structure=structure)
    q, k, v = (to_dev(torch, t) for t in (qb, kb, vb))
    monkeypatch.delenv("LSSAR_EXACT_WEIGHTS", raising=False)
    out_f, st_f = api.lssar_attn_fwd_train(q, k, v, p=p, mode=MODE_LSSAR)
    monkeypatch.setenv("LSSAR_EXACT_WEIGHTS", "1")
    out_e, st_e = api.lssar_attn_fwd_train(q, k, v, p=p, mode=MODE_LSSAR)
    monkeypatch.delenv("LSSAR_EXACT_WEIGHTS")
    torch.cuda.synchronize()
    of, oe = (t.float().cpu().numpy().astype(np.float64) for t in (out_f, out_e))
    wf, we = (t.cpu().numpy()[..., 3].astype(np.float64) for t in (st_f, st_e))
    # a row's weight sum moves by at most 2e-4 of itself, so its output by at
    # most 2 * 2e-4 * max|v|; a weight that crosses a rounding boundary of the
    # bf16 P fed to the tensor core moves by one bf16 step (2^-8 of itself,
    # at most 2^-8 max|v| on the output); then one bf16 rounding of the output
    vmax = np.abs(bf16_bits_to_f64(vb)).max()
    diff = np.abs(of - oe) - bf16_ulp(np.maximum(np.abs(of), np.abs(oe)))
    assert diff.max() <= (4e-4 + 2.0 ** -8) * vmax, (diff.max(), np.abs(of - oe).max())
    rel = np.abs(wf - we) / we
    assert rel.max() <= 2e-4, rel.max()
    moved = wf != we
    assert not moved[..., :3].any()          # rows 1-3 (O = 0) keep the exact weights
    # W moves on most iid rows at p = 15; where one weight dominates (the
    # needle rows, p = 64) W is that weight plus terms below its fp32
    # rounding step, so it moves on fewer rows
    assert moved.mean() > min_moved, moved.mean()
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    rows = sample_rows(L, seed=6)
    for h in range(H):
        ref = attention_forward(qf[0, h], kf[0, h], vf[0, h], MODE_LSSAR, p, rows=rows)
        assert np.abs(of[0, h, rows - 1] - ref).max() <= tol(MODE_LSSAR, p)
    check_error_word()


@pytest.mark.parametrize("odd_ulps", [1, 4, 16, 64])
@pytest.mark.parametrize("p", [3, 15])
def test_near_uniform_rows(torch_mod, odd_ulps, p):
    # Rows of i-1 equal keys and one key that differs by odd_ulps bf16 steps in
    # one component: the LSSA row is uniform up to a small spread, and Key
    # design 2 then puts all weight on the odd key (if it scores higher) or
    # spreads it evenly over the equal keys.  The kernel reads a row as the
    # 0/0 (prefix-mean) row when sp2(m) - theta <= 1e-4 sp2(m) + 1e-6.
    #
    # What the fp16 score operands can resolve: rounding q and k to fp16 moves
    # the score difference dz of the odd key and the others by at most
    # 2^-11 a_i (a_i = log2(e) ln d ln i; Cauchy-Schwarz on the rounding
    # errors).  What the fp32 softplus can resolve: for z >= 0 it is accurate
    # to about 1e-6 of its value, but for z < 0 (softplus below 1) the
    # MUFU lg2 near 1 and the product-form sum leave about 1e-4 of it, which
    # a near-uniform row (tiny sp2(m) - theta) amplifies.  Rows whose |dz|
    # exceeds twice the fp16 bound and whose largest score is >= 0 are decided
    # the same way in the kernel as in exact arithmetic and must match the
    # oracle element by element.
    # Rows the kernel flags as uniform (read back from the training statistics:
    # kappa = 0) must return the prefix mean, and must be within the fp16
    # resolution of uniform; no row far from uniform may be flagged.  Every
    # row's output is a convex combination of the values.
    from lssar_attn_fwd_gb300 import api
    from oracle import l2_normalize_rows, lssa_rows
    torch = torch_mod
    B, H, L, d = 1, 2, 512, 64
    qb, kb, vb = make_qkv(B, H, L, d, seed=odd_ulps, structure="odd_key", odd_ulps=odd_ulps)
    q, k, v = (to_dev(torch, t) for t in (qb, kb, vb))
    out, st = api.lssar_attn_fwd_train(q, k, v, p=p, mode=MODE_LSSAR)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    flagged = st.cpu().numpy()[..., 1] == 0.0            # kappa = 0: read as uniform
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    rows = np.arange(1, L + 1)
    decided = flagged_rows = 0
    for h in range(H):
        ref = attention_forward(qf[0, h], kf[0, h], vf[0, h], MODE_LSSAR, p)
        a = lssa_rows(qf[0, h], kf[0, h], rows, d)
        den_rel = (a.max(1) - 1.0 / rows) / a.max(1)
        ai = np.log(d) * np.log(rows) / np.log(2.0)
        qh, kh = l2_normalize_rows(qf[0, h]), l2_normalize_rows(kf[0, h])
        dz = ai * (qh @ (kh[1] - kh[0]))                  # odd key minus the equal keys, log2 units
        zmax = ai * np.maximum(qh @ kh[0], np.where(rows >= 2, qh @ kh[1], -np.inf))
        sure = (np.abs(dz) > 2.0 * 2.0 ** -11 * ai) & (zmax >= 0.0)
        sure[0] = True                                    # row 1 attends one key only
        e = np.abs(got[0, h] - ref).max(1)
        assert (e[sure] <= tol(MODE_LSSAR, p)).all(), (e[sure].max(), rows[sure][e[sure].argmax()])
        fl = flagged[0, h]
        fl[:3] = False                                    # rows 1-3 have O = 0: no threshold
        pm = np.cumsum(vf[0, h], axis=0) / rows[:, None]
        assert (np.abs(got[0, h, fl] - pm[fl]).max(initial=0.0) <= 2e-2)
        # a row whose odd key scores higher by more than the fp16 resolution
        # has sp2(m) - theta of at least about 2^-10 a_i sigma(z) (i-1)/i,
        # far above the band: the kernel never flags it.  (When the odd key
        # scores lower, sp2(m) - theta = (sp2(z_a) - sp2(z_b)) / i can fall in
        # the band; the exact answer, the mean over the equal keys, is then
        # within |v| / (i - 1) of the prefix mean and the parity check above
        # covers it.)
        assert not (fl & sure & (dz > 0)).any()
        cummin = np.minimum.accumulate(vf[0, h], axis=0)
        cummax = np.maximum.accumulate(vf[0, h], axis=0)
        assert (got[0, h] >= cummin - 2e-2).all() and (got[0, h] <= cummax + 2e-2).all()
        decided += int(sure.sum())
        flagged_rows += int(fl.sum())
    # the sweep spans the band: perturbations of 1 and 4 bf16 steps stay below
    # the fp16 resolution on every row (and reach the band on many), those of
    # 16 and 64 steps are resolved on most rows
    if odd_ulps >= 16:
        assert decided >= 50, decided
    else:
        assert flagged_rows >= 10, flagged_rows
    check_error_word()
