"""Pins for the float64 oracle (CPU only).

Each test ties the oracle to something other than itself: a second scalar
transcription on tiny inputs, closed forms derived by hand, limits stated in
the notes, library routines for the softmax special case, and invariants.
A plausible slip in the oracle (wrong log base, 0-based row index, O on the
wrong rows, missing L1 step, transposed product, mask before softplus...)
fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import (
    MODE_LSSA,
    MODE_LSSAR,
    MODE_SIGMOID_RW,
    MODE_SOFTMAX,
    MODE_SOFTMAX_RW,
    attention_bruteforce,
    attention_forward,
    lssa_rows,
    reweight_rows,
    softplus,
)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALL_MODES = (MODE_SOFTMAX, MODE_LSSA, MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW)
RW_MODES = (MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW)


def rand_qkv(L, d, seed, lead=()):
    rng = np.random.default_rng(seed)
    shape = lead + (L, d)
    return (rng.standard_normal(shape), rng.standard_normal(shape), rng.standard_normal(shape))


# --- second transcription -------------------------------------------------

@pytest.mark.parametrize("L,d", [(1, 4), (5, 4), (17, 16), (32, 8)])
@pytest.mark.parametrize("mode,p", [(MODE_SOFTMAX, 1), (MODE_LSSA, 1), (MODE_LSSAR, 1),
                                    (MODE_LSSAR, 3), (MODE_LSSAR, 15), (MODE_SOFTMAX_RW, 3),
                                    (MODE_SOFTMAX_RW, 15), (MODE_SIGMOID_RW, 3), (MODE_SIGMOID_RW, 15)])
def test_bruteforce_agrees(L, d, mode, p):
    q, k, v = rand_qkv(L, d, seed=L * 100 + d)
    ref = attention_bruteforce(q.tolist(), k.tolist(), v.tolist(), mode, p)
    got = attention_forward(q, k, v, mode, p)
    np.testing.assert_allclose(got, np.array(ref), rtol=1e-10, atol=1e-12)


def test_bruteforce_agrees_zero_bias():
    q, k, v = rand_qkv(24, 8, seed=7)
    ref = attention_bruteforce(q.tolist(), k.tolist(), v.tolist(), MODE_LSSAR, 3, o_override=0.0)
    got = attention_forward(q, k, v, MODE_LSSAR, 3, o_override=0.0)
    np.testing.assert_allclose(got, np.array(ref), rtol=1e-10, atol=1e-12)


# --- structural facts from the definitions --------------------------------

@pytest.mark.parametrize("mode,p", [(MODE_SOFTMAX, 1), (MODE_LSSA, 1), (MODE_LSSAR, 3), (MODE_LSSAR, 15),
                                    (MODE_SOFTMAX_RW, 15), (MODE_SIGMOID_RW, 15)])
def test_rows_sum_to_one(mode, p):
    # Every stage ends with an L1 normalisation (Key designs 1 and 2), so
    # V = ones gives an output of exactly ones.
    q, k, _ = rand_qkv(96, 16, seed=3)
    out = attention_forward(q, k, np.ones_like(q), mode, p)
    np.testing.assert_allclose(out, 1.0, atol=1e-12)


@pytest.mark.parametrize("mode,p", [(MODE_SOFTMAX, 1), (MODE_LSSA, 1), (MODE_LSSAR, 3), (MODE_LSSAR, 200),
                                    (MODE_SOFTMAX_RW, 15), (MODE_SIGMOID_RW, 3)])
def test_first_row_is_first_value(mode, p):
    # Row 1 attends one token: log 1 = 0, softplus(0) = ln 2 normalises to 1.
    q, k, v = rand_qkv(10, 8, seed=4)
    out = attention_forward(q, k, v, mode, p)
    np.testing.assert_allclose(out[0], v[0], rtol=0, atol=1e-15)


def test_causality():
    # The multiplicative mask M': row i never sees keys or values after i.
    q, k, v = rand_qkv(40, 8, seed=5)
    k2, v2 = k.copy(), v.copy()
    k2[20:] = 9.0 * np.random.default_rng(1).standard_normal(k2[20:].shape)
    v2[20:] = -7.0
    for mode, p in ((MODE_SOFTMAX, 1), (MODE_LSSA, 1), (MODE_LSSAR, 3)):
        a = attention_forward(q, k, v, mode, p)
        b = attention_forward(q, k2, v2, mode, p)
        np.testing.assert_array_equal(a[:20], b[:20])
        assert np.abs(a[20:] - b[20:]).max() > 1e-3


def test_l2_normalisation_makes_scale_irrelevant():
    # Q and K rows are L2-normalised (Key design 1): positive per-row scale
    # factors leave LSSA / LSSAR unchanged, but change softmax.
    q, k, v = rand_qkv(30, 8, seed=6)
    rng = np.random.default_rng(2)
    sq = rng.uniform(0.1, 10.0, size=(30, 1))
    sk = rng.uniform(0.1, 10.0, size=(30, 1))
    for mode, p in ((MODE_LSSA, 1), (MODE_LSSAR, 3), (MODE_LSSAR, 15)):
        np.testing.assert_allclose(attention_forward(q * sq, k * sk, v, mode, p),
                                   attention_forward(q, k, v, mode, p), rtol=1e-9, atol=1e-12)
    assert np.abs(attention_forward(q * sq, k * sk, v, MODE_SOFTMAX)
                  - attention_forward(q, k, v, MODE_SOFTMAX)).max() > 1e-3


def test_identical_keys_give_prefix_mean():
    # Uniform scores: LSSA weights are 1/i (Key design 1).  In LSSAR rows 1-3
    # (O = 0) all re-weighted entries are equal; from row 4 on every entry is
    # ReLU(1 - 1) = 0, the 0/0 case read as the uniform prefix mean.
    L, d = 48, 16
    rng = np.random.default_rng(8)
    q = rng.standard_normal((L, d))
    k = np.tile(rng.standard_normal((1, d)), (L, 1))
    v = rng.standard_normal((L, d))
    mean = np.cumsum(v, axis=0) / np.arange(1, L + 1)[:, None]
    for mode, p in ((MODE_LSSA, 1), (MODE_LSSAR, 1), (MODE_LSSAR, 3), (MODE_LSSAR, 15)):
        np.testing.assert_allclose(attention_forward(q, k, v, mode, p), mean, atol=1e-12)


def test_zero_query_rows():
    # A zero query has all-zero cosine scores (norm clamped): uniform LSSA row.
    q, k, v = rand_qkv(12, 8, seed=9)
    q[5] = 0.0
    q[1] = 0.0
    out_a = attention_forward(q, k, v, MODE_LSSA)
    out_r = attention_forward(q, k, v, MODE_LSSAR, 3)
    for r in (1, 5):
        np.testing.assert_allclose(out_a[r], v[:r + 1].mean(axis=0), atol=1e-12)
        np.testing.assert_allclose(out_r[r], v[:r + 1].mean(axis=0), atol=1e-12)


def test_p1_zero_bias_reduces_to_lssa():
    # With p = 1 and O = 0, ReLU(i a) = i a and the second L1 step undoes the
    # factor i: re-weighting is the identity (Key design 2).
    q, k, v = rand_qkv(64, 16, seed=10)
    np.testing.assert_allclose(attention_forward(q, k, v, MODE_LSSAR, 1, o_override=0.0),
                               attention_forward(q, k, v, MODE_LSSA), rtol=1e-10, atol=1e-12)


def test_bias_only_on_rows_from_four():
    # O is zero on rows 1-3: rows 1-3 of LSSAR are unchanged by forcing O = 0,
    # while later rows change.
    q, k, v = rand_qkv(20, 8, seed=11)
    a = attention_forward(q, k, v, MODE_LSSAR, 3)
    b = attention_forward(q, k, v, MODE_LSSAR, 3, o_override=0.0)
    np.testing.assert_allclose(a[:3], b[:3], rtol=1e-12, atol=1e-14)
    assert np.all(np.abs(a[3:] - b[3:]).max(axis=1) > 1e-6)


def test_rows_two_three_closed_form():
    # With O = 0, ReLU^p(i a_j) normalised is sp_j^p / sum_k sp_k^p (the
    # factor i / S1 cancels), sp_j = log(1 + exp(ln d ln i cos(q_i, k_j))).
    for d in (4, 16, 64):
        q, k, v = rand_qkv(3, d, seed=d)
        for p in (1, 3, 15):
            out = attention_forward(q, k, v, MODE_LSSAR, p)
            for i in (2, 3):
                c = math.log(d) * math.log(i)
                sp = []
                for j in range(i):
                    cos = float(q[i - 1] @ k[j]) / (np.linalg.norm(q[i - 1]) * np.linalg.norm(k[j]))
                    sp.append(math.log(1.0 + math.exp(c * cos)))
                w = np.array(sp) ** p
                np.testing.assert_allclose(out[i - 1], (w / w.sum()) @ v[:i], rtol=1e-10, atol=1e-12)


def test_golden_threshold_case():
    with open(os.path.join(GOLDEN, "threshold_row4.json")) as f:
        g = json.load(f)
    q, k, v = (np.array(g[n], dtype=np.float64) for n in ("q", "k", "v"))
    e = g["expected"]
    for p in g["p_values"]:
        out = attention_forward(q, k, v, MODE_LSSAR, p)
        np.testing.assert_allclose(out[3], e["lssar_row4_any_p"], atol=1e-12)
        np.testing.assert_allclose(out[1], e["lssar_row2_any_p"], atol=1e-12)
    np.testing.assert_allclose(attention_forward(q, k, v, MODE_LSSA)[1], e["lssa_row2"], atol=1e-12)
    for mode in ALL_MODES:
        np.testing.assert_allclose(attention_forward(q, k, v, mode, 3)[0], e["row1_all_modes"], atol=0)


def test_large_p_tends_to_argmax():
    # lim_{p->inf} of the re-weighted row is one-hot on the largest entry
    # (Key design 2).  Needle rows: query i points at key j(i).
    L, d = 32, 16
    rng = np.random.default_rng(12)
    k = rng.standard_normal((L, d))
    v = rng.standard_normal((L, d))
    j = np.array([rng.integers(0, i + 1) for i in range(L)])
    q = k[j] / np.linalg.norm(k[j], axis=1, keepdims=True) + 0.05 * rng.standard_normal((L, d))
    rows = np.arange(1, L + 1)
    a = lssa_rows(q, k, rows, d)
    w200 = reweight_rows(a, rows, 200)
    w3 = reweight_rows(a, rows, 3)
    w15 = reweight_rows(a, rows, 15)
    arg = np.argmax(a, axis=1)
    np.testing.assert_array_equal(arg[4:], j[4:])
    top = w200[np.arange(L), arg]
    assert np.all(top >= 1.0 - 1e-6)
    # sharpening grows with p: the argmax weight is non-decreasing in p
    t3, t15 = w3[np.arange(L), arg], w15[np.arange(L), arg]
    assert np.all(t15 >= t3 - 1e-15) and np.all(top >= t15 - 1e-15)
    out = attention_forward(q, k, v, MODE_LSSAR, 200)
    np.testing.assert_allclose(out[4:], v[j[4:]], atol=1e-5)


def test_softmax_matches_library_sdpa():
    torch = pytest.importorskip("torch")
    q, k, v = rand_qkv(50, 16, seed=13, lead=(2, 3))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=True).numpy()
    np.testing.assert_allclose(attention_forward(q, k, v, MODE_SOFTMAX), ref, rtol=1e-10, atol=1e-12)


def test_softplus_special_values():
    # log(1 + e^x): ln 2 at 0, x + log1p(e^-x) identity, e^x for very negative x
    assert softplus(0.0) == pytest.approx(math.log(2.0), abs=0, rel=1e-16)
    for x in (-40.0, -3.0, 0.5, 7.0, 40.0, 700.0):
        ref = math.log1p(math.exp(x)) if x < 700 else x
        assert softplus(x) == pytest.approx(ref, rel=1e-15)
    assert softplus(-800.0) == 0.0


def test_row_subsets_and_blocks_agree():
    q, k, v = rand_qkv(70, 8, seed=14, lead=(2,))
    full = attention_forward(q, k, v, MODE_LSSAR, 15, block=256)
    small = attention_forward(q, k, v, MODE_LSSAR, 15, block=7)
    np.testing.assert_allclose(small, full, rtol=1e-13, atol=1e-15)
    rows = np.array([70, 1, 33, 4, 2])
    sub = attention_forward(q, k, v, MODE_LSSAR, 15, rows=rows)
    np.testing.assert_allclose(sub, full[:, rows - 1], rtol=1e-13, atol=1e-15)


def test_length_scale_grows_sharpness():
    # The factor ln d ln i raises the effective inverse temperature with the
    # row index: for identical score patterns, a later row is sharper.
    d = 16
    rng = np.random.default_rng(15)
    kv = rng.standard_normal((8, d))
    q = rng.standard_normal((1, d))
    k = np.concatenate([np.tile(kv, (4, 1))])          # 32 keys: the 8-key pattern repeated
    s8 = lssa_rows(q, k, np.array([8]), d)[0, :8]
    s32 = lssa_rows(q, k, np.array([32]), d)[0, :32].reshape(4, 8).sum(axis=0)
    ent = lambda w: -(w * np.log(w)).sum()
    assert ent(s32) < ent(s8)


# --- ablation modes (the notes' ablation table) ---------------------------

def test_softmax_reweight_p1_zero_bias_is_library_sdpa():
    # p = 1 and O = 0 make re-weighting the identity, so re-weighting on a
    # softmax normaliser reduces to plain softmax attention.
    torch = pytest.importorskip("torch")
    q, k, v = rand_qkv(40, 16, seed=21)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        is_causal=True).numpy()[0]
    got = attention_forward(q, k, v, MODE_SOFTMAX_RW, 1, o_override=0.0)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_softmax_reweight_rows_two_three_closed_form():
    # Rows 2-3 (O = 0): weights proportional to softmax_j^p, i.e. to
    # exp(p * q.k_j / sqrt(d)).
    d = 8
    q, k, v = rand_qkv(3, d, seed=22)
    for p in (1, 3, 15):
        out = attention_forward(q, k, v, MODE_SOFTMAX_RW, p)
        for i in (2, 3):
            sc = np.array([float(q[i - 1] @ k[j]) / math.sqrt(d) for j in range(i)])
            w = np.exp(p * (sc - sc.max()))
            np.testing.assert_allclose(out[i - 1], (w / w.sum()) @ v[:i], rtol=1e-10, atol=1e-12)


def test_sigmoid_reweight_rows_two_three_closed_form():
    # Rows 2-3 (O = 0): weights proportional to sigmoid(ln d ln i cos)^p.
    for d in (4, 16):
        q, k, v = rand_qkv(3, d, seed=30 + d)
        for p in (1, 3, 15):
            out = attention_forward(q, k, v, MODE_SIGMOID_RW, p)
            for i in (2, 3):
                c = math.log(d) * math.log(i)
                sg = []
                for j in range(i):
                    cos = float(q[i - 1] @ k[j]) / (np.linalg.norm(q[i - 1]) * np.linalg.norm(k[j]))
                    sg.append(1.0 / (1.0 + math.exp(-c * cos)))
                w = np.array(sg) ** p
                np.testing.assert_allclose(out[i - 1], (w / w.sum()) @ v[:i], rtol=1e-10, atol=1e-12)


def test_sigmoid_golden_threshold_case():
    # The hand-derived row-4 case holds for the sigmoid normaliser too:
    # sigmoid(c) + sigmoid(-c) = 1 gives 4a - 1 = 2 sigmoid(+-c) - 1, positive
    # for the two aligned keys only.
    with open(os.path.join(GOLDEN, "threshold_row4.json")) as f:
        g = json.load(f)
    q, k, v = (np.array(g[n], dtype=np.float64) for n in ("q", "k", "v"))
    for p in g["p_values"]:
        out = attention_forward(q, k, v, MODE_SIGMOID_RW, p)
        np.testing.assert_allclose(out[3], g["expected"]["lssar_row4_any_p"], atol=1e-12)


@pytest.mark.parametrize("mode", RW_MODES)
def test_reweight_modes_identical_keys_prefix_mean(mode):
    L, d = 30, 8
    rng = np.random.default_rng(23)
    q = rng.standard_normal((L, d))
    k = np.tile(rng.standard_normal((1, d)), (L, 1))
    v = rng.standard_normal((L, d))
    mean = np.cumsum(v, axis=0) / np.arange(1, L + 1)[:, None]
    np.testing.assert_allclose(attention_forward(q, k, v, mode, 15), mean, atol=1e-12)


def test_reweight_modes_large_p_argmax():
    # lim_{p->inf}: one-hot on the row's largest entry (Key design 2).  Rows
    # are kept where the second-largest re-weighting input is below 0.9 of the
    # largest, so that (0.9)^400 is negligible; the argmax is that of the raw
    # scores (q.k for the softmax normaliser, the cosine for the sigmoid one).
    L, d = 32, 16
    rng = np.random.default_rng(24)
    k = rng.standard_normal((L, d))
    v = rng.standard_normal((L, d))
    j = np.array([rng.integers(0, i + 1) for i in range(L)])
    q = 4.0 * k[j] / np.linalg.norm(k[j], axis=1, keepdims=True)
    kn = k / np.linalg.norm(k, axis=1, keepdims=True)
    rows = np.arange(1, L + 1)
    from oracle.lssar_oracle import softmax_rows, sigmoid
    for mode, sc, a in ((MODE_SOFTMAX_RW, q @ k.T / math.sqrt(d), softmax_rows(q, k, rows, d)),
                        (MODE_SIGMOID_RW, q @ kn.T, lssa_rows(q, k, rows, d, phi=sigmoid))):
        sc = np.where(np.tril(np.ones((L, L), bool)), sc, -np.inf)
        y = np.sort(np.maximum(rows[:, None] * a - 1.0, 0.0), axis=1)
        clear = (y[:, -2] < 0.9 * y[:, -1]) & (rows >= 4)
        assert clear.sum() > 10
        out = attention_forward(q, k, v, mode, 400)
        arg = np.argmax(sc, axis=1)
        np.testing.assert_allclose(out[clear], v[arg[clear]], atol=1e-6)
