"""The seeded input generator (shared by oracle tests, GPU tests and bench)."""

import numpy as np
import pytest

from lssar_attn_fwd_gb300.inputs import (
    WORKLOADS,
    bf16_bits_to_f64,
    f32_to_bf16_bits,
    make_qkv,
    needle_targets,
)


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * s for s in (1e-30, 1e-3, 1.0, 1e5, 1e30)])
    # include exact ties to check round-half-to-even
    ties = (np.arange(1, 2000, dtype=np.uint32) << 15 | 0x3F800000).view(np.float32)
    x = np.concatenate([x, ties, -ties])
    ours = f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_deterministic_and_shaped():
    a = make_qkv(1, 2, 64, 16, seed=3)
    b = make_qkv(1, 2, 64, 16, seed=3)
    c = make_qkv(1, 2, 64, 16, seed=4)
    for x, y in zip(a, b):
        assert x.shape == (1, 2, 64, 16) and x.dtype == np.uint16
        np.testing.assert_array_equal(x, y)
    assert not np.array_equal(a[0], c[0])


def test_iid_is_standard_normal():
    q, k, v = make_qkv(1, 4, 512, 64, seed=0)
    for t in (q, k, v):
        f = bf16_bits_to_f64(t)
        assert abs(f.mean()) < 0.01 and abs(f.std() - 1.0) < 0.01


def test_needle_structure():
    B, H, L, d = 1, 2, 256, 64
    q, k, v = make_qkv(B, H, L, d, seed=0, structure="needle")
    j = needle_targets(B, H, L, d, seed=0)
    assert j.min() >= 1 and np.all(j <= np.arange(1, L + 1)[None, None, :])
    qf, kf = bf16_bits_to_f64(q), bf16_bits_to_f64(k)
    nq = np.linalg.norm(qf, axis=-1)
    assert abs(nq.mean() - 1.0) < 0.02
    kn = kf / np.linalg.norm(kf, axis=-1, keepdims=True)
    qn = qf / nq[..., None]
    hits = 0
    for h in range(H):
        cos = qn[0, h] @ kn[0, h].T
        cos = np.where(np.tril(np.ones((L, L), bool)), cos, -np.inf)
        hits += np.sum(np.argmax(cos, axis=1) == j[0, h] - 1)
    assert hits / (H * L) > 0.99


def test_workload_table():
    assert WORKLOADS["extrap"].shape == (1, 12, 8192, 64)
    assert WORKLOADS["needle"].structure == "needle"
    assert WORKLOADS["wide"].d == 128


@pytest.mark.parametrize("ulps", [1, 16])
def test_odd_key_structure(ulps):
    q, k, v = make_qkv(2, 3, 40, 64, seed=7, structure="odd_key", odd_ulps=ulps)
    assert q.shape == k.shape == v.shape == (2, 3, 40, 64)
    for b in range(2):
        for h in range(3):
            kh = k[b, h]
            # every key equals key 1 except key 2, which differs in one component
            assert (kh[2:] == kh[0]).all()
            diff = np.nonzero(kh[1] != kh[0])[0]
            assert diff.size == 1
            c = diff[0]
            assert int(kh[1, c]) - int(kh[0, c]) == ulps      # bit pattern moved by `ulps` steps
            assert abs(bf16_bits_to_f64(kh[1, c])) > abs(bf16_bits_to_f64(kh[0, c]))   # away from zero
    a = make_qkv(2, 3, 40, 64, seed=7, structure="odd_key", odd_ulps=ulps)
    assert all((x == y).all() for x, y in zip(a, (q, k, v)))
