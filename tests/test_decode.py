"""GPU parity of the decode forward (one query row per head at position L)
against row L of the float64 oracle."""

import numpy as np
import pytest

from lssar_attn_fwd_gb300.inputs import (
    MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW, MODE_SOFTMAX, MODE_SOFTMAX_RW,
    bf16_bits_to_f64, make_qkv)
from oracle import attention_forward

pytestmark = pytest.mark.gpu

ALL = [(MODE_SOFTMAX, 1), (MODE_LSSA, 1), (MODE_LSSAR, 3), (MODE_LSSAR, 15),
       (MODE_SOFTMAX_RW, 15), (MODE_SIGMOID_RW, 15), (MODE_LSSAR, 64)]


def tol(mode, p):
    return 5e-2 if (mode in (MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW) and p >= 15) else 2e-2


@pytest.fixture(scope="module")
def torch_mod():
    import torch
    from lssar_attn_fwd_gb300 import api, build
    build.build()
    api.load_library()
    return torch


def decode(torch, qb, kb, vb, p, mode):
    from lssar_attn_fwd_gb300 import api
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    q_last = dev(qb[:, :, -1])
    out = api.lssar_attn_decode(q_last, dev(kb), dev(vb), p=p, mode=mode)
    torch.cuda.synchronize()
    assert api.device_error_word() == 0
    return out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("L", [1, 2, 3, 4, 255, 1000, 4097, 9000])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_matches_last_row(torch_mod, L, d, decode_path):
    B, H = 2, 3
    qb, kb, vb = make_qkv(B, H, L, d, seed=L + d)
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    for mode, p in ALL:
        got = decode(torch_mod, qb, kb, vb, p, mode)
        for b in range(B):
            for h in range(H):
                ref = attention_forward(qf[b, h], kf[b, h], vf[b, h], mode, p, rows=np.array([L]))[0]
                err = np.abs(got[b, h] - ref).max()
                assert err <= tol(mode, p), (L, d, mode, p, b, h, err)


def test_decode_needle_16k(torch_mod):
    B, H, L, d = 1, 12, 16384, 64
    qb, kb, vb = make_qkv(B, H, L, d, seed=0, structure="needle")
    qf, kf, vf = (bf16_bits_to_f64(t) for t in (qb, kb, vb))
    got = decode(torch_mod, qb, kb, vb, 15, MODE_LSSAR)
    for h in range(H):
        ref = attention_forward(qf[0, h], kf[0, h], vf[0, h], MODE_LSSAR, 15, rows=np.array([L]))[0]
        assert np.abs(got[0, h] - ref).max() <= 5e-2


def test_decode_equals_prefill_last_row(torch_mod):
    # the decode entry and the prefill kernel agree on row L
    torch = torch_mod
    from lssar_attn_fwd_gb300 import api
    qb, kb, vb = make_qkv(2, 4, 1500, 64, seed=9)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    full = api.lssar_attn_fwd(dev(qb), dev(kb), dev(vb), p=15, mode=MODE_LSSAR)
    torch.cuda.synchronize()
    last = full[:, :, -1].float().cpu().numpy()
    got = decode(torch, qb, kb, vb, 15, MODE_LSSAR)
    assert np.abs(got - last).max() <= 5e-2


@pytest.fixture(params=["cluster", "grid", "split"])
def decode_path(request, monkeypatch):
    # cluster: one thread-block cluster per head (the default wherever the
    # head's cache fits 16 chunks); grid: the cooperative launch with a grid
    # barrier; split: separate score / weight / combine launches
    if request.param != "cluster":
        monkeypatch.setenv("LSSAR_DECODE_PATH", request.param)
    else:
        monkeypatch.delenv("LSSAR_DECODE_PATH", raising=False)
    return request.param


@pytest.mark.parametrize("d", [64, 128])
def test_decode_many_heads(torch_mod, d, decode_path):
    # 768 heads (more CTAs than can be resident at once on the grid path, which
    # then runs as three launches); sampled heads against the oracle
    B, H, L = 8, 96, 300
    qb, kb, vb = make_qkv(B, H, L, d, seed=d)
    for mode, p in [(MODE_LSSAR, 15), (MODE_SOFTMAX, 1)]:
        got = decode(torch_mod, qb, kb, vb, p, mode)
        for b, h in ((0, 0), (3, 50), (7, 95)):
            qf, kf, vf = (bf16_bits_to_f64(t[b, h]) for t in (qb, kb, vb))
            ref = attention_forward(qf, kf, vf, mode, p, rows=np.array([L]))[0]
            assert np.abs(got[b, h] - ref).max() <= tol(mode, p), (d, mode, b, h)


def test_decode_long_single_head(torch_mod, decode_path):
    # one head, 40000 keys: a cluster of 16 chunks, or (grid path) hundreds of
    # chunks of one head that meet at the grid barrier, the last one to finish
    # combining them
    B, H, L, d = 1, 1, 40000, 64
    qb, kb, vb = make_qkv(B, H, L, d, seed=5)
    qf, kf, vf = (bf16_bits_to_f64(t[0, 0]) for t in (qb, kb, vb))
    for mode, p in [(MODE_LSSAR, 15), (MODE_SOFTMAX_RW, 3)]:
        got = decode(torch_mod, qb, kb, vb, p, mode)
        ref = attention_forward(qf, kf, vf, mode, p, rows=np.array([L]))[0]
        assert np.abs(got[0, 0] - ref).max() <= tol(mode, p), mode


def test_decode_beyond_cluster_reach(torch_mod):
    # 70000 keys in one head: more than 16 chunks of 4096, so the default path
    # is the cooperative launch
    B, H, L, d = 1, 1, 70000, 64
    qb, kb, vb = make_qkv(B, H, L, d, seed=11)
    qf, kf, vf = (bf16_bits_to_f64(t[0, 0]) for t in (qb, kb, vb))
    got = decode(torch_mod, qb, kb, vb, 15, MODE_LSSAR)
    ref = attention_forward(qf, kf, vf, MODE_LSSAR, 15, rows=np.array([L]))[0]
    assert np.abs(got[0, 0] - ref).max() <= 5e-2


def expected_cluster_split(BH, L, sms):
    """The cluster path's split of each head's cache: about one wave of four
    CTAs per SM (at least one chunk, at most 16), chunks a multiple of 64 keys
    and at most 4096; None when no split fits."""
    nch = min(max(4 * sms // BH, 1), 16)
    chunk = -(-L // nch)
    chunk = -(-chunk // 64) * 64
    if chunk > 4096:
        return None
    return -(-L // chunk), chunk


@pytest.mark.parametrize("B,H,L,d", [(8, 12, 16384, 64), (64, 12, 2048, 64), (1, 32, 32768, 128),
                                     (4, 16, 4096, 128), (2, 3, 1, 64), (1, 1, 70000, 64)])
def test_decode_plan(torch_mod, B, H, L, d, monkeypatch):
    from lssar_attn_fwd_gb300 import api
    monkeypatch.delenv("LSSAR_DECODE_PATH", raising=False)
    sms = torch_mod.cuda.get_device_properties(0).multi_processor_count
    plan = api.decode_plan(B, H, L, d)
    exp = expected_cluster_split(B * H, L, sms)
    if exp is None:   # longer than 16 chunks of 4096 keys: grid or three launches
        assert plan["path"] in (1, 2) and plan["launches"] == (1 if plan["path"] == 1 else 3)
    else:
        assert (plan["path"], plan["launches"]) == (0, 1)
        assert (plan["chunks"], plan["chunk_rows"]) == exp
    assert plan["chunk_rows"] % 64 == 0 and plan["chunk_rows"] <= 4096
    assert (plan["chunks"] - 1) * plan["chunk_rows"] < L <= plan["chunks"] * plan["chunk_rows"]
    monkeypatch.setenv("LSSAR_DECODE_PATH", "split")
    split = api.decode_plan(B, H, L, d)
    assert (split["path"], split["launches"]) == (2, 3)
