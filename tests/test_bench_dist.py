"""Host-side logic of bench.py's multi-rank path, on two gloo ranks (CPU)."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.reduce_max_over_ranks([1.0 + rank, 10.0 * (world - rank)], "cpu")
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        for r in range(world):
            assert out[r] == [2.0, 20.0]


def test_single_rank_and_whole_job_value():
    import bench
    assert bench.reduce_max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]
    # weak scaling: N ranks each doing F flops in T ms
    assert bench.whole_job_tflops(4, 2e12, 1000.0) == pytest.approx(8.0)


def test_reference_arm_silent_on_other_ranks(monkeypatch, capsys):
    import argparse
    import bench
    from lssar_attn_fwd_gb300.inputs import WORKLOADS, MODE_LSSAR
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(steps=2, warmup=3, gpus=2)
    bench.run_reference(args, WORKLOADS["tiny"], MODE_LSSAR, 3)
    assert capsys.readouterr().out == ""
