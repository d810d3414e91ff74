"""The replicas path of bench.py on CPU: two gloo ranks agree on the slowest rank's time and
report the whole-job throughput; the reference arm prints from rank 0 only."""
import io
import json
import os
import socket
import sys
import contextlib

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = 10.0 * (rank + 1)          # rank 1 is the slow one
        ms = bench._max_over_ranks(local_ms)
        value = bench._job_value(64 * 40, world, 5, ms)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == 20.0
    assert value == pytest.approx(world * 64 * 40 * 5 / 0.020)


def test_single_process_is_its_own_max():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(3.5) == 3.5
    assert bench._job_value(100, 1, 2, 1000.0) == pytest.approx(200.0)


def test_reference_arm_prints_on_rank0_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    import oracle

    class Args:
        T, ref_tokens, layers, steps, warmup = 4, 1, 2, 1, 0

    monkeypatch.setattr(oracle, "build", lambda *a, **k: None)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(Args(), world=2, rank=1)
    assert buf.getvalue() == ""
