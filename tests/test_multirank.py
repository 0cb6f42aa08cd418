"""Multi-rank host logic of bench.py on CPU: two gloo ranks (replicas of the
single-GPU path; the reduction is the max of the per-rank step times)."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms_local = [5.0, 7.5][rank]
        ms, value = bench.job_throughput(ms_local, 8192, world, torch.device("cpu"))
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_job_throughput_takes_the_slowest_rank_and_all_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for ms, value in res.values():
        assert ms == 7.5
        assert value == pytest.approx(2 * 8192 / 7.5e-3)


def test_single_rank_needs_no_process_group():
    import bench

    assert not dist.is_initialized()
    ms, value = bench.job_throughput(4.0, 1000, 1)
    assert ms == 4.0 and value == pytest.approx(1000 / 4e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert rc == 0 and buf.getvalue() == ""
