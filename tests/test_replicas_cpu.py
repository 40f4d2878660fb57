"""Multi-process host logic of the benchmark on CPU (gloo, world size 2).

On several GPUs the path runs as independent replicas: no exchange during the
work, one reduction at the end (maximum time over ranks, summed work).  These
tests run that reduction with real processes over gloo on 127.0.0.1, and show
that a rank leaving before the collective makes the others fail within a short
process-group timeout instead of waiting for ever."""
from __future__ import annotations

import datetime
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port, timeout_s=60):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=timeout_s))


def _aggregate_worker(rank, world, port, out):
    import torch.distributed as dist

    import bench

    _init(rank, world, port)
    local_ms = [30.0, 45.0][rank]
    local_units = [1.0e12, 1.5e12][rank]
    t, u = bench.aggregate(local_ms, local_units, world)
    out[rank] = (t, u)
    dist.destroy_process_group()


def _leaver_worker(rank, world, port, out):
    import torch.distributed as dist

    import bench

    _init(rank, world, port, timeout_s=5)
    if rank == 1:
        dist.destroy_process_group()  # leaves between steps, before the final reduction
        out[rank] = "left"
        return
    try:
        bench.aggregate(10.0, 1.0, world)
        out[rank] = "completed"
    except Exception as exc:  # noqa: BLE001
        out[rank] = "error: " + type(exc).__name__


def _spawn(fn):
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    mp.start_processes(fn, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    return dict(out)


def test_replica_aggregation_max_time_sum_work():
    out = _spawn(_aggregate_worker)
    assert set(out) == {0, 1}
    for t, u in out.values():
        assert t == pytest.approx(45.0)
        assert u == pytest.approx(2.5e12)


def test_rank_leaving_before_reduction_is_detected():
    out = _spawn(_leaver_worker)
    assert out[1] == "left"
    assert out[0].startswith("error"), out[0]


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")

    def no_oracle(*a, **k):
        raise AssertionError("rank 1 ran the oracle")

    monkeypatch.setattr(bench, "run_oracle_subprocess", no_oracle)
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]) == 0
