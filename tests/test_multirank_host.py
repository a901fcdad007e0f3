"""Host logic of the N > 1 benchmark run, on CPU with two gloo ranks.

The fused forward shards into independent work items, so a multi-GPU run is
N replicas with no collective on the data path; the only cross-rank steps are
the barrier, the max-over-ranks of the step time and the whole-job rate.  Those
run here as two spawned processes on the gloo backend (127.0.0.1).
"""
from __future__ import annotations

import multiprocessing as mp
import os
import socket
import sys
import types

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, step_ms: float, queue) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench

    w, r, local = bench.init_ranks()
    cpu = torch.device("cpu")
    slowest = bench.max_over_ranks(step_ms, w, cpu)
    rate = bench.job_throughput(1000.0, w, slowest)
    dist.barrier()
    queue.put((r, w, local, slowest, rate))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_step_and_sum_the_work():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    steps = [3.0, 5.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, steps[r], queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, (r, w, local, slowest, rate) in enumerate(results):
        assert (r, w, local) == (rank, 2, rank)
        assert slowest == max(steps)
        # 2 ranks x 1000 units in 5 ms
        assert rate == pytest.approx(2 * 1000.0 / 5e-3)


def test_single_rank_needs_no_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.init_ranks() == (1, 0, 0)
    assert bench.max_over_ranks(2.5, 1, None) == 2.5
    assert bench.job_throughput(10.0, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = types.SimpleNamespace(steps=1, warmup=3)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
