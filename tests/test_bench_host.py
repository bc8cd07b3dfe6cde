"""Host logic of bench.py without a GPU: the max-over-ranks timing and the
whole-job value on two gloo ranks, and the reference arm's rank handling."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    t = bench.reduce_max(1.5 * (rank + 1), "gloo")
    v = bench.aggregate_value(256, world, 10, t)
    bench.barrier()
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_two_rank_max_time_and_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in out:
        assert t == pytest.approx(3.0)  # slowest rank's time
        assert v == pytest.approx(256 * 2 * 10 / 3.0)  # every rank's sequences


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max(2.5, None) == 2.5
    assert bench.aggregate_value(256, 1, 4, 2.0) == 512.0
    peak, src = bench.measured_peaks()
    assert peak > 0 and src in ("measured", "fallback")


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
