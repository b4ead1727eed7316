"""Host logic of bench.py's multi-replica run, on CPU: two gloo ranks.

The sampler path shards by rows with no exchange step (independent replicas), so
the only cross-rank logic is the timing: the slowest rank's time, whole-job rows
per second, rank 0 alone printing, and the reference arm running on rank 0 only.
"""
import importlib.util
import io
import os
import socket
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        ms = b.max_over_ranks(10.0 * (rank + 1), "cpu")
        out.put((rank, ms, b.job_rows_per_second(world, 64, 100, ms)))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_reaches_every_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    for _, ms, value in got:
        assert ms == pytest.approx(20.0)
        # 2 replicas x 64 rows x 100 steps in 20 ms
        assert value == pytest.approx(2 * 64 * 100 / 0.020)


def test_job_rows_per_second_is_weak_scaling():
    b = _bench()
    one = b.job_rows_per_second(1, 64, 1000, 29.0)
    two = b.job_rows_per_second(2, 64, 1000, 29.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(64 * 1000 / 0.029)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    b = _bench()
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        workload = "tiny"
        steps = 1
        warmup = 0
        gpus = 2

    buf = io.StringIO()
    with redirect_stdout(buf):
        b.run_reference(Args())
    assert buf.getvalue() == ""
