"""World-size-2 checks of bench.py's multi-rank host logic on CPU (gloo):
the step time is the max over ranks, and the CPU reference arm runs on rank 0
only (other ranks return without work)."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.reduce_max(10.0 * (rank + 1))
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_step_time_is_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 20.0, 1: 20.0}


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "cpu_baseline", lambda *a, **k: called.append(1))
    bench.run_reference(bench.argparse.Namespace(workload=1, steps=2, warmup=1, batch=None))
    assert not called and capsys.readouterr().out == ""


def test_reduce_max_without_a_process_group_is_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
