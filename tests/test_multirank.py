"""Replicas-only multi-GPU bookkeeping of bench.py, on CPU with gloo ranks:
the slowest rank's time sets the job time, `value` counts every rank's work,
and the reference arm prints on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_max, value = bench.aggregate(10.0 * (rank + 1), 2e12, world, dist)
    dist.barrier()
    out.put((rank, ms_max, value))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_and_whole_job_value(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    slowest = 10.0 * world
    for rank, ms_max, value in got:
        assert ms_max == slowest
        assert value == pytest.approx(2e12 * world / (slowest * 1e-3) / 1e12)


def test_single_rank_aggregate():
    import bench
    ms, v = bench.aggregate(4.0, 1e12, 1, None)
    assert ms == 4.0 and v == pytest.approx(250.0)


def test_reference_arm_silent_on_other_ranks(monkeypatch, capsys):
    import bench
    from fa_inputs import WORKLOADS
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, gpus = 3, 3, 2
    assert bench.run_reference(A(), WORKLOADS["tiny"]) == 0
    assert capsys.readouterr().out == ""
