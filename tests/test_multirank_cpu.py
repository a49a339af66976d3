"""The multi-rank logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

The layer shards over tokens with no exchange, so N GPUs run N replicas.  What the bench
does across ranks is (1) give every rank its own activation batches, (2) take the job's
time as the maximum over ranks, (3) report the whole job's throughput as the units all
ranks processed over that time, and (4) let only rank 0 run the CPU reference arm.
"""
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


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank 1 is the slow one for the first value, rank 0 for the second
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank], world, "cpu")
        seeds = bench.batch_seeds(rank, 4)
        all_seeds = [None] * world
        dist.all_gather_object(all_seeds, seeds)
        out.put((rank, got, all_seeds))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_max_and_draw_disjoint_batches():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, all_seeds in res:
        assert got == [2.0, 5.0]
        flat = [s for ss in all_seeds for s in ss]
        assert len(flat) == len(set(flat))


def test_job_rate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_rate(100.0, 1, 2.0) == 50.0
    assert bench.job_rate(100.0, 4, 2.0) == 200.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, gpus = 1, 0, 2
    bench.run_reference(A(), None)          # returns before touching the workload
    assert capsys.readouterr().out == ""
