"""Replica (N > 1) logic of bench.py on the CPU with two gloo ranks.

The path has no exchange step, so multi-GPU runs are independent replicas:
the only cross-rank operations are the barrier around the timed region and
the max over ranks of the step time; the reference arm runs on rank 0 only.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, local = bench.dist_env()
    bench.barrier(w)
    # each replica reports its own step time; the job's time is the slowest
    mx = bench.max_over_ranks(1.5 + rank, w, torch.device("cpu"))
    one = bench.max_over_ranks(2.0, 1, torch.device("cpu"))  # world 1: no collective
    dist.destroy_process_group()
    q.put((rank, r, w, local, mx, one))


def test_two_replicas_barrier_and_max_over_ranks():
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
    assert [o[:4] for o in out] == [(0, 0, 2, 0), (1, 1, 2, 1)]
    assert all(o[4] == 2.5 for o in out) and all(o[5] == 2.0 for o in out)


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""
