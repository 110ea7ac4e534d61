"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each timing its
own replica, agree on the max-over-ranks time and pass the barriers."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, local = bench._dist()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(world)
    got = bench.reduce_max(1.5 + rank, world)   # each rank's own elapsed time
    bench.barrier(world)
    results[rank] = got
    dist.destroy_process_group()


def test_two_rank_max_timing():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert dict(results) == {0: 2.5, 1: 2.5}


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)


def test_reference_arm_quiet_on_other_ranks(monkeypatch, capsys):
    """Under torchrun only rank 0 runs the oracle arm; other ranks exit quietly."""
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1"])
    assert capsys.readouterr().out == ""
