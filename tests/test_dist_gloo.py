"""World-size-2 gloo run of the benchmark's multi-rank host logic on CPU:
max-over-ranks timing, summed bytes, barrier."""
import os
import sys
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        ms, nbytes = bench.aggregate(10.0 + 5.0 * rank, 1000 * (rank + 1))
        out[rank] = (ms, nbytes)
    finally:
        dist.destroy_process_group()


def test_aggregate_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == (15.0, 3000.0) and out[1] == (15.0, 3000.0)


def test_aggregate_single_process():
    import bench
    assert bench.aggregate(3.0, 7) == (3.0, 7)


def test_reference_arm_non_zero_rank_exits_quietly(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""
