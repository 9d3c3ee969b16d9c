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


def test_reference_arm_json_contract(capsys, monkeypatch):
    """The reference arm (the CPU oracle) prints one JSON line with the
    contract's keys; its ratio against our arm uses the same metric, unit and
    direction."""
    import json
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"]) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["higher_is_better"] is True and d["steps"] == 3 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1


def test_bench_untile_index_matches_oracle(orc):
    """The benchmark's quality report reads scale bytes back through the same
    layout as the oracle's untile."""
    import numpy as np
    import bench
    rng = np.random.default_rng(4)
    for M, K in ((129, 160), (300, 2880), (128, 256)):
        tiled = rng.integers(0, 256, orc.scale_bytes(M, K), dtype=np.uint8)
        idx = bench.tiled_scale_index(M, K).numpy()
        assert np.array_equal(tiled[idx], orc.untile(tiled, M, K // 32))
