"""The benchmark's multi-rank path on the CPU: two gloo ranks aggregate their
step times (the slowest rank's) and tokens (all ranks') into the whole-job
throughput, as the GPU run does over NCCL."""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        value, total_ms = bench.aggregate(10.0 * (rank + 1), 8192, 5, "cpu")
        results[rank] = (value, total_ms)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_uses_slowest_rank_and_all_tokens():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        value, total_ms = results[r]
        assert total_ms == pytest.approx(20.0)
        assert value == pytest.approx(2 * 8192 * 5 / 0.020 / 1e6)


def test_single_process_aggregation_is_local():
    import bench
    value, total_ms = bench.aggregate(4.0, 1000, 2, "cpu")
    assert total_ms == 4.0 and value == pytest.approx(1000 * 2 / 0.004 / 1e6)


def test_reference_arm_prints_once_on_rank_zero():
    """Under a multi-rank launch the reference arm (the oracle on the host
    cores) runs on rank 0 alone and prints one JSON line; other ranks exit 0
    without work or output."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = []
    for rank in (0, 1):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2")
        r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                            "--steps", "1", "--warmup", "0", "--ref-tokens", "64"],
                           capture_output=True, text=True, env=env, cwd=root, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append([ln for ln in r.stdout.splitlines() if ln.strip()])
    assert outs[1] == []
    assert len(outs[0]) == 1
    line = json.loads(outs[0][0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
