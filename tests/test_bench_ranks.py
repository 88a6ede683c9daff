"""The multi-replica aggregation of bench.py on CPU: two gloo ranks each time
their own replica; the reported rate uses the slowest rank's time and counts
both replicas' work (replicas only -- no collective on the data path)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        out[rank] = (ms, bench.whole_job_rate(1e12, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_rank_rate_uses_slowest_rank_and_all_work():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        ms, rate = out[r]
        assert ms == 5.0                                   # max over ranks
        assert rate == pytest.approx(1e12 * 2 / 5e-3 / 1e12)  # both replicas' work


def test_single_rank_is_the_local_time():
    assert bench.max_over_ranks(4.0) == 4.0
    assert bench.whole_job_rate(2e12, 1, 1.0) == pytest.approx(2000.0)


def test_reference_arm_prints_one_line_from_rank_zero_under_torchrun():
    """`bench.py --impl reference` under torchrun with two CPU ranks: rank 0
    times the oracle and prints one JSON line; rank 1 exits without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
