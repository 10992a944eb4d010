"""The benchmark's multi-rank host logic on CPU: world-size-2 gloo ranks for
the max-over-ranks timing and the whole-job rate, and the reference arm
under torchrun with two ranks (rank 0 alone works and prints)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r took (r + 1) * 10 ms: the job took the slowest rank's time
        ms = bench.max_over_ranks((rank + 1) * 10.0, world, "cpu")
        rate = bench.whole_job_rate(world, 8192, 50, ms)
        out[rank] = (ms, rate)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_with_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 20.0
    assert res[0][1] == res[1][1] == pytest.approx(2 * 8192 * 50 / 0.020)


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_rate(1, 100, 10, 1000.0) == pytest.approx(1000.0)
    seeds = {bench.rank_seed(3, r) for r in range(8)}
    assert len(seeds) == 8 and bench.rank_seed(3, 0) == 3


def test_reference_arm_under_torchrun_two_ranks():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--reference-tokens", "4"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
