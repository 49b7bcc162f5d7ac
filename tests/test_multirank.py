"""The N > 1 path on the CPU with world size 2 over gloo: the timing
reduction bench.py uses (maximum over ranks, then a barrier), the whole-job
throughput of weak scaling, and the reference arm under torchrun (rank 0
prints the one JSON line; the other rank exits without work)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    got = bench.max_over_ranks(torch, [1.0 + rank, 10.0 - rank, 0.5 * rank], "cpu")
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(got, f)
    dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for rank in range(2):
        with open(tmp_path / f"rank{rank}.json") as f:
            assert json.load(f) == [2.0, 10.0, 0.5]  # every rank gets the per-entry maximum


def test_whole_job_throughput_is_weak_scaling():
    import bench
    one = bench.whole_job_gbs(1, 581_861_376, 50, 0.02)
    assert one == pytest.approx(581_861_376 * 50 / 0.02 / 1e9)
    assert bench.whole_job_gbs(4, 581_861_376, 50, 0.02) == pytest.approx(4 * one)


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-rows", "8"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
