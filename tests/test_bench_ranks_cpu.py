"""The benchmark's multi-rank host logic on CPU (gloo, world size 2).

With N GPUs every rank steps its own replica of the workload; the ranks meet
only in a barrier around the timed region and in a max over the per-rank step
times (the slowest replica sets the step time).  The reference arm runs on
rank 0 alone.  No GPU is involved.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        bench.rank_barrier(world)
        got = bench.rank_max(1.5 * (rank + 1), world, torch.device("cpu"))
        # a single-rank call returns its own value without any collective
        alone = bench.rank_max(7.0, 1, torch.device("cpu"))
        bench.rank_barrier(world)
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got, "alone": alone}, f)


def test_rank_max_and_barrier_two_ranks(tmp_path):
    world = 2
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True, start_method="spawn")
    for r in range(world):
        with open(tmp_path / f"rank{r}.json") as f:
            d = json.load(f)
        assert d["max"] == pytest.approx(3.0)  # max of 1.5 and 3.0, seen by both ranks
        assert d["alone"] == 7.0


def _reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", str(world),
                           "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                          capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _reference(1, 2)
    assert r1.returncode == 0, r1.stderr[-2000:]
    assert r1.stdout.strip() == ""  # the other ranks exit 0 without work
    r0 = _reference(0, 2)
    assert r0.returncode == 0, r0.stderr[-2000:]
    lines = [l for l in r0.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
