"""The N > 1 host path of bench.py on CPU (gloo, world size 2): replicas
only, no collective on the data path; the step time is the slowest rank's,
the whole-job value counts every replica, and the reference arm runs on
rank 0 alone."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch

    sys.path.insert(0, ROOT)
    import bench

    torch.distributed.init_process_group(
        "gloo", rank=rank, world_size=world, init_method=f"tcp://127.0.0.1:{port}"
    )
    mine = 1.5 + 2.0 * rank  # rank 1 is the slow replica
    got = bench.max_over_ranks(mine, world)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"mine": mine, "max": got}, f)
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()


def test_step_time_is_the_slowest_rank(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    vals = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert [v["max"] for v in vals] == [3.5, 3.5]


def test_whole_job_value_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench

    one = bench.whole_job_gbs(1, 620_000_000, 0.125)
    assert bench.whole_job_gbs(2, 620_000_000, 0.125) == pytest.approx(2 * one)
    assert one == pytest.approx(4960.0)
    assert bench.max_over_ranks(7.0, 1) == 7.0


def test_reference_arm_under_torchrun_prints_once():
    cmd = [
        sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
        "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
        os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
        "--config", "1",
    ]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["value"] > 0
