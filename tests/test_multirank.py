"""The benchmark's multi-rank path on CPU: two gloo ranks (the data path has
no collective; only the timing is reduced).  Checks that every rank sees the
slowest rank's time, that the job throughput counts every rank's work, and
that the reference arm runs on rank 0 only."""
from __future__ import annotations

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


def _worker(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_setup()
        assert (w, r) == (world, rank)
        t = bench.max_over_ranks(1.0 + rank)        # rank 1 is the slow one
        v = bench.job_throughput(2e12, 10, w, t)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{t} {v}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timing(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    vals = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(2)]
    for t, v in vals:
        assert float(t) == 2.0                       # the max over ranks
        assert abs(float(v) - 2 * 2e12 * 10 / 2.0 / 1e12) < 1e-9


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(1e12, 4, 1, 2.0) == 2.0


def test_reference_arm_only_rank0_prints(tmp_path):
    """Under torchrun the reference arm runs on rank 0 alone; rank 1 exits 0
    without output and without work."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert res.returncode == 0 and res.stdout.strip() == ""


@pytest.mark.slow
def test_reference_arm_prints_one_line(tmp_path):
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "s256",
                          "--steps", "2", "--warmup", "1", "--ref-seconds", "2"],
                         env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    import json
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
