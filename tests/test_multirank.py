"""The benchmark's multi-rank path on CPU: two gloo ranks (the data path has
no collective; only the timing is reduced).  Checks that every rank sees the
slowest rank's time, that the job throughput counts every rank's work, that
the column slabs of one GEMM tile its columns exactly, and that the reference
arm runs on rank 0 only."""
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


def _slab_worker(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import gemm_inputs as gi
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rows = []
        for n_total, align in [(8192, 8192 // world), (4100, 256), (1000, 64), (3, 1), (0, 64)]:
            n0, n1 = gi.slab_bounds(n_total, world, rank, align)
            got = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
            dist.all_gather(got, torch.tensor([n0, n1], dtype=torch.int64))
            rows.append(f"{n_total} {align} " + " ".join(f"{int(t[0])}:{int(t[1])}" for t in got))
        # This rank's slab of the 256^3 workload made twice as wide: a
        # fingerprint of its B slab, gathered so the parent can compare.
        case = gi.column_slab_case("s256", world, rank)
        fp = torch.tensor([float(case.B.float().sum()), float(case.B.float()[0, :8].sum())], dtype=torch.float64)
        fps = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(fps, fp)
        rows.append("fp " + " ".join(f"{float(t[0])!r},{float(t[1])!r}" for t in fps))
        with open(os.path.join(out_dir, f"slab{rank}.txt"), "w") as f:
            f.write("\n".join(rows) + "\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_column_slabs_tile_n(tmp_path):
    """Each rank computes its own slab bounds; gathered over gloo, the slabs
    are contiguous, disjoint, in rank order, multiples of the alignment but
    the last, and cover [0, n_total) exactly.  The two ranks draw different
    B slabs, and rank 0's is the single-GPU workload's B."""
    import torch.multiprocessing as mp
    sys.path.insert(0, ROOT)
    import gemm_inputs as gi
    port = _free_port()
    mp.spawn(_slab_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    views = [open(tmp_path / f"slab{r}.txt").read().splitlines() for r in range(2)]
    assert views[0] == views[1]                      # both ranks saw the same gathered bounds
    for line in views[0][:-1]:
        parts = line.split()
        n_total, align = int(parts[0]), int(parts[1])
        bounds = [tuple(int(x) for x in p.split(":")) for p in parts[2:]]
        assert bounds[0][0] == 0 and bounds[-1][1] == n_total
        for (a0, a1), (b0, b1) in zip(bounds, bounds[1:]):
            assert a1 == b0 and a0 <= a1
        for a0, a1 in bounds[:-1]:
            assert a0 % align == 0 and (a1 - a0) % align == 0
    fps = [tuple(float(v) for v in p.split(",")) for p in views[0][-1].split()[1:]]
    assert fps[0] != fps[1]
    b0 = gi.config_case("s256").B.float()
    assert fps[0] == (float(b0.sum()), float(b0[0, :8].sum()))


def test_slab_bounds_rejects_bad_arguments():
    sys.path.insert(0, ROOT)
    import gemm_inputs as gi
    for args in [(10, 0, 0, 1), (10, 2, 2, 1), (10, 2, 0, 0), (-1, 2, 0, 1)]:
        with pytest.raises(ValueError):
            gi.slab_bounds(*args)
