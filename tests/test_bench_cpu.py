"""bench.py on the CPU: the multi-rank timing helpers over gloo (world size 2)
and the reference arm's JSON line, alone and under torchrun.  No GPU."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    import torch.distributed as dist

    sys.path.insert(0, str(ROOT))
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        got = bench.max_over_ranks(float(rank + 1) * 1.5, world)  # each rank's own timing
        bench.barrier(world)
        Path(out_dir, f"rank{rank}.json").write_text(json.dumps({"max": got}))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    """Every rank gets the slowest rank's time (the bench's max over ranks)."""
    import torch.multiprocessing as mp

    port = free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert json.loads(Path(tmp_path, f"rank{r}.json").read_text())["max"] == pytest.approx(3.0)


def _check_reference_line(line: dict):
    assert line["impl"] == "reference"
    assert line["metric"].startswith("weight GB/s")
    assert line["unit"] == "GB/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["dtype"] == "f64" and line["data"] == "synthetic"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["cpu_baseline"]["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "m_sweep_5120x5120_4b_g64"


def test_reference_arm_json_line():
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1",
                          "--ref-budget", "2"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    _check_reference_line(json.loads(lines[0]))


def test_reference_arm_under_torchrun_world2():
    """Rank 0 alone prints the line; the other rank exits 0 without work."""
    port = free_port()
    res = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                          "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
                          "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-budget", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    _check_reference_line(line)
    assert line["n_gpus"] == 2
