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


def test_headline_fits_the_stdout_tail():
    """The last stdout line carries every headline key and stays well under the
    1500 characters of stdout that a caller keeping only the tail sees, with
    realistic worst-case field widths."""
    sys.path.insert(0, str(ROOT))
    import bench

    per_m = [{"M": m, "us_per_call": 12345.678, "frac_hbm": 0.123456} for m in range(1, 17)]
    roof = {"bound": "hbm", "achieved": 99999.9, "peak": 6777.6, "unit": "GB/s", "frac": 0.1234,
            "traffic": 14889984.0, "peak_source": "measured", "kernel": "qmm_mma_kernel,qmm_own_kernel,qmm_tma_kernel"}
    cpu = {"value": 0.04062, "unit": "GB/s", "cores": 1, "host_cores": 144, "kind": "oracle",
           "sample": "M=1..16, rows 0..5119 of 5120, 1 thread, 123.4 s"}
    e2e = {"value": 12345.67, "unit": "GB/s", "h2d_bytes_per_step": 1392640, "d2h_bytes_per_step": 1392640}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    line = bench.headline_line(value=123456.78, world=8, steps=20000, warmup=200, ms_per_step=0.123456,
                               workload="m_sweep_5120x5120_4b_g64", shape=(5120, 5120, 4, 64), ncopy=38,
                               copy_mb=560.3, l2_mb=132.1, roofline=roof, per_m=per_m, e2e=e2e, cpu=cpu,
                               launches=320000, clocks=clocks)
    text = json.dumps(line, separators=(",", ":"))
    assert len(text) < 1300, len(text)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "cpu_baseline",
                "gpu_launches", "clocks"):
        assert key in line
    assert line["config"]["workload"] == "m_sweep_5120x5120_4b_g64"
    assert len(line["per_m_us"]) == 16 and len(line["per_m_frac"]) == 16
