"""The benchmark's CPU-side contract: the reference arm (the oracle timed on
a bounded sample of the headline workload) prints one JSON line with the
keys the line needs, without a GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["rows"] == 4096 and d["config"]["V"] == 131072


def test_cpu_baseline_single_and_row_partitioned():
    # the oracle timed single-threaded and over every host core, on a small
    # bf16 case of the headline's kind
    import bench
    import workloads
    case = workloads.vsweep(V=4096, rows=96)
    b = bench.cpu_baseline(case, 0.5, partitioned_seconds=1.0)
    assert b["kind"] == "oracle" and b["cores"] == 1 and b["value"] > 0
    p = b["row_partitioned"]
    assert p["cores"] == bench.host_cores() >= 1 and p["value"] > 0 and p["unit"] == "GB/s"


def test_gpus_flag_launches_the_ranks_itself():
    # --gpus 2 without a launcher: bench.py starts two ranks itself
    # (torch.distributed.run on 127.0.0.1); the reference arm runs on rank 0
    # only and prints the one line
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"], capture_output=True,
                       text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1 and json.loads(lines[0])["impl"] == "reference"


def test_gpus_flag_must_match_the_launcher_world_size():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT, env=env)
    assert r.returncode != 0 and "WORLD_SIZE is 1" in r.stderr
