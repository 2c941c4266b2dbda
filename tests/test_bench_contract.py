"""The benchmark's output contract, checked on the CPU through its reference arm (the fp64 oracle
timed on the host cores): one JSON line with the required keys, printed by rank 0 alone when the
script runs as several ranks (gloo; the other ranks exit 0 without printing)."""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]
REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches")


def _env():
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""  # the reference arm needs no GPU; keep the ranks on gloo
    env["PYTHONPATH"] = str(ROOT) + os.pathsep + env.get("PYTHONPATH", "")
    return env


def _json_lines(out):
    return [json.loads(line) for line in out.splitlines() if line.startswith("{")]


def _check_line(line, n):
    for key in REQUIRED:
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["n_gpus"] == n and line["steps"] == 1 and line["warmup"] == 3
    assert line["value"] > 0 and line["higher_is_better"] is True and line["vs_baseline"] is None
    assert line["config"]["workload"] == "tiny_f32"
    # the GPU arm prints the same object (bench.workload_config), so the two lines compare
    sys.path.insert(0, str(ROOT))
    import bench
    from preconditioned_delta_rule_gb300 import workloads as W
    assert line["config"] == json.loads(json.dumps(bench.workload_config(W.WORKLOADS["tiny_f32"])))
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_one_line():
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-budget", "0.3",
           "--workload", "tiny_f32"]
    p = subprocess.run(cmd, cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = _json_lines(p.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 1)


def test_reference_arm_under_two_ranks():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--ref-budget", "0.3", "--workload", "tiny_f32"]
    p = subprocess.run(cmd, cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = _json_lines(p.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 2)
