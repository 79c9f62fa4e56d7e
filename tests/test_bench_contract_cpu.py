"""bench.py's reference arm (the oracle timed on the host cores) keeps the JSON-line contract:
one line with the metric, unit and config of the GPU arm, "impl": "reference", a cpu_baseline
describing the run and an e2e block with no host-device bytes; under torchrun only rank 0
prints.  Runs on the CPU in a few seconds."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(args, env=None):
    r = subprocess.run([sys.executable] + args, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=env or os.environ.copy())
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(line) for line in r.stdout.splitlines() if line.startswith("{")]


def test_reference_arm_line():
    lines = run(["bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3"])
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["metric"].startswith("weight-stream GB/s")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def free_port() -> int:
    """A port the kernel hands out as free right now (bound to port 0, then released)."""
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_two_ranks_prints_once():
    env = os.environ.copy()
    env["MASTER_ADDR"] = "127.0.0.1"
    lines = run(["-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                 "--master-port", str(free_port()), "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                 "--warmup", "3"], env=env)
    assert len(lines) == 1 and lines[0]["impl"] == "reference"
