"""The benchmark's reference arm on CPU: `bench.py --impl reference` times the
float64 oracle on a bounded sample and prints one JSON line with the keys the
benchmark contract fixes (the same metric, unit and config as the GPU arm,
an e2e object with zero copy bytes and a cpu_baseline describing the run)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["1", "7", "9"])
def test_reference_arm_prints_the_contract_line(workload):
    d = _run("--impl", "reference", "--workload", workload, "--steps", "3", "--warmup", "3")
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["unit"] == "KV-tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    kv = {"1": "bf16", "7": "fp4", "9": "fp4v41"}[workload]
    assert d["config"]["kv_dtype"] == kv


def test_gpus_flag_must_match_the_launchers_world_size():
    # a launcher that started one rank while --gpus says two is an error, not
    # a silent one-GPU run
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "LOCAL_RANK")}
    env["WORLD_SIZE"] = "1"
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--workload", "1",
                        "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=env)
    assert r.returncode != 0
    assert "WORLD_SIZE=1" in r.stderr


def test_gpus_flag_without_a_launcher_starts_its_own_ranks():
    # --gpus 2 with no launcher: bench.py re-starts itself under
    # torch.distributed.run with two ranks (gloo here); the ranks' own world
    # size check passes only if both were started, and rank 0 alone prints
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--workload", "1",
                        "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["impl"] == "reference"


def test_two_ranks_through_torchrun_print_one_line():
    # the launcher the N>1 contract names (gloo on this CPU host): two ranks
    # start, rank 0 alone prints, both exit 0
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--gpus", "2", "--workload", "1", "--steps", "3", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["impl"] == "reference"
