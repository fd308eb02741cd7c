"""The benchmark's reference arm (the CPU oracle, as it stands) keeps the
benchmark's output contract: one JSON line with the arm's metric, a
cpu_baseline describing the run and an end-to-end entry with no host-device
bytes.  Under torchrun only rank 0 runs and prints; the other ranks exit 0
without work.  Runs on CPU: the arm uses no GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(stdout):
    return [json.loads(l) for l in stdout.splitlines() if l.strip().startswith("{")]


def _check_line(line, n_gpus, steps, workload):
    assert line["impl"] == "reference"
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["n_gpus"] == n_gpus and line["steps"] == steps and line["warmup"] >= 3
    assert line["dtype"] == "f64" and line["vs_baseline"] is None
    assert line["config"]["workload"].startswith(workload + ":")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["unit"] == line["unit"]
    assert cb["cores"] >= 1 and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("workload", ["decode", "skew"])
def test_reference_arm_prints_one_contract_line(workload):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 1, 1, workload)
    if workload == "skew":
        assert "16 of 4096 tokens" in lines[0]["cpu_baseline"]["sample"]


def test_reference_arm_under_torchrun_runs_on_rank_0_only():
    pytest.importorskip("torch")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 2, 1, "decode")


def test_bench_parity_fields_on_a_stand_in():
    """The benchmark's parity entry compares the step's outputs with the
    oracle's layer by layer: fed the oracle's own outputs rounded to bf16 it
    reports a rounding-sized error and exact routing, and a changed id is seen."""
    torch = pytest.importorskip("torch")
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    kept = []
    base = bench.cpu_baseline("decode", budget_s=2.0, layers=2, keep=kept)
    assert base["kind"] == "oracle" and len(kept) == 2
    outs = [torch.from_numpy(o.astype(np.float32)).to(torch.bfloat16) for _, o, _ in kept]
    ids = [i.copy() for _, _, i in kept]
    p = bench.parity_vs_oracle(outs, ids, kept)
    assert p["layers"] == 2 and p["routing_exact"] is True
    assert 0 < p["max_err_over_rms"] < p["bar"]["max_err_over_rms"]
    assert 0 < p["mean_rel_err"] < p["bar"]["mean_rel_err"]
    ids[1][0, 0] ^= 1
    assert bench.parity_vs_oracle(outs, ids, kept)["routing_exact"] is False
