"""The benchmark's command line on CPU: the reference arm (the FP64 oracle on the
host cores) prints one JSON line with the contract's keys, for a fixed-layout and
a packed workload, and under a two-process launch only rank 0 prints."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _json_lines(text):
    return [json.loads(l) for l in text.splitlines() if l.startswith("{")]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _check_reference_line(d, workload):
    assert d["impl"] == "reference"
    assert d["config"]["workload"] == workload
    assert d["unit"] == "token·heads/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] >= 3
    assert d["dtype"] == "f64" and d["data"] == "synthetic"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and workload in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("workload", ["fixed_b1_t64_h2", "packed_4x1024_h96"])
def test_reference_arm_prints_one_contract_line(workload):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], workload)


def test_reference_arm_under_two_ranks_prints_once():
    port = _free_port()
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--workload", "fixed_b1_t64_h2", "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], "fixed_b1_t64_h2")
    assert lines[0]["n_gpus"] == 2


def test_algorithmic_bytes():
    """The roofline's compulsory bytes: per token 512 Hqk + 770 Hv forward (q, k, v, g, beta read,
    o written) and 1024 Hqk + 1284 Hv backward (the same reads plus do, the five token gradients
    written), 1536 Hqk + 2054 Hv together; per unit two 64 KiB states each way."""
    sys.path.insert(0, ROOT)
    import bench
    ab = bench.algorithmic_bytes(8192, 96, 96, 768)
    assert ab["fwd"] == 8192 * (512 * 96 + 770 * 96) + 768 * 2 * 65536 == 1_108_869_120
    assert ab["bwd"] == 8192 * (1024 * 96 + 1284 * 96) + 768 * 2 * 65536 == 1_915_748_352
    ab = bench.algorithmic_bytes(55_196, 8, 64, 1536)
    assert ab["fwd"] + ab["bwd"] == 55_196 * (1536 * 8 + 2054 * 64) + 1536 * 262_144
