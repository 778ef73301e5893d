"""The benchmark's GPU arm on a small workload: one JSON line carrying every key
of the contract (roofline, CPU baseline, end-to-end leg, clocks, launch count),
for a fixed-layout and a packed workload."""

import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


@pytest.mark.parametrize("workload,units,launches", [("fixed_b1_t64_h2", 2, 3), ("packed_24mixed_hqk8_hv64", 1536, 4)])
def test_bench_line_contract(workload, units, launches):
    args = [sys.executable, "bench.py", "--workload", workload, "--steps", "3", "--warmup", "3"]
    if units > 100:
        args.append("--no-cpu-baseline")  # the oracle sample of the large workload takes ~10 s
    r = subprocess.run(args, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["config"]["workload"] == workload and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "token·heads/s" and d["higher_is_better"] is True
    assert d["ms_per_step"] > 0 and d["scaling"] == "weak" and d["data"] == "synthetic"
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    assert rf["kernel"] in ("kda_fwd_kernel", "kda_bwd_kernel")
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    assert d["gpu_launches"] == launches * 3
    if units <= 100:
        cb = d["cpu_baseline"]
        assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and workload in cb["sample"]
