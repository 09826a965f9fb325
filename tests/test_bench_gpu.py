"""The benchmark's JSON line on a short run (GPU required): every key the
output contract names is present and consistent — the metric's value and
unit, the kernel roofline against the measured peaks, the end-to-end figure
through the host-buffer call with its copied bytes, the CPU oracle baseline,
the sampled clocks and the launch count — for the two-token headline step
and one one-token workload timed alongside it."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5", "--warmup", "3", "--also", "uniform_b32",
           "--no-absorb", "--no-indexer", "--cpu-budget", "1", "--cpu-budget-other", "0.5", "--e2e-steps", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]  # one JSON line, from rank 0
    return json.loads(lines[0])


def test_headline_keys_and_values(line):
    for k in ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches",
              "clocks"]:
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 5 and line["warmup"] == 3
    assert line["unit"] == "TFLOP/s" and line["value"] > 0 and line["ms_per_step"] > 0
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["data"] == "synthetic"
    assert line["config"]["workload"] == "mtp_b64" and line["config"]["batch"] == 64
    assert line["gpu_launches"] > 0


def test_roofline_block(line):
    rf = line["roofline"]
    assert rf["bound"] in ("hbm", "tensor") and rf["unit"] in ("GB/s", "TFLOP/s")
    assert rf["peak"] > 0 and 0 < rf["frac"] < 1.5
    assert abs(rf["achieved"] / rf["peak"] - rf["frac"]) < 1e-9
    assert rf["traffic"] is None or rf["traffic"] > 0


def test_e2e_cpu_baseline_and_clocks(line):
    e = line["e2e"]
    assert e["value"] > 0 and e["unit"] == line["unit"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["value"] < line["value"]  # host copies are inside its timed region
    c = line["cpu_baseline"]
    assert c["kind"] == "oracle" and c["value"] > 0 and c["cores"] >= 1 and c["sample"]
    cl = line["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(cl)


def test_other_workloads_are_timed_alongside(line):
    other = line["other_workloads"]["uniform_b32"]
    assert other["us_per_call"] > 0 and other["us_decode_kernel"] > 0
    assert other["roofline"]["bound"] == "hbm" and 0 < other["roofline"]["frac"] < 1.5
    assert other["cpu_baseline"]["value"] > 0
