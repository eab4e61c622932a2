"""The benchmark's output contract, end to end on a GB300: bench.py on the batch-1 workload
prints one JSON line whose figures agree with one another (value = the step's algorithmic
bytes over its time, the roofline fraction = achieved over peak, achieved = the attention's
bytes over its per-launch time), with the end-to-end leg, the oracle baseline and the clock
record present, and the attention timed alone no slower than the whole step."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "b1_h32x8_l2k", "--steps", "20",
           "--warmup", "3", "--no-per-workload", "--cpu-seconds", "0.5"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def close(a, b, rel=1e-9):
    return abs(a - b) <= rel * max(abs(a), abs(b))


def test_contract_keys(line):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 20 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["unit"] == "GB/s" and line["scaling"] == "weak"
    assert line["config"]["workload"] == "b1_h32x8_l2k" and line["data"] == "synthetic"
    assert line["gpu_launches"] == 2 * line["steps"]
    assert line["vs_baseline"] is None


def test_value_is_bytes_over_step_time(line):
    nb = line["config"]["bytes_per_step"]
    assert nb["total"] == nb["kv"] + nb["w_o"] + nb["q_out"]
    assert close(line["value"], nb["total"] / (line["ms_per_step"] * 1e-3) / 1e9)
    assert close(line["config"]["step_hbm_frac"], line["value"] / line["roofline"]["peak"])


def test_roofline_is_achieved_over_peak(line):
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert close(rf["achieved"], rf["algorithmic_bytes_per_launch"] / (rf["us_per_launch"] * 1e-6) / 1e9)
    assert close(rf["frac"], rf["achieved"] / rf["peak"])
    assert rf["traffic"] is None or rf["traffic"] > 0
    # the attention alone (graph replay) is part of the step
    assert rf["us_per_launch"] <= line["ms_per_step"] * 1e3


def test_e2e_and_baseline_legs(line):
    e2e = line["e2e"]
    nb = line["config"]["bytes_per_step"]
    assert e2e["unit"] == "GB/s" and e2e["h2d_bytes_per_step"] >= nb["total"] - nb["q_out"]
    assert e2e["d2h_bytes_per_step"] == 2 * line["config"]["B"] * line["config"]["hidden"]
    assert close(e2e["value"], nb["total"] / (e2e["us_per_step"] * 1e-6) / 1e9, rel=1e-6)
    assert e2e["value"] < line["value"]  # the copies are inside its timed region
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0 and cpu["sample"]


def test_clock_record(line):
    c = line["clocks"]
    assert c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)
