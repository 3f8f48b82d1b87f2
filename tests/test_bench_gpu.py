"""bench.py on the GPU: one short run, its JSON line checked against the
contract it reports under (keys, units, the arithmetic between them, the
roofline block, the end-to-end block and the clock record).  Timing values
themselves are not judged here, only that they are consistent."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    r = subprocess.run([sys.executable, "bench.py", "--steps", "4", "--warmup", "3",
                        "--no-cpu-baseline", "--no-small-tokens", "--no-other-workloads"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    out = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(out) == 1, r.stdout[-2000:]
    return json.loads(out[0])


def test_contract_keys(line):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 4 and line["warmup"] == 3
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["scaling"] == "weak" and line["dtype"] == "bf16"
    assert line["vs_baseline"] is None
    assert "workload" in line["config"]
    assert line["config"]["S"] == 4096 and line["config"]["H"] == 7168


def test_value_is_step_bytes_over_step_time(line):
    step_bytes = sum(c["algorithmic_bytes"] for k, c in line["per_call"].items()
                     if k in ("plan", "dispatch", "combine"))
    gbs = step_bytes / (line["ms_per_step"] * 1e-3) / 1e9
    assert abs(gbs - line["value"]) <= 1e-6 * line["value"] + 1e-3


def test_roofline_block(line):
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert abs(rf["achieved"] - rf["algorithmic_bytes"] / (rf["us"] * 1e-6) / 1e9) \
        <= 1e-3 * rf["achieved"]
    # the slowest launch of the step cannot be longer than the step
    assert rf["us"] <= line["ms_per_step"] * 1e3
    if rf["traffic"] is not None:
        assert 0.5 * rf["algorithmic_bytes"] < rf["traffic"] < 1.5 * rf["algorithmic_bytes"]


def test_e2e_block(line):
    e = line["e2e"]
    assert e["unit"] == line["unit"]
    S, H, K = 4096, 7168, 8
    assert e["h2d_bytes_per_step"] == S * H * 2 + S * K * 4 + S * K * 4
    assert e["d2h_bytes_per_step"] == S * H * 2
    assert 0 < e["value"] < line["value"]          # the host copies only add time


def test_launches_and_clocks(line):
    # plan, dispatch and combine per timed step at this shape
    assert line["gpu_launches"] == 3 * line["steps"]
    c = line["clocks"]
    assert c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)
