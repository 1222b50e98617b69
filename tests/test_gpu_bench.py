"""bench.py end to end on the GPU, on the small workload: one JSON line with every key its readers use
(roofline, clocks, end-to-end leg, launch count, CPU baseline), consistent with itself."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def line():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "1", "--steps", "20", "--warmup", "3",
           "--sustained-seconds", "0", "--cpu-seconds", "1", "--e2e-steps", "5"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    return json.loads(lines[0])


def test_bench_line_has_the_contract_keys(line):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "clocks", "e2e", "gpu_launches", "cpu_baseline"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 20 and line["warmup"] >= 3
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["config"]["workload"] == "gemm_512_f16_f32"


def test_bench_value_matches_its_step_time(line):
    flops = 2.0 * 512 ** 3
    assert line["value"] > 0
    assert line["value"] == pytest.approx(flops / (line["ms_per_step"] * 1e-3) / 1e12, rel=1e-6)


def test_bench_roofline_and_clocks(line):
    r = line["roofline"]
    assert r["bound"] in ("hbm", "tensor") and r["peak"] > 0 and r["unit"] in ("GB/s", "TFLOP/s")
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-6)
    assert "traffic" in r and (r["traffic"] is None or r["traffic"] > 0)
    c = line["clocks"]
    assert c["sm_max_mhz"] > 0 and 0 < c["sm_mhz"] <= c["sm_max_mhz"] and isinstance(c["reasons"], list)


def test_bench_launches_e2e_and_cpu_baseline(line):
    # One launch of this library per timed step at least (the 512^3 product is one kernel).
    assert line["gpu_launches"] >= line["steps"]
    e = line["e2e"]
    assert e["value"] > 0 and e["unit"] == line["unit"]
    assert e["h2d_bytes_per_step"] == 2 * 512 * 512 * 2 and e["d2h_bytes_per_step"] == 512 * 512 * 4
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    assert cb["check"]["passed"]
