"""Host-side logic of bench.py that needs no GPU: the algorithmic byte counts behind the roofline and
the lookup of the committed DRAM traffic, which must be withdrawn once the kernel's sources change."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from bf16_tensor_core_gb300 import workloads as W  # noqa: E402


# Least traffic of one product, worked out by hand from each workload's shapes: A and B read once,
# C written once, C_in read when beta != 0, the bias read once (element sizes 2 for f16/bf16,
# 4 for f32, 1 for E4M3, 18 bytes per 32 Q4_0 weights).
@pytest.mark.parametrize("wid, want", [
    (1, 512 * 512 * 2 * 2 + 512 * 512 * 4),                                  # 2,097,152
    (2, 3 * 4096 * 4096 * 2),                                                 # 100,663,296
    (3, 2048 * 4096 * 2 + 4096 * 11008 * 2 + 2048 * 11008 * 2 + 11008 * 2),  # 152,065,536
    (4, 1000 * 2050 * 2 + 2050 * 3000 * 2 + 2 * 1000 * 3000 * 4),            # 40,400,000
    (5, 3 * 8192 * 8192 * 2),                                                 # 402,653,184
    (6, 2048 * 4096 * 2 + 11008 * 128 * 18 + 2048 * 11008 * 2 + 11008 * 2),
    (7, 4096 * 2 + 4096 * 4096 * 2 + 4096 * 2),
    (9, 2 * 4096 * 4096 + 4096 * 4096 * 2),
    (10, 4096 * 2 + 4096 * 128 * 18 + 4096 * 2),
])
def test_algorithmic_bytes(wid, want):
    assert bench.algorithmic_bytes(W.WORKLOADS[wid]) == want


def test_algorithmic_bytes_of_the_gate_workload_match_its_flop_ratio():
    w = W.WORKLOADS[2]
    flops = 2 * w.M * w.N * w.K
    assert round(flops / bench.algorithmic_bytes(w)) == 1365


def _entries():
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for name, v in d.items():
        for e in (v if isinstance(v, list) else [v]):
            yield name, e


def test_traffic_file_entries_are_complete():
    names = {w.name for w in W.WORKLOADS.values()}
    for name, e in _entries():
        assert name in names, name
        assert e["kernel"] in ("gb300::gemm_tc_kernel", "gb300::gemv_kernel", "gb300::gemv_q4_0_kernel")
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
        assert e["gpu_time_ns"] > 0 and len(e["kernel_hash"]) == 16
        assert set(bench.TRAFFIC_PLAN_KEYS) <= set(e["plan"]), e["plan"]
        # The capture command runs committed files only, with the clocks left alone.
        assert "bench.py" in e["source"] and "--clock-control none" in e["source"]


def test_traffic_is_reported_only_for_the_current_kernel_sources_and_schedule(monkeypatch):
    name, e = next((n, e) for n, e in _entries() if n == "gemm_4096_f16_f16")
    real = bench._kernel_hash
    monkeypatch.setattr(bench, "_kernel_hash", lambda kernel="gb300::gemm_tc_kernel": e["kernel_hash"])
    plan = dict(e["plan"], tiles_m=16)                   # fields outside the schedule key do not matter
    got, src = bench._traffic(name, e["kernel"], plan)
    assert got == e["dram_bytes_per_launch"] and "ncu" in src
    # Another config, another schedule of the same config, or changed sources: no figure.
    for k, v in (("config", plan["config"] + 1), ("raster_group", plan["raster_group"] + 1),
                 ("dp_tiles", plan["dp_tiles"] + 1), ("clusters", plan["clusters"] - 1)):
        assert bench._traffic(name, e["kernel"], dict(plan, **{k: v})) == (None, None), k
    monkeypatch.setattr(bench, "_kernel_hash", lambda kernel="gb300::gemm_tc_kernel": "0" * 16)
    assert bench._traffic(name, e["kernel"], plan) == (None, None)
    monkeypatch.setattr(bench, "_kernel_hash", real)


def test_kernel_hash_depends_on_the_kernel_family():
    assert bench._kernel_hash("gb300::gemm_tc_kernel") != bench._kernel_hash("gb300::gemv_kernel")
    assert bench._kernel_hash("gb300::gemv_kernel") == bench._kernel_hash("gb300::gemv_q4_0_kernel")


@pytest.mark.parametrize("wid", [1, 3, 4])
def test_check_rows_accepts_the_rounded_oracle_and_rejects_a_planted_error(wid):
    """The bench's in-line parity check: the oracle's own rows rounded to the output type pass; the
    same rows with one element moved by 10 bounds, or one NaN, fail."""
    import torch
    w = W.WORKLOADS[wid]
    w = W.with_changes(w, M=16, N=min(w.N, 96), K=min(w.K, 256))
    d = W.generate(w)
    rows = 8
    want = {}
    bench.oracle_block_time(w, d, rows, w.N, 2, want)
    ref = want["ref"]
    got = torch.from_numpy(ref.copy()).to(W.DTYPES[w.dtype_out])
    rep = bench.check_rows(w, d, ref, got)
    assert rep["passed"] and rep["n"] == rows * w.N and rep["n_bad"] == 0
    # The stated bound, 1e-4 * K * max|A| * max|B| (scaled by |alpha| > 1), plus a margin of 1 for the
    # output rounding and epilogue terms; the planted error is ten times that.
    bound = 1e-4 * w.K * float(d["A"].float().abs().max()) * float(d["B"].float().abs().max())
    bad = got.clone().to(torch.float64)
    bad[3, 5] += 10.0 * (bound * max(1.0, abs(w.alpha)) + 1.0)
    assert not bench.check_rows(w, d, ref, bad.to(W.DTYPES[w.dtype_out]))["passed"]
    nan = got.clone()
    nan[0, 0] = float("nan")
    assert not bench.check_rows(w, d, ref, nan)["passed"]


def test_nvml_summary_decodes_reasons_inside_the_window():
    s = bench.NvmlSampler.__new__(bench.NvmlSampler)     # no NVML here: fill the samples by hand
    s.max_mhz = 2070
    # (time, SM MHz, watts, reason bits): 0x4 software power cap, 0x8 hardware slowdown (outside the window),
    # 0x40 hardware thermal slowdown, 0x1 idle (not a reported reason)
    s.rows = [(0.5, 1000, 100.0, 0x8), (1.0, 2070, 900.0, 0x0), (1.5, 1900, 1390.0, 0x4), (2.0, 1800, 1300.0, 0x41),
              (3.5, 500, 50.0, 0x8)]
    c = s.summarize(1.0, 2.0)
    assert c["samples"] == 3 and c["sm_mhz"] == 1900 and c["sm_max_mhz"] == 2070 and c["power_w_max"] == 1390.0
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert s.summarize(5.0, 6.0)["samples"] == 0
    # A region shorter than the sampling period (a graph of a few short steps) takes the samples nearest it,
    # within 20 ms, and says so.
    s.rows = [(10.000, 2070, 900.0, 0x0), (10.0005, 2060, 910.0, 0x0), (10.0010, 2050, 920.0, 0x4), (10.5, 1000, 1.0, 0x8)]
    c = s.summarize(10.0006, 10.0008)
    assert c["samples"] == 3 and c["sm_mhz"] == 2060 and c["reasons"] == ["sw_power_cap"] and "window" in c


def test_nvidia_smi_summary_reads_the_active_reasons():
    import datetime
    t = datetime.datetime(2026, 1, 2, 3, 4, 5)
    def row(sec, mhz, hw, hwt, swt, cap):
        ts = (t + datetime.timedelta(seconds=sec)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return [ts, "0", str(mhz), "2070", "700.5", "0x0", hw, hwt, swt, cap]
    rows = [row(0, 2070, "Not Active", "Not Active", "Not Active", "Not Active"),
            row(1, 1500, "Not Active", "Not Active", "Not Active", "Active"),
            row(2, 1400, "Active", "Not Active", "Not Active", "Not Active"),
            row(9, 300, "Not Active", "Active", "Active", "Not Active")]
    t0 = t.timestamp() - 0.5
    c = bench.ClockSampler.summarize(rows, t0, t0 + 3.0)
    assert c["samples"] == 3 and c["sm_mhz"] == 1500 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]


@pytest.mark.parametrize("wid", [4, 6, 10])
def test_cublas_context_declines_products_torch_has_no_single_call_for(wid):
    """The cuBLAS context leg returns None, before touching the device, where torch has no single call for the
    product: Q4_0 weights (6, 10) and 16-bit inputs with another output type (4: f16 in, f32 out)."""
    assert bench.cublas_context(W.WORKLOADS[wid], None, None, None, None, None, 1, 1, None) is None
