"""Benchmark of the GB300 dense GEMM: one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload 1..10]

A step is one gemm_run (the whole hot path: tensor maps, TMA ring, tcgen05 MMAs, epilogue)
over the workload's seeded synthetic inputs.  Default workload: 4096^3, f16 in, f32
accumulate, f16 out.  Two timing protocols, both on the device with CUDA events after W untimed
warm-up steps, the K timed steps bracketed by a barrier and a device synchronise:
  rotate (the headline by default): inputs larger than L2.  The operands (and C) are copied into
    enough sets that one pass over them moves more than 3 x L2, so every step reads its operands
    from HBM; the K steps run back to back from CUDA graphs (one graph per pass over the sets),
    with one event pair around them all, so the per-call host cost is not on the device's clock.
  flush: a 256 MiB write before every step, each step alone between its own two events (the
    launch latency of every step is then part of its time).
The protocol not chosen with --l2 is measured as well and reported under other_protocol.
Several GPUs (torchrun) run independent replicas of the same GEMM: the product has no data
exchange, so there is no collective in the timed path (weak scaling).

--impl reference times the CPU oracle (plain f64 triple loop) on the same workload, one
bounded block of C per step, on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

FLUSH_BYTES = 256 << 20
METRIC = "GEMM TFLOP/s and % of dense f16 tensor roofline at 4096\u00b3 (1\u00d7GB300)"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # 200 steps keep a 4096^3 timed region near 17 ms, inside the time the power cap takes to engage (a
    # 2000-step region, 170 ms, ran 9 % slower under sw_power_cap); the sustained leg reports the capped rate.
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2,
                    help="1..10 (6, 10: Q4_0 weights through gemm_run_q4_0; 7, 8, 10: decode shapes, HBM-bound)")
    ap.add_argument("--config", type=int, default=-1)
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic stream serialization")
    ap.add_argument("--raster-group", type=int, default=0,
                    help="tile rows per raster group (the handle option; 0: the planner's)")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the bench line: every 16-bit config on workloads 1-5 under the rotate protocol, "
                         "the planner's pick marked; one JSON line per (workload, config), then a markdown table")
    ap.add_argument("--sweep-workloads", default="1,2,3,4,5")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0: same as --steps, capped at 200")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--context-cublas", action="store_true",
                    help="also time torch.matmul (cuBLAS) on the same inputs and protocol, as context")
    ap.add_argument("--l2", choices=["rotate", "flush"], default="rotate",
                    help="headline protocol: 'rotate' runs the K steps back to back from CUDA graphs over rotating "
                         "operand sets larger than L2 in all; 'flush' times each step alone after a 256 MiB write. "
                         "The other protocol is always measured too and reported beside the headline.")
    ap.add_argument("--sustained-seconds", type=float, default=4.0,
                    help="back-to-back steps (warm L2) after the timed region, to expose power or thermal limits; "
                         "0 skips them")
    return ap.parse_args()


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _peaks() -> tuple[dict, str]:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return json.loads(p.read_text()), "measured"
        except Exception:
            pass
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _kernel_hash(kernel: str = "gb300::gemm_tc_kernel") -> str:
    """Hash of one kernel's own sources: the tensor-core kernel (its template, PTX wrappers and
    TUs) or the small-M CUDA-core kernels (their file and the helpers they include)."""
    h = hashlib.sha256()
    csrc = ROOT / "bf16_tensor_core_gb300" / "csrc"
    if kernel.startswith("gb300::gemv"):
        files = [csrc / "gemm_gemv.cu", csrc / "q4_block.cuh", csrc / "gemm_kernel.cuh", csrc / "ptx_sm103.cuh"]
    else:
        files = [csrc / "gemm_kernel.cuh", csrc / "ptx_sm103.cuh", *sorted(csrc.glob("gemm_cfg*.cu"))]
    for f in files:
        h.update(f.name.encode())
        h.update(f.read_bytes())
    return h.hexdigest()[:16]


# The schedule fields that decide which operand lines a launch reads; a traffic figure taken under
# another schedule does not describe this launch.
TRAFFIC_PLAN_KEYS = ("config", "clusters", "stream_k", "dp_tiles", "raster_group")


def _traffic(workload_name: str, kernel: str, plan: dict):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, if it was
    taken on that kernel, with the current sources and the same schedule (else None)."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None, None
    try:
        d = json.loads(p.read_text())
        entries = d.get(workload_name) or []
        for e in entries if isinstance(entries, list) else [entries]:   # one entry per kernel and config
            same_plan = all(e.get("plan", {}).get(k) == plan.get(k) for k in TRAFFIC_PLAN_KEYS)
            if e.get("kernel") == kernel and same_plan and e.get("kernel_hash") == _kernel_hash(kernel):
                return e.get("dram_bytes_per_launch"), e.get("source")
    except Exception:
        pass
    return None, None


def _window(rows, ts, t0: float, t1: float, least: int = 3, reach: float = 0.02):
    """The samples inside [t0, t1]; when fewer than `least` fall inside (a region shorter than a few
    sampling periods), the `least` samples nearest the region's middle among those within `reach`
    seconds of it.  Returns (rows, widened)."""
    sel = [r for r in rows if t0 <= ts(r) <= t1]
    if len(sel) >= least:
        return sel, False
    near = [r for r in rows if t0 - reach <= ts(r) <= t1 + reach]
    if len(near) <= len(sel):
        return sel, False
    mid = 0.5 * (t0 + t1)
    return sorted(near, key=lambda r: abs(ts(r) - mid))[:least], True


class NvmlSampler:
    """SM clock, power and clock-event reasons read through NVML (read-only queries) by a thread
    polling every ~0.5 ms, so that even a timed region of a few milliseconds gets samples."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str):
        import ctypes
        import threading
        self.rows = []
        self._stop = threading.Event()
        self._thread = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            dev = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(dev)) != 0:
                return
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            u32, u64 = ctypes.c_uint, ctypes.c_ulonglong
            mx = u32()
            nv.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx))     # 1 = NVML_CLOCK_SM
            self.max_mhz = mx.value

            def run():
                clk, pw, rs = u32(), u32(), u64()
                while not self._stop.is_set():
                    t = time.time()
                    ok = nv.nvmlDeviceGetClockInfo(dev, 1, ctypes.byref(clk)) == 0
                    nv.nvmlDeviceGetPowerUsage(dev, ctypes.byref(pw))
                    reasons_fn(dev, ctypes.byref(rs))
                    if ok:
                        self.rows.append((t, clk.value, pw.value / 1000.0, rs.value))
                    time.sleep(0.0005)
            self._thread = threading.Thread(target=run, daemon=True)
            self._thread.start()
        except Exception:
            self._thread = None

    @property
    def ok(self) -> bool:
        return self._thread is not None

    def stop(self):
        self._stop.set()
        if self._thread:
            self._thread.join(timeout=2)

    def summarize(self, t0: float, t1: float) -> dict:
        sel, widened = _window(self.rows, lambda r: r[0], t0, t1)
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "nvml"}
        reasons = sorted({n for r in sel for bit, n in self.REASONS.items() if r[3] & bit})
        out = {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": self.max_mhz,
               "power_w_max": max(r[2] for r in sel), "reasons": reasons, "samples": len(sel), "source": "nvml"}
        if widened:
            out["window"] = "the timed region was shorter than the sampling period: the 3 samples nearest it"
        return out


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples, kept only inside [t_start, t_end]."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-i", device_id,
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> list[list[str]]:
        if not self.proc:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        return [[c.strip() for c in ln.split(",")] for ln in out.splitlines() if ln.count(",") >= 9]

    @staticmethod
    def summarize(rows, t0: float, t1: float) -> dict:
        stamped = []
        for r in rows:
            try:
                stamped.append((_dt.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp(), r))
            except ValueError:
                continue
        sel = [r for _, r in _window(stamped, lambda x: x[0], t0, t1)[0]]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[2]) for r in sel if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in sel if r[3].replace(".", "").isdigit()]
        pw = [float(r[4]) for r in sel if r[4].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in sel for n, v in zip(names, r[6:10]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(sel)}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (all ranks call it; one process: the value itself)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(flops_per_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job TFLOP/s of `world` independent replicas, each running `steps` steps, timed by the
    slowest rank (weak scaling: the work per rank is fixed)."""
    return world * flops_per_step * steps / max_seconds / 1e12


def algorithmic_bytes(w) -> int:
    """Least traffic of one product: read A and B once, write C once (and read C_in, bias)."""
    ein = 1 if w.dtype_in in ("e4m3", "e5m2") else 2
    eout = 4 if w.dtype_out == "f32" else 2
    b_bytes = w.N * (w.K // 32) * 18 if w.layoutB == "q4_0" else w.K * w.N * ein
    n = w.M * w.K * ein + b_bytes + w.M * w.N * eout
    if w.beta != 0.0:
        n += w.M * w.N * eout
    if w.dist_bias is not None:
        n += w.N * eout
    return n


def _cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_block_time(w, d, rows: int, cols: int, nthreads: int, want=None) -> tuple[float, float]:
    """Time the oracle on the block C[0:rows, 0:cols] (full K).  Returns (seconds, flops); the block
    itself goes to want["ref"] when a dict is passed."""
    import oracle
    A = d["A"][:rows] if w.layoutA == "row" else d["A"][:, :rows].contiguous()
    B = d["B"][:, :cols].contiguous() if w.layoutB == "row" else d["B"][:cols]
    Cin = d["Cin"][:rows, :cols].contiguous() if d["Cin"] is not None else None
    bias = d["bias"][:cols].contiguous() if d["bias"] is not None else None
    code = {"f16": oracle.OR_F16, "bf16": oracle.OR_BF16, "f32": oracle.OR_F32}
    la = oracle.OR_ROW if w.layoutA == "row" else oracle.OR_COL
    t0 = time.perf_counter()
    if w.layoutB == "q4_0":
        ref = oracle.gemm_ref_q4_0(rows, cols, w.K, A, la, d["B"][:cols].numpy(), alpha=w.alpha, beta=w.beta,
                                   Cin=Cin, dtype_cin=code[w.dtype_out], bias=bias, dtype_bias=code[w.dtype_out],
                                   nthreads=nthreads)
    else:
        ref = oracle.gemm_ref(rows, cols, w.K, A, la, B, oracle.OR_ROW if w.layoutB == "row" else oracle.OR_COL,
                              _oracle_code(w.dtype_in),
                              alpha=w.alpha, beta=w.beta, Cin=Cin, dtype_cin=code[w.dtype_out], bias=bias,
                              dtype_bias=code[w.dtype_out], nthreads=nthreads)
    dt = time.perf_counter() - t0
    if want is not None:
        want["ref"] = ref
    return dt, 2.0 * rows * cols * w.K


def _oracle_code(dtype: str) -> int:
    import oracle
    return {"f16": oracle.OR_F16, "bf16": oracle.OR_BF16, "f32": oracle.OR_F32, "e4m3": oracle.OR_E4M3,
            "e5m2": oracle.OR_E5M2}[dtype]


def check_rows(w, d, ref, got) -> dict:
    """The GPU's rows 0..r-1 of C (all columns) against the oracle's, with the tests' element bound."""
    import numpy as np
    import torch

    import oracle
    rows = ref.shape[0]
    got = got.to(torch.float64).numpy()
    maxA = float(d["A"].float().abs().max()) if w.K > 0 else 0.0
    if w.layoutB == "q4_0":
        Wf = oracle.q4_0_to_f16(d["B"].numpy(), w.N, w.K).view(np.float16).astype(np.float64)
        maxB = float(np.abs(Wf).max())
    else:
        maxB = float(d["B"].float().abs().max()) if w.K > 0 else 0.0
    cin = d["Cin"][:rows].to(torch.float64).numpy() if (d["Cin"] is not None and w.beta != 0.0) else None
    bias = d["bias"].to(torch.float64).numpy() if d["bias"] is not None else None
    mag = oracle.epilogue_magnitude(ref, w.beta, cin, bias)
    rep = oracle.check(got, ref, w.K, maxA, maxB, _oracle_code(w.dtype_out), alpha=w.alpha, epi_mag=mag)
    return {"rows": rows, "passed": bool(rep["passed"]), "n": rep["n"], "n_bad": rep["n_bad"],
            "max_abs_err": float(rep.get("max_abs_err", float("nan"))),
            "worst_err_over_bound": float(rep.get("worst_ratio", float("nan")))}


def cpu_baseline(w, d, budget_s: float, gpu_rows=None) -> dict:
    """The oracle as it stands, all host cores, on a bounded block of the workload: whole rows of C
    (all columns, full K), grown until the block takes about half the budget; when even all of C
    takes less, the whole product is repeated to fill the budget.  With gpu_rows(r) (the GPU's
    first r rows of C from one fresh step), the same block is also checked element by element."""
    cores = _cpu_cores()
    rows, cols = min(w.M, cores), w.N
    want = {}
    dt, fl = oracle_block_time(w, d, rows, cols, cores, want)
    while dt < budget_s / 2 and rows < w.M:
        grow = max(2, int(budget_s / 2 / max(dt, 1e-3)))
        rows = min(w.M, rows * grow)
        rows = max(cores, rows - rows % cores) if rows < w.M else rows
        dt, fl = oracle_block_time(w, d, rows, cols, cores, want)
    reps, total_s, total_fl = 1, dt, fl
    while total_s < budget_s / 2:
        dt, fl = oracle_block_time(w, d, rows, cols, cores)
        reps, total_s, total_fl = reps + 1, total_s + dt, total_fl + fl
    what = (f"rows 0..{rows - 1} of {w.M}" if rows < w.M else f"all {w.M} rows") + f" x all {cols} columns, full K={w.K}"
    if reps > 1:
        what += f", {reps} passes"
    out = {"value": total_fl / total_s / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
           "sample": f"{what}; {total_s:.1f} s on {cores} threads", "seconds": total_s}
    if gpu_rows is not None:
        out["check"] = check_rows(w, d, want["ref"], gpu_rows(rows))
    return out


def cublas_context(w, A, B, bias, C, flush, steps, warmup, stream, sets=None):
    """cuBLAS through torch on the same device inputs, timed like our arm: torch.matmul / torch.addmm for
    16-bit inputs, torch._scaled_mm (unit scales, alpha folded into A's scale) for 8-bit ones.  `value` is
    the flush protocol (L2 flushed, CUDA events around each call); with `sets`, `rotate` is the rotate
    protocol (the calls on the rotating operand sets captured in one CUDA graph, replayed back to back).
    Context only: None where torch has no single call for the product (Q4_0 weights, or an output type
    other than the inputs' for 16-bit inputs)."""
    import numpy as np
    import torch
    f8 = w.dtype_in in ("e4m3", "e5m2")
    if w.layoutB == "q4_0" or (not f8 and (w.dtype_in not in ("f16", "bf16") or w.dtype_out != w.dtype_in)):
        return None
    if f8 and (w.beta != 0.0 or w.layoutA != "row" or w.layoutB != "col"):
        return None

    def make_call(A, B, C):
        a = A if w.layoutA == "row" else A.t()
        b = B if w.layoutB == "row" else B.t()
        a, b = a[: w.M, : w.K], b[: w.K, : w.N]
        if f8:                      # row-major A, column-major B (B stored N x K)
            sa = torch.tensor(w.alpha, dtype=torch.float32, device=A.device)
            sb = torch.tensor(1.0, dtype=torch.float32, device=A.device)
            odt = C.dtype
            return lambda: torch._scaled_mm(a, b, sa, sb, bias=bias, out_dtype=odt)
        out = torch.empty(w.M, w.N, dtype=C.dtype, device=C.device)
        cin = C[: w.M, : w.N].clone() if w.beta != 0.0 else None
        if cin is not None:
            return lambda: torch.addmm(cin, a, b, beta=w.beta, alpha=w.alpha, out=out)
        if bias is not None:
            return lambda: torch.addmm(bias, a, b, alpha=w.alpha, out=out)
        if w.alpha == 1.0:
            return lambda: torch.mm(a, b, out=out)
        return lambda: torch.addmm(out, a, b, beta=0.0, alpha=w.alpha, out=out)

    try:
        call = make_call(A, B, C)
        with torch.cuda.stream(stream):
            for _ in range(max(warmup, 3)):
                flush.zero_()
                call()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for e0, e1 in evs:
                flush.zero_()
                e0.record(stream)
                call()
                e1.record(stream)
        torch.cuda.synchronize()
    except (RuntimeError, TypeError) as e:       # e.g. no 8-bit matmul for this device in this torch
        return {"unavailable": f"{type(e).__name__}: {str(e).splitlines()[0][:160]}"}
    ms = float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs]))
    res = {"value": w.flops / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
           "call": ("torch._scaled_mm" if f8 else
                    "torch.addmm" if (w.beta != 0.0 or bias is not None or w.alpha != 1.0) else "torch.mm"),
           "note": "cuBLAS through torch on the same inputs and timing protocols; context, not a baseline"}
    if sets:
        calls = [make_call(bs["A"], bs["B"], bs["C"]) for bs in sets]
        us = graph_step_us(lambda j, st: calls[j](), len(calls))
        res["rotate"] = {"value": w.flops / (us / 1e6) / 1e12, "unit": "TFLOP/s", "us_per_step": us,
                         "sets": len(calls)}
    return res


def _workload(args):
    from bf16_tensor_core_gb300 import workloads as W
    return W.WORKLOADS[args.workload]


def _config_dict(w, args, extra=None) -> dict:
    c = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dtype_in": w.dtype_in, "dtype_out": w.dtype_out,
         "layoutA": w.layoutA, "layoutB": w.layoutB, "alpha": w.alpha, "beta": w.beta,
         "bias": w.dist_bias is not None, "inputs": "seeded synthetic, " + w.note,
         "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}
    if extra:
        c.update(extra)
    return c


# ------------------------------------------------------------------------------------------ reference
def run_reference(args, rank, world):
    if rank != 0:
        return
    from bf16_tensor_core_gb300 import workloads as W
    w = _workload(args)
    d = W.generate(w)
    cores = _cpu_cores()
    total_steps = args.steps + args.warmup
    # Block per step sized so the whole run stays within a few minutes.
    budget = max(0.01, min(2.0, 150.0 / max(total_steps, 1)))
    rows, cols = min(w.M, cores), min(w.N, 256)
    dt, _ = oracle_block_time(w, d, rows, cols, cores)
    while dt < budget / 2 and (rows < w.M or cols < w.N):
        if cols < w.N:
            cols = min(w.N, cols * 2)
        else:
            rows = min(w.M, rows * 2)
        dt, _ = oracle_block_time(w, d, rows, cols, cores)
    while dt > budget and cols > 16:
        cols = max(16, cols // 2)
        dt, _ = oracle_block_time(w, d, rows, cols, cores)
    for _ in range(args.warmup):
        oracle_block_time(w, d, rows, cols, cores)
    tot, flops = 0.0, 0.0
    for _ in range(args.steps):
        t, f = oracle_block_time(w, d, rows, cols, cores)
        tot += t
        flops += f
    value = flops / tot / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": _config_dict(w, args, {"sample_per_step": f"C[0:{rows}, 0:{cols}] with full K={w.K}"}),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"per step the block C[0:{rows}, 0:{cols}], full K={w.K}"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------ sweep
def graph_step_us(step_on, n_sets: int, reps: int = 20) -> float:
    """Mean device time per step of n_sets steps (one per operand set) captured in one CUDA graph and
    replayed `reps` times back to back (the rotate protocol)."""
    import numpy as np
    import torch
    stream = torch.cuda.current_stream()
    for j in range(n_sets):
        step_on(j, stream.cuda_stream)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for j in range(n_sets):
            step_on(j, cap.cuda_stream)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    evs[0].record(stream)
    for i in range(reps):
        graph.replay()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    return float(np.mean([evs[i].elapsed_time(evs[i + 1]) * 1e3 / n_sets for i in range(reps)]))


def run_sweep(args, local):
    """Every 16-bit config (and the planner's automatic choice) on the chosen workloads."""
    import torch

    import __graft_entry__
    from bf16_tensor_core_gb300 import gemm as G
    from bf16_tensor_core_gb300 import workloads as W
    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    l2 = getattr(torch.cuda.get_device_properties(local), "L2_cache_size", 132 << 20)
    configs = [c for c in range(G.gemm_num_configs())
               if G.gemm_config_info(c)[1].in_bytes == 2 and not G.gemm_config_info(c)[1].b_q4_0]
    rows = []
    for wid in [int(x) for x in args.sweep_workloads.split(",")]:
        w = W.WORKLOADS[wid]
        d = W.generate(w)
        A, B = d["A"].to(dev), d["B"].to(dev)
        bias = d["bias"].to(dev) if d["bias"] is not None else None
        C0 = (d["Cin"].to(dev) if d["Cin"] is not None
              else torch.empty(w.M, w.N, dtype=W.DTYPES[w.dtype_out], device=dev))
        n_sets = max(2, min(512, -(-3 * l2 // algorithmic_bytes(w)) + 1))
        sets = [(A, B, C0)] + [(A.clone(), B.clone(), C0.clone()) for _ in range(n_sets - 1)]
        for cfg in [-1] + configs:
            g = G.Gemm(local, config=cfg)

            def step_on(j, st, g=g):
                a, b, c = sets[j]
                g.run(a, b, c, M=w.M, N=w.N, K=w.K, layoutA=w.layoutA, layoutB=w.layoutB, alpha=w.alpha,
                      beta=w.beta, bias=bias, stream=st)
            us = graph_step_us(step_on, n_sets)
            plan = g.last_plan()
            if g.status() != G.GEMM_OK:
                raise RuntimeError(f"sweep: {w.name} config {cfg}: {g.last_error()}")
            g.close()
            row = {"workload": w.name, "config": cfg, "plan_config": plan.get("config"),
                   "stream_k": plan.get("stream_k"), "clusters": plan.get("clusters"), "us_per_step": us,
                   "tflops": w.flops / us / 1e6, "n_sets": n_sets}
            rows.append(row)
            print(json.dumps(row), flush=True)
        del sets
        torch.cuda.empty_cache()
    # the table: one row per workload, one column per config, the planner's pick in bold
    names = sorted({r["workload"] for r in rows}, key=lambda n: [r["workload"] for r in rows].index(n))
    print("| workload | " + " | ".join(f"config {c}" for c in configs) + " | planner |")
    print("|---|" + "---|" * (len(configs) + 1))
    for n in names:
        auto = next(r for r in rows if r["workload"] == n and r["config"] == -1)
        cells = []
        for c in configs:
            r = next(r for r in rows if r["workload"] == n and r["config"] == c)
            cell = f"{r['us_per_step']:.1f} us ({r['tflops']:.0f})"
            cells.append(f"**{cell}**" if c == auto["plan_config"] else cell)
        print(f"| {n} | " + " | ".join(cells) + f" | config {auto['plan_config']}: {auto['us_per_step']:.1f} us |")


# ------------------------------------------------------------------------------------------ ours
def run_ours(args, rank, world, local):
    import numpy as np
    import torch
    import torch.distributed as dist

    import __graft_entry__
    from bf16_tensor_core_gb300 import gemm as G
    from bf16_tensor_core_gb300 import workloads as W

    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = _workload(args)
    d = W.generate(w)
    A = d["A"].to(dev)
    B = d["B"].to(dev)
    bias = d["bias"].to(dev) if d["bias"] is not None else None
    Cin_host = d["Cin"]
    C = (Cin_host.to(dev).clone() if Cin_host is not None
         else torch.empty(w.M, w.N, dtype=W.DTYPES[w.dtype_out], device=dev))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    g = G.Gemm(local, config=args.config, pdl=0 if args.no_pdl else 1, raster_group=args.raster_group)
    stream = torch.cuda.current_stream(dev)
    s_handle = stream.cuda_stream

    def barrier():
        if world > 1:
            dist.barrier()

    # Rotating operand sets: S copies of the inputs (and of C), so that the set a step reads was last
    # touched S - 1 steps earlier, with more than 3 x L2 of other traffic in between: every step reads
    # its operands from HBM without a flush between steps.
    l2_bytes = torch.cuda.get_device_properties(local).L2_cache_size if hasattr(
        torch.cuda.get_device_properties(local), "L2_cache_size") else 132 << 20
    set_bytes = algorithmic_bytes(w)
    n_sets = max(2, min(512, -(-3 * l2_bytes // max(set_bytes, 1)) + 1))
    sets = [dict(A=A, B=B, C=C)]
    for _ in range(n_sets - 1):
        sets.append(dict(A=A.clone(), B=B.clone(), C=C.clone()))

    def step_on(j, st=None):
        bs = sets[j]
        if w.layoutB == "q4_0":
            g.run_q4_0(bs["A"], bs["B"], bs["C"], M=w.M, N=w.N, K=w.K, layoutA=w.layoutA, alpha=w.alpha, beta=w.beta,
                       bias=bias, stream=st)
        else:
            g.run(bs["A"], bs["B"], bs["C"], M=w.M, N=w.N, K=w.K, layoutA=w.layoutA, layoutB=w.layoutB,
                  alpha=w.alpha, beta=w.beta, bias=bias, stream=st)

    def step():
        step_on(0, s_handle)

    # warm-up: every set at least once (workspaces reach their size before any capture)
    for i in range(max(args.warmup, 3, n_sets)):
        flush.zero_()
        step_on(i % n_sets, s_handle)
    torch.cuda.synchronize()
    st = g.status()
    if st != G.GEMM_OK:
        raise RuntimeError(f"warm-up failed: {g.last_error()}")

    # One graph over all sets (a pass), one over the first K % S sets; K steps = K // S passes + the rest.
    n_pass, n_rest = args.steps // n_sets, args.steps % n_sets
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    launches0 = g.launches
    graph_pass = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_pass, stream=cap):
        for j in range(n_sets):
            step_on(j, cap.cuda_stream)
    launches_per_step = (g.launches - launches0) / n_sets
    graph_rest = None
    if n_rest:
        graph_rest = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_rest, stream=cap):
            for j in range(n_rest):
                step_on(j, cap.cuda_stream)
    torch.cuda.synchronize()
    graph_pass.replay()                       # one untimed pass on the graph path
    torch.cuda.synchronize()

    uuid = str(torch.cuda.get_device_properties(local).uuid)
    dev_id = uuid if uuid.startswith("GPU-") else ("GPU-" + uuid)
    nvml = NvmlSampler(dev_id)
    sampler = None if nvml.ok else ClockSampler(dev_id)
    time.sleep(0.3)
    switch = sys.getswitchinterval()
    sys.setswitchinterval(0.0002)          # let the sampler thread run between launches

    def timed_rotate():
        """K steps back to back from the graphs; events between passes give a per-pass distribution."""
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_pass + 2)]
        barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        with torch.cuda.stream(stream):
            evs[0].record(stream)
            for i in range(n_pass):
                graph_pass.replay()
                evs[i + 1].record(stream)
            if graph_rest is not None:
                graph_rest.replay()
            evs[n_pass + 1].record(stream)
        torch.cuda.synchronize()
        barrier()
        t1 = time.time()
        total_ms = evs[0].elapsed_time(evs[n_pass + 1])
        per_step = np.array([evs[i].elapsed_time(evs[i + 1]) / n_sets for i in range(n_pass)])
        if per_step.size == 0:                # fewer steps than operand sets: the rest graph alone
            per_step = np.array([total_ms / args.steps])
        return total_ms, per_step, t0, t1

    def timed_flush():
        """Each step alone between two events, after a 256 MiB write (cold L2, per-step launch cost included)."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        t1 = time.time()
        times = np.array([e0.elapsed_time(e1) for e0, e1 in evs])
        return float(times.sum()), times, t0, t1

    first, second = (timed_rotate, timed_flush) if args.l2 == "rotate" else (timed_flush, timed_rotate)
    total_ms, times_ms, t_start, t_end = first()
    other_ms, other_times, o_start, o_end = second()
    launches = int(round(launches_per_step * args.steps))
    plan = g.last_plan()

    # Sustained: the same step back to back (no flush, warm L2) for a few seconds, so that power or
    # thermal limits show in the clocks.  Reported beside the cold-L2 value, never as it.
    sustained = None
    if args.sustained_seconds > 0:
        batch = max(1, int(0.01 / max(float(np.median(times_ms)) / 1e3, 1e-7)))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts0 = time.time()
        n_sus = 0
        s0.record(stream)
        while time.time() - ts0 < args.sustained_seconds:
            for _ in range(batch):
                step()
            n_sus += batch
            torch.cuda.synchronize()
        s1.record(stream)
        torch.cuda.synchronize()
        ts1 = time.time()
        t_sus = s0.elapsed_time(s1) / 1e3
        sustained = {"seconds": t_sus, "steps": n_sus, "value": w.flops * n_sus / t_sus / 1e12, "unit": "TFLOP/s",
                     "ms_per_step": t_sus / n_sus * 1e3, "l2": "warm: back-to-back steps, no flush (not the headline)"}
    sys.setswitchinterval(switch)
    if sampler is None:
        nvml.stop()
        summarize = nvml.summarize
    else:
        rows = sampler.stop()
        summarize = lambda a, b: ClockSampler.summarize(rows, a, b)
    clocks = summarize(t_start, t_end)
    other_clocks = summarize(o_start, o_end)
    if sustained:
        sustained["clocks"] = summarize(ts0, ts1)
    st = g.status()
    if st != G.GEMM_OK:
        raise RuntimeError(f"timed run failed: {g.last_error()}")
    total_s = max_over_ranks(total_ms / 1e3, world, dev)
    value = replica_throughput(w.flops, args.steps, world, total_s)
    ms_per_step = total_s / args.steps * 1e3
    other_s = max_over_ranks(other_ms / 1e3, world, dev)
    l2_text = {
        "rotate": (f"inputs larger than L2: {n_sets} rotating operand sets (A, B, C and C_in each; "
                   f"{n_sets * set_bytes / 1e6:.0f} MB in all, over 3 x the {l2_bytes / 1e6:.0f} MB L2), no flush"),
        "flush": f"{FLUSH_BYTES >> 20} MiB write between timed steps (cold L2 every step)"}
    timing_text = {
        "rotate": (f"the K steps back to back from CUDA graphs ({n_sets} steps per graph, one per operand set), "
                   "one event pair around all of them on the launching stream"),
        "flush": "CUDA events around each gemm_run on its stream, the flush outside them"}
    other = "flush" if args.l2 == "rotate" else "rotate"
    other_line = {"protocol": other, "value": replica_throughput(w.flops, args.steps, world, other_s),
                  "unit": "TFLOP/s", "ms_per_step": other_s / args.steps * 1e3, "l2": l2_text[other],
                  "timing": timing_text[other],
                  "step_ms": {"mean": float(other_times.mean()), "median": float(np.median(other_times)),
                              "best": float(other_times.min()), "p90": float(np.percentile(other_times, 90))},
                  "clocks": other_clocks}

    # end to end through the public call with host buffers
    e2e = None
    if not args.no_e2e:
        n_e2e = args.e2e_steps or min(args.steps, 200)
        A_pin = d["A"].pin_memory()
        B_pin = d["B"].pin_memory()
        Cin_pin = Cin_host.pin_memory() if Cin_host is not None else None
        C_pin = torch.empty(w.M, w.N, dtype=W.DTYPES[w.dtype_out]).pin_memory()
        h2d = A_pin.numel() * A_pin.element_size() + B_pin.numel() * B_pin.element_size()
        if Cin_pin is not None:
            h2d += Cin_pin.numel() * Cin_pin.element_size()
        d2h = C_pin.numel() * C_pin.element_size()

        # Two device buffer sets on three streams: step k copies its inputs in (H2D stream), runs
        # gemm_run on them (compute stream) and copies C out (D2H stream); events order each set's
        # reuse, so step k+1's copy-in and step k-1's copy-out overlap step k's product.
        e2e_sets = [dict(A=A, B=B, C=C)]
        e2e_sets.append(dict(A=torch.empty_like(A), B=torch.empty_like(B), C=torch.empty_like(C)))
        C_pins = [C_pin, torch.empty_like(C_pin).pin_memory()]
        s_in, s_mm, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()

        def run_set(bs, st):
            if w.layoutB == "q4_0":
                g.run_q4_0(bs["A"], bs["B"], bs["C"], M=w.M, N=w.N, K=w.K, layoutA=w.layoutA, alpha=w.alpha,
                           beta=w.beta, bias=bias, stream=st.cuda_stream)
            else:
                g.run(bs["A"], bs["B"], bs["C"], M=w.M, N=w.N, K=w.K, layoutA=w.layoutA, layoutB=w.layoutB,
                      alpha=w.alpha, beta=w.beta, bias=bias, stream=st.cuda_stream)

        def e2e_steps(n, first_ev=None, last_ev=None):
            done_mm, done_out = [None, None], [None, None]
            for k in range(n):
                j = k % 2
                bs = e2e_sets[j]
                if done_mm[j] is not None:
                    s_in.wait_event(done_mm[j])          # set j's previous product has read A and B
                if done_out[j] is not None:
                    s_in.wait_event(done_out[j])         # ... and its C has been copied out
                if k == 0 and first_ev is not None:
                    first_ev.record(s_in)
                with torch.cuda.stream(s_in):
                    bs["A"].copy_(A_pin, non_blocking=True)
                    bs["B"].copy_(B_pin, non_blocking=True)
                    if Cin_pin is not None:
                        bs["C"].copy_(Cin_pin, non_blocking=True)
                in_done = ev()
                in_done.record(s_in)
                s_mm.wait_event(in_done)
                if done_out[j] is not None:
                    s_mm.wait_event(done_out[j])
                run_set(bs, s_mm)
                done_mm[j] = ev()
                done_mm[j].record(s_mm)
                s_out.wait_event(done_mm[j])
                with torch.cuda.stream(s_out):
                    C_pins[j].copy_(bs["C"], non_blocking=True)
                done_out[j] = ev()
                done_out[j].record(s_out)
            if last_ev is not None:
                s_out.wait_stream(s_in)
                s_out.wait_stream(s_mm)
                last_ev.record(s_out)

        e2e_steps(3)
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_steps(n_e2e, e0, e1)
        torch.cuda.synchronize()
        barrier()
        t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
        e2e = {"value": replica_throughput(w.flops, n_e2e, world, t_e2e), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "note": ("pinned host A, B (and C_in) copied in, gemm_run, C copied out, every step; two device "
                        "buffer sets on three streams (copy-in, product, copy-out) overlap consecutive steps")}

    if rank != 0:
        return
    peaks, src = _peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    peak_note = "cuBLAS bf16 burst (f16 and bf16 share the dense tensor rate)"
    if w.dtype_in in ("e4m3", "e5m2"):       # the FP8 rate: the measured 16-bit peak x the nominal 4.5 / 2.25
        peak *= 2.0
        peak_note = "cuBLAS bf16 burst x 2 (nominal dense FP8 / bf16 rate 4.5 / 2.25 PFLOP/s)"
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    achieved = w.flops / (ms_per_step / 1e3) / 1e12
    n_sms = torch.cuda.get_device_properties(local).multi_processor_count
    alg_bytes = algorithmic_bytes(w)
    if plan.get("gemv"):
        kernel = "gb300::gemv_q4_0_kernel" if w.layoutB == "q4_0" else "gb300::gemv_kernel"
    else:
        kernel = "gb300::gemm_tc_kernel"
    traffic, traffic_src = _traffic(w.name, kernel, plan)
    if w.flops / alg_bytes < peak * 1e12 / (hbm * 1e9):      # below the ridge: the stream of bytes bounds it
        gbs = alg_bytes / (ms_per_step / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": traffic,
                "peak_source": f"{src}: STREAM-style copy", "kernel": kernel,
                "algorithmic_bytes_per_launch": alg_bytes, "algorithmic_flops_per_launch": w.flops,
                "avg_launch_ms": ms_per_step}
    else:
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic,
                "peak_source": f"{src}: {peak_note}",
                "kernel": kernel, "algorithmic_flops_per_launch": w.flops,
                "algorithmic_bytes_per_launch": alg_bytes, "avg_launch_ms": ms_per_step}
    if plan.get("kernels", 1) > 1:
        roof["launches_per_step"] = plan["kernels"]
        roof["note"] = ("avg_launch_ms is the whole step (every launch of the call), so achieved is a lower "
                        "bound for the dominant kernel")
    if traffic is not None:
        roof["traffic_source"] = traffic_src
    if sustained and roof["bound"] == "tensor":
        sp = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1900.0))) * (
            2.0 if w.dtype_in in ("e4m3", "e5m2") else 1.0)
        sustained["peak_sustained"] = sp
        sustained["frac_of_sustained_peak"] = sustained["value"] / sp
    if clocks.get("sm_mhz"):
        clk_peak = 8192.0 * n_sms * clocks["sm_mhz"] * 1e6 / 1e12 * (2.0 if w.dtype_in in ("e4m3", "e5m2") else 1.0)
        roof["clock_roofline_tflops"] = clk_peak
        roof["frac_of_clock_roofline"] = achieved / clk_peak
        roof["clock_roofline_note"] = "8192 dense f16 FLOP/clk/SM x SMs x median SM clock in the timed window"
    line = {"metric": METRIC,
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype_in, "data": "synthetic", "impl": "ours",
            "config": _config_dict(w, args, {"l2": l2_text[args.l2], "kernel_config": plan.get("config", args.config),
                                             "plan": {k: plan[k] for k in ("block_m", "block_n", "block_k", "stages",
                                                                           "tiles_m", "tiles_n", "clusters",
                                                                           "stream_k", "dp_tiles", "raster_group",
                                                                           "transposed", "gemv", "q4_dequant", "kernels")
                                                      if k in plan},
                                             "timing": timing_text[args.l2]}),
            "roofline": roof, "clocks": clocks, "gpu_launches": launches, "e2e": e2e,
            "step_ms": {"mean": float(times_ms.mean()), "median": float(np.median(times_ms)),
                        "best": float(times_ms.min()), "p90": float(np.percentile(times_ms, 90)),
                        "best_value": w.flops / (float(times_ms.min()) / 1e3) / 1e12,
                        "note": ("rank 0's per-step times in the timed region: per graph pass / steps per pass "
                                 "(rotate), or each step's own event pair (flush)")},
            "other_protocol": other_line,
            "sustained": sustained}
    if args.context_cublas:
        line["context_cublas"] = cublas_context(w, A, B, bias, C, flush, args.steps, args.warmup, stream, sets)
    if world == 1 and not args.no_cpu_baseline:
        def gpu_rows(r):
            if Cin_host is not None:
                C.copy_(Cin_host.to(dev))
            step()
            torch.cuda.synchronize()
            return C[:r].cpu()
        line["cpu_baseline"] = cpu_baseline(w, d, args.cpu_seconds, gpu_rows)
    print(json.dumps(line), flush=True)


def main():
    args = _args()
    rank, world, local = _dist()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (torch.cuda.is_available() and args.impl == "ours") else "gloo"
        dist.init_process_group(backend)
    if args.sweep:
        if rank == 0:
            run_sweep(args, int(os.environ.get("LOCAL_RANK", "0")))
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, int(os.environ.get("LOCAL_RANK", "0")))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
