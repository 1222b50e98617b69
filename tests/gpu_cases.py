"""Shared helpers of the GPU tests: run one GEMM through the C ABI and compare it with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bf16_tensor_core_gb300 import gemm as G
from bf16_tensor_core_gb300 import workloads as W

OR_CODE = {"f16": oracle.OR_F16, "bf16": oracle.OR_BF16, "f32": oracle.OR_F32, "e4m3": oracle.OR_E4M3,
           "e5m2": oracle.OR_E5M2}
OR_LAYOUT = {"row": oracle.OR_ROW, "col": oracle.OR_COL}


def device_inputs(d: dict) -> dict:
    return {k: (v.cuda() if v is not None else None) for k, v in d.items()}


def alloc_c(w: W.Workload, d: dict, ldc: int | None = None, fill: float = float("nan")) -> torch.Tensor:
    ldc = ldc or w.N
    if d.get("Cin") is not None:
        C = d["Cin"].cuda().contiguous()
        if C.size(1) != ldc:
            Cp = torch.full((w.M, ldc), fill, dtype=C.dtype, device="cuda")
            Cp[:, : C.size(1)] = C
            C = Cp
        return C
    return torch.full((w.M, ldc), fill, dtype=W.DTYPES[w.dtype_out], device="cuda")


def run_gpu(g: G.Gemm, w: W.Workload, d_dev: dict, C: torch.Tensor, stream=None) -> None:
    g.run(d_dev["A"], d_dev["B"], C, M=w.M, N=w.N, K=w.K, layoutA=w.layoutA, layoutB=w.layoutB,
          alpha=w.alpha, beta=w.beta, bias=d_dev["bias"], stream=stream)


def reference(w: W.Workload, d: dict, rows=None, cols=None) -> np.ndarray:
    return oracle.gemm_ref(w.M, w.N, w.K, d["A"], OR_LAYOUT[w.layoutA], d["B"], OR_LAYOUT[w.layoutB],
                           OR_CODE[w.dtype_in], alpha=w.alpha, beta=w.beta, Cin=d["Cin"],
                           dtype_cin=OR_CODE[w.dtype_out], bias=d["bias"], dtype_bias=OR_CODE[w.dtype_out],
                           rows=rows, cols=cols)


def compare(w: W.Workload, d: dict, C_out: torch.Tensor, rows=None, cols=None) -> dict:
    """Element-by-element check of the GPU output (rows x cols sub-grid) against the oracle."""
    ref = reference(w, d, rows, cols)
    got = C_out[:, : w.N].cpu()
    if rows is not None:
        got = got[torch.as_tensor(rows, dtype=torch.long)]
    if cols is not None:
        got = got[:, torch.as_tensor(cols, dtype=torch.long)]
    got = got.to(torch.float64).numpy()
    maxA = float(d["A"].float().abs().max()) if w.K > 0 else 0.0
    maxB = float(d["B"].float().abs().max()) if w.K > 0 else 0.0
    cin = None
    if d["Cin"] is not None and w.beta != 0.0:
        cin = d["Cin"][:, : w.N]
        if rows is not None:
            cin = cin[torch.as_tensor(rows, dtype=torch.long)]
        if cols is not None:
            cin = cin[:, torch.as_tensor(cols, dtype=torch.long)]
        cin = cin.to(torch.float64).numpy()
    bias = None
    if d["bias"] is not None:
        bias = d["bias"].to(torch.float64).numpy()
        if cols is not None:
            bias = bias[np.asarray(cols)]
    mag = oracle.epilogue_magnitude(ref, w.beta, cin, bias)
    return oracle.check(got, ref, w.K, maxA, maxB, OR_CODE[w.dtype_out], alpha=w.alpha, epi_mag=mag)


def sample_indices(n: int, count: int, seed: int, tile: int = 128) -> list[int]:
    """Random indices plus every tile boundary (multiples of `tile`, +-1) and the last index."""
    rng = np.random.default_rng(seed)
    s = set(int(x) for x in rng.choice(n, size=min(count, n), replace=False))
    for b in range(0, n + tile, tile):
        for x in (b - 1, b, b + 1):
            if 0 <= x < n:
                s.add(x)
    s.add(n - 1)
    return sorted(s)
