"""Seeded synthetic inputs for the dense GEMM (no GEMM arithmetic lives here).

This module is the one piece both the CUDA path's tests/benchmark and the CPU
oracle's tests use: it only draws and stores input values.  Values are drawn in
f64 on the torch CPU generator and rounded to nearest-even into the stored
dtype; the stored bytes are the inputs both sides read.

The five named workloads follow the shapes, dtypes, layouts and value
distributions of the GEMMs discussed on the pages:
  * 512^3 and 4096^3 / 8192^3 square products ("Optimizing GEMMs using tcgen05 -
    Part 2", section 5 onward, measures 4096^3 fp16),
  * a prefill-shaped 2048 x 11008 x 4096 projection with a per-column bias
    ("02 - Tiled wmma f16 prefill GEMM", sections 1-2: prefill of a 7B model at
    2K tokens; synthetic N(0, 0.02) weights stand in for trained ones),
  * a ragged 1000 x 3000 x 2050 product with B stored transposed (N x K, the NT
    layout of that page's gemm_f16_nt kernel) and alpha/beta on an input C.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
          "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype_in: str = "f16"
    dtype_out: str = "f32"
    layoutA: str = "row"        # row: M x K (K contiguous); col: stored K x M
    layoutB: str = "row"        # row: K x N (N contiguous); col: stored N x K; q4_0: N rows of Q4_0 blocks
    alpha: float = 1.0
    beta: float = 0.0
    dist_a: tuple = ("uniform", -1.0, 1.0)
    dist_b: tuple = ("uniform", -1.0, 1.0)
    dist_bias: tuple | None = None
    dist_cin: tuple | None = None
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def _seed(cfg: int) -> int:
    return 20261202 + 100 * cfg


# The five workloads, in order (index 1..5).
WORKLOADS = {
    1: Workload("gemm_512_f16_f32", 512, 512, 512, "f16", "f32", "row", "row", 1.0, 0.0,
                ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0), None, None, _seed(1),
                "512^3, f16 in U[-1,1], f32 out"),
    2: Workload("gemm_4096_f16_f16", 4096, 4096, 4096, "f16", "f16", "row", "row", 1.0, 0.0,
                ("normal_sqrtk",), ("normal_sqrtk",), None, None, _seed(2),
                "4096^3, f16 in N(0,1)/sqrt(K), f16 out"),
    3: Workload("prefill_2048x11008x4096_bf16_bias", 2048, 11008, 4096, "bf16", "bf16", "row", "row",
                1.0, 0.0, ("normal", 1.0), ("normal", 0.02), ("normal", 0.02), None, _seed(3),
                "prefill projection, bf16 in, bf16 out, fused per-column bias"),
    4: Workload("ragged_1000x3000x2050_nt_f32_ab", 1000, 3000, 2050, "f16", "f32", "row", "col",
                0.5, 1.0, ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0), None, ("uniform", -1.0, 1.0),
                _seed(4), "ragged edges, B stored N x K, alpha=0.5, beta=1 on C_in"),
    5: Workload("gemm_8192_f16_f16", 8192, 8192, 8192, "f16", "f16", "row", "row", 1.0, 0.0,
                ("normal_sqrtk",), ("normal_sqrtk",), None, None, _seed(5),
                "8192^3, f16 in N(0,1)/sqrt(K), f16 out"),
    9: Workload("gemm_4096_e4m3_f16", 4096, 4096, 4096, "e4m3", "f16", "row", "col", 1.0, 0.0,
                ("normal", 1.0), ("normal", 1.0), None, None, _seed(9),
                "4096^3 with E4M3 inputs drawn N(0,1) and rounded to E4M3, K-major A and B (B stored N x K), "
                "f16 out"),
    7: Workload("decode_1x4096x4096_f16", 1, 4096, 4096, "f16", "f16", "row", "col", 1.0, 0.0,
                ("normal", 1.0), ("normal", 0.02), None, None, _seed(7),
                "one token through a 4096 x 4096 f16 weight stored N x K (HBM-bound, intensity ~1 FLOP/B)"),
    8: Workload("decode_64x4096x4096_f16", 64, 4096, 4096, "f16", "f16", "row", "col", 1.0, 0.0,
                ("normal", 1.0), ("normal", 0.02), None, None, _seed(8),
                "64 tokens through a 4096 x 4096 f16 weight stored N x K (HBM-bound)"),
    6: Workload("prefill_2048x11008x4096_q4_0_bias", 2048, 11008, 4096, "f16", "f16", "row", "q4_0",
                1.0, 0.0, ("normal", 1.0), ("q4_0", 0.02), ("normal", 0.02), None, _seed(6),
                "prefill projection with Q4_0 weights (random valid blocks, |w| <= 0.04), f16 activations, "
                "f16 out, fused per-column bias"),
    10: Workload("decode_1x4096x4096_q4_0", 1, 4096, 4096, "f16", "f16", "row", "q4_0", 1.0, 0.0,
                 ("normal", 1.0), ("q4_0", 0.02), None, None, _seed(10),
                 "one token through a 4096 x 4096 weight in Q4_0 blocks (4.5 bits per weight, HBM-bound)"),
}


def _draw(shape, dist, K, g) -> torch.Tensor:
    kind = dist[0]
    if kind == "uniform":
        lo, hi = dist[1], dist[2]
        return torch.rand(shape, generator=g, dtype=torch.float64) * (hi - lo) + lo
    if kind == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float64) * dist[1]
    if kind == "normal_sqrtk":
        return torch.randn(shape, generator=g, dtype=torch.float64) / math.sqrt(max(K, 1))
    raise ValueError(f"unknown distribution {dist}")


def stored_shape_a(w: Workload, lda: int | None = None):
    if w.layoutA == "row":
        return (w.M, lda or w.K)
    return (w.K, lda or w.M)


def stored_shape_b(w: Workload, ldb: int | None = None):
    if w.layoutB == "q4_0":
        return (w.N, ldb or w.K // 32 * Q4_0_BLOCK_BYTES)
    if w.layoutB == "row":
        return (w.K, ldb or w.N)
    return (w.N, ldb or w.K)


def generate(w: Workload, *, lda=None, ldb=None, ldc=None) -> dict:
    """Draw A, B, then bias or C_in (in that order) on the CPU generator seeded with w.seed.

    Returns CPU tensors in the stored layout: A, B (dtype_in; uint8 Q4_0 blocks for layoutB
    "q4_0"), bias (N, dtype_out) or None, Cin (M x ldc, dtype_out) or None.  Padding columns of a wider leading
    dimension are drawn too (their values never enter the product).
    """
    g = torch.Generator().manual_seed(w.seed)
    din = DTYPES[w.dtype_in]
    dout = DTYPES[w.dtype_out]
    A = _draw(stored_shape_a(w, lda), w.dist_a, w.K, g).to(din)
    if w.layoutB == "q4_0":     # uint8 blocks from their own generator (seed + 1)
        B = q4_0_blocks(w.N, w.K, w.seed + 1, ldbq=ldb, scale=w.dist_b[1])
    else:
        B = _draw(stored_shape_b(w, ldb), w.dist_b, w.K, g).to(din)
    bias = _draw((w.N,), w.dist_bias, w.K, g).to(dout) if w.dist_bias else None
    Cin = _draw((w.M, ldc or w.N), w.dist_cin, w.K, g).to(dout) if w.dist_cin else None
    return {"A": A, "B": B, "bias": bias, "Cin": Cin}


def problem(M, N, K, *, dtype_in="f16", dtype_out="f32", layoutA="row", layoutB="row",
            alpha=1.0, beta=0.0, bias=False, seed=1, name="problem",
            dist=("uniform", -1.0, 1.0)) -> Workload:
    """An ad-hoc workload (tail sweeps, layout and dtype coverage)."""
    return Workload(name, M, N, K, dtype_in, dtype_out, layoutA, layoutB, alpha, beta,
                    dist, dist, dist if bias else None, dist if beta != 0.0 else None, seed)


def with_changes(w: Workload, **kw) -> Workload:
    return replace(w, **kw)


# ----------------------------------------------------------------------------------------
# structured inputs whose products have closed forms (used by exactness tests)
# ----------------------------------------------------------------------------------------
def identity(rows: int, cols: int, dtype: str) -> torch.Tensor:
    """rows x cols partial identity: 1 where i == j."""
    t = torch.zeros(rows, cols, dtype=torch.float64)
    n = min(rows, cols)
    t[torch.arange(n), torch.arange(n)] = 1.0
    return t.to(DTYPES[dtype])


def permutation(n: int, seed: int) -> torch.Tensor:
    """A random permutation of range(n) (int64)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randperm(n, generator=g)


def permutation_matrix(perm: torch.Tensor, dtype: str) -> torch.Tensor:
    """P with P[i, perm[i]] = 1, so (P @ X)[i] = X[perm[i]]."""
    n = perm.numel()
    t = torch.zeros(n, n, dtype=torch.float64)
    t[torch.arange(n), perm] = 1.0
    return t.to(DTYPES[dtype])


def ones(rows: int, cols: int, dtype: str) -> torch.Tensor:
    return torch.ones(rows, cols, dtype=DTYPES[dtype])


def small_ints(rows: int, cols: int, dtype: str, seed: int, lo: int = -3, hi: int = 3) -> torch.Tensor:
    """Integers uniform in [lo, hi] (exact in f16 and bf16)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (rows, cols), generator=g, dtype=torch.int64).to(DTYPES[dtype])


# ----------------------------------------------------------------------------------------
# Q4_0-quantised weights (bytes only: the dequantisation itself is the method's, not here)
# ----------------------------------------------------------------------------------------
Q4_0_BLOCK_BYTES = 18      # f16 scale + 16 bytes of nibbles per 32 weights


def q4_0_blocks(N: int, K: int, seed: int, *, ldbq: int | None = None, scale: float = 0.02) -> torch.Tensor:
    """N rows of K/32 random valid Q4_0 blocks as a uint8 tensor of shape (N, ldbq).

    Block layout ("02 . 8m/8m(2) -- Tiled wmma f16 prefill GEMM", section 3.2): a little-endian
    f16 scale d, then 16 bytes whose nibbles are the quantised weights.  d is drawn U[-2s, 2s] / 8
    in f64 and rounded to f16, so |d * (q - 8)| <= 2 s stays far inside f16 (the page's test
    draws "small d" for the same reason); nibbles are uniform in 0..15.  Padding bytes of a wider
    pitch are drawn too (never read).
    """
    assert K % 32 == 0
    nb = K // 32
    pitch = ldbq or nb * Q4_0_BLOCK_BYTES
    assert pitch >= nb * Q4_0_BLOCK_BYTES
    g = torch.Generator().manual_seed(seed)
    raw = torch.randint(0, 256, (N, pitch), generator=g, dtype=torch.int64).to(torch.uint8)
    d = ((torch.rand((N, nb), generator=g, dtype=torch.float64) * 4.0 - 2.0) * scale / 8.0).to(torch.float16)
    dbits = d.view(torch.int16).to(torch.int64) & 0xFFFF
    blocks = raw[:, :nb * Q4_0_BLOCK_BYTES].reshape(N, nb, Q4_0_BLOCK_BYTES).clone()
    blocks[:, :, 0] = (dbits & 0xFF).to(torch.uint8)
    blocks[:, :, 1] = (dbits >> 8).to(torch.uint8)
    raw[:, :nb * Q4_0_BLOCK_BYTES] = blocks.reshape(N, nb * Q4_0_BLOCK_BYTES)
    return raw
