"""Pins for the CPU oracle: checks against facts fixed by the formats and the mathematics.

None of these re-types the oracle's formula.  They compare it with exhaustive
library conversions, hand-derived fixtures, exact rational arithmetic, integer
matmul, closed forms (identity, permutation, all-ones) and invariants (layout,
leading dimension, sampling).  ``tests/test_oracle_mutations.py`` plants
plausible mistakes in a copy of the oracle and shows that these pins catch them.
"""
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from oracle import OR_BF16, OR_COL, OR_F16, OR_F32, OR_ROW
from bf16_tensor_core_gb300 import workloads as W

GOLDEN = Path(__file__).parent / "golden"


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


# ----------------------------------------------------------------------------------------
# decode of the stored operands
# ----------------------------------------------------------------------------------------
def pin_decode_f16_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_f16(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_decode_bf16_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    ref = t.to(torch.float64).numpy()
    got = oracle.decode_bf16(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_decode_f32_sample():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    special = np.array([0, 1, 0x007fffff, 0x00800000, 0x3f800000, 0x7f7fffff, 0x80000001,
                        0x7f800000, 0xff800000], dtype=np.uint32)
    bits = np.concatenate([bits, special])
    with np.errstate(invalid="ignore"):
        ref = bits.view(np.float32).astype(np.float64)
    got = oracle.decode_f32(bits.view(np.float32))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_decode_golden():
    n = 0
    for line in (GOLDEN / "half_decode.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        fmt, hexbits, val = line.split()
        bits = np.array([int(hexbits, 16)], dtype=np.uint16)
        got = (oracle.decode_f16 if fmt == "f16" else oracle.decode_bf16)(bits)[0]
        assert got == float(val), (fmt, hexbits, got, val)
        n += 1
    assert n >= 15


# ----------------------------------------------------------------------------------------
# the product itself
# ----------------------------------------------------------------------------------------
def _read_golden_gemm():
    d = {}
    for line in (GOLDEN / "gemm_small.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key in ("alpha", "beta"):
            d[key] = float(vals[0])
        elif key == "bias":
            d[key] = np.array([float(v) for v in vals[1:]])
        else:
            r, c = int(vals[0]), int(vals[1])
            d[key] = np.array([float(v) for v in vals[2:]]).reshape(r, c)
    return d


def pin_golden_small_gemm():
    g = _read_golden_gemm()
    A = torch.tensor(g["A"]).to(torch.float16)
    B = torch.tensor(g["B"]).to(torch.float16)
    ab = oracle.gemm_ref(2, 2, 3, A, OR_ROW, B, OR_ROW, OR_F16)
    assert np.array_equal(ab, g["AB"])
    Cin = torch.tensor(g["Cin"], dtype=torch.float32)
    bias = torch.tensor(g["bias"], dtype=torch.float32)
    c = oracle.gemm_ref(2, 2, 3, A, OR_ROW, B, OR_ROW, OR_F16, alpha=g["alpha"], beta=g["beta"],
                        Cin=Cin, dtype_cin=OR_F32, bias=bias, dtype_bias=OR_F32)
    assert np.array_equal(c, g["C"])


def pin_identity():
    M, N, K = 37, 29, 45
    B = W.small_ints(K, N, "f16", 1, -200, 200)
    I = W.identity(M, K, "f16")
    c = oracle.gemm_ref(M, N, K, I, OR_ROW, B, OR_ROW, OR_F16)
    expect = np.zeros((M, N))
    expect[: min(M, K)] = _f64(B)[: min(M, K)]
    assert np.array_equal(c, expect)
    A = W.small_ints(M, K, "bf16", 2, -100, 100)
    I2 = W.identity(K, N, "bf16")
    c2 = oracle.gemm_ref(M, N, K, A, OR_ROW, I2, OR_ROW, OR_BF16)
    expect2 = np.zeros((M, N))
    expect2[:, : min(K, N)] = _f64(A)[:, : min(K, N)]
    assert np.array_equal(c2, expect2)


def pin_permutation():
    n, N = 33, 19
    perm = W.permutation(n, 5)
    P = W.permutation_matrix(perm, "f16")
    rng_b = W.generate(W.problem(n, N, n, seed=9))["B"]  # n x N, U[-1,1] f16
    c = oracle.gemm_ref(n, N, n, P, OR_ROW, rng_b, OR_ROW, OR_F16)
    assert np.array_equal(c, _f64(rng_b)[perm.numpy()])
    # A * P permutes columns: (A P)[:, j] = A[:, inv(perm)[j]]
    A = W.generate(W.problem(N, n, n, seed=10))["A"]     # N x n
    c2 = oracle.gemm_ref(N, n, n, A, OR_ROW, P, OR_ROW, OR_F16)
    inv = torch.argsort(perm).numpy()
    assert np.array_equal(c2, _f64(A)[:, inv])


def pin_all_ones():
    M, N, K = 21, 34, 77
    one_a = W.ones(M, K, "f16")
    one_b = W.ones(K, N, "f16")
    c = oracle.gemm_ref(M, N, K, one_a, OR_ROW, one_b, OR_ROW, OR_F16)
    assert np.array_equal(c, np.full((M, N), float(K)))
    B = W.generate(W.problem(M, N, K, seed=11))["B"]
    col_sums = np.array([sum(float(B[k, j]) for k in range(K)) for j in range(N)])
    c2 = oracle.gemm_ref(M, N, K, one_a, OR_ROW, B, OR_ROW, OR_F16)
    assert np.allclose(c2, np.broadcast_to(col_sums, (M, N)), rtol=0, atol=1e-12)
    A = W.generate(W.problem(M, N, K, seed=12))["A"]
    row_sums = np.array([sum(float(A[i, k]) for k in range(K)) for i in range(M)])
    c3 = oracle.gemm_ref(M, N, K, A, OR_ROW, one_b, OR_ROW, OR_F16)
    assert np.allclose(c3, np.broadcast_to(row_sums[:, None], (M, N)), rtol=0, atol=1e-12)


def pin_small_integers_exact():
    for (M, N, K, dt, code) in [(40, 50, 300, "f16", OR_F16), (31, 17, 129, "bf16", OR_BF16)]:
        A = W.small_ints(M, K, dt, 21)
        B = W.small_ints(K, N, dt, 22)
        c = oracle.gemm_ref(M, N, K, A, OR_ROW, B, OR_ROW, code)
        ref = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy()
        assert np.array_equal(c, ref.astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 7), (7, 16, 17), (17, 33, 16), (3, 2, 33)])
def test_brute_force_exact_rational(M, N, K):
    """Tiny shapes: exact rational arithmetic, then one rounding to f64."""
    w = W.problem(M, N, K, alpha=0.75, beta=-1.5, bias=True, seed=M * 100 + N * 10 + K)
    d = W.generate(w)
    c = oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16, alpha=0.75, beta=-1.5,
                        Cin=d["Cin"], dtype_cin=OR_F32, bias=d["bias"], dtype_bias=OR_F32)
    A = [[Fraction(float(v)) for v in row] for row in d["A"].tolist()]
    B = [[Fraction(float(v)) for v in row] for row in d["B"].tolist()]
    Cin = d["Cin"].tolist()
    bias = d["bias"].tolist()
    assert np.all(np.isfinite(c))
    for i in range(M):
        for j in range(N):
            s = sum(A[i][k] * B[k][j] for k in range(K))
            exact = Fraction(0.75) * s + Fraction(-1.5) * Fraction(Cin[i][j]) + Fraction(bias[j])
            assert abs(Fraction(c[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 48) + Fraction(1, 2 ** 80)


def pin_library_matmul_agreement():
    for (M, N, K, dt) in [(64, 80, 96, "f16"), (33, 65, 200, "bf16")]:
        code = OR_F16 if dt == "f16" else OR_BF16
        d = W.generate(W.problem(M, N, K, dtype_in=dt, seed=31))
        c = oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, code)
        ref = _f64(d["A"]) @ _f64(d["B"])
        assert np.allclose(c, ref, rtol=1e-12, atol=1e-12)


def pin_layouts_equivalent():
    M, N, K = 23, 41, 57
    d = W.generate(W.problem(M, N, K, seed=41))
    base = oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16)
    At = d["A"].t().contiguous()   # stored K x M
    Bt = d["B"].t().contiguous()   # stored N x K
    assert np.array_equal(oracle.gemm_ref(M, N, K, At, OR_COL, d["B"], OR_ROW, OR_F16), base)
    assert np.array_equal(oracle.gemm_ref(M, N, K, d["A"], OR_ROW, Bt, OR_COL, OR_F16), base)
    assert np.array_equal(oracle.gemm_ref(M, N, K, At, OR_COL, Bt, OR_COL, OR_F16), base)
    ref = _f64(d["A"]) @ _f64(d["B"])
    assert np.allclose(base, ref, rtol=1e-12, atol=1e-12)


def pin_leading_dimension_padding_not_read():
    M, N, K = 19, 26, 35
    d = W.generate(W.problem(M, N, K, seed=51))
    base = oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16)
    nan = float("nan")
    Ap = torch.full((M, K + 5), nan, dtype=torch.float16)
    Ap[:, :K] = d["A"]
    Bp = torch.full((K, N + 3), nan, dtype=torch.float16)
    Bp[:, :N] = d["B"]
    c = oracle.gemm_ref(M, N, K, Ap, OR_ROW, Bp, OR_ROW, OR_F16)
    assert np.array_equal(c, base)
    Cin = torch.full((M, N + 7), nan, dtype=torch.float32)
    Cin[:, :N] = 1.0
    c2 = oracle.gemm_ref(M, N, K, Ap, OR_ROW, Bp, OR_ROW, OR_F16, beta=1.0, Cin=Cin)
    assert np.array_equal(c2, base + 1.0)


def pin_epilogue_closed_forms():
    M, N, K = 12, 18, 30
    w = W.problem(M, N, K, alpha=0.0, beta=0.5, bias=True, seed=61)
    d = W.generate(w)
    expect = 0.5 * _f64(d["Cin"]) + _f64(d["bias"])[None, :]
    c = oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16, alpha=0.0, beta=0.5,
                        Cin=d["Cin"], bias=d["bias"])
    assert np.array_equal(c, expect)
    # K = 0: the product is empty, C = beta*C_in + bias
    c0 = oracle.gemm_ref(M, N, 0, None, OR_ROW, None, OR_ROW, OR_F16, alpha=2.0, beta=0.5,
                         Cin=d["Cin"], bias=d["bias"])
    assert np.array_equal(c0, expect)
    # beta = 0: C_in is not read, even when it holds NaN
    nanc = torch.full((M, N), float("nan"), dtype=torch.float32)
    c1 = oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16, beta=0.0, Cin=nanc)
    assert np.all(np.isfinite(c1))
    # alpha scales the product only, the bias is added unscaled
    cb = oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16, alpha=-2.0,
                         bias=d["bias"], dtype_bias=OR_F32)
    ab = _f64(d["A"]) @ _f64(d["B"])
    assert np.allclose(cb, -2.0 * ab + _f64(d["bias"])[None, :], rtol=1e-12, atol=1e-12)


def pin_half_cin_and_bias():
    """C_in and bias stored as bf16 (half outputs keep them in the output dtype)."""
    M, N, K = 9, 14, 20
    w = W.problem(M, N, K, dtype_in="bf16", dtype_out="bf16", beta=1.0, bias=True, seed=71)
    d = W.generate(w)
    c = oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_BF16, beta=1.0,
                        Cin=d["Cin"], dtype_cin=OR_BF16, bias=d["bias"], dtype_bias=OR_BF16)
    ref = _f64(d["A"]) @ _f64(d["B"]) + _f64(d["Cin"]) + _f64(d["bias"])[None, :]
    assert np.allclose(c, ref, rtol=1e-12, atol=1e-12)


def pin_sampling_matches_full():
    M, N, K = 50, 60, 70
    d = W.generate(W.problem(M, N, K, seed=81, bias=True))
    full = oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16, bias=d["bias"])
    rows = [0, 7, 49, 13]
    cols = [59, 0, 31]
    assert np.array_equal(oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16,
                                          bias=d["bias"], rows=rows), full[rows])
    assert np.array_equal(oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16,
                                          bias=d["bias"], cols=cols), full[:, cols])
    sub = oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16, bias=d["bias"],
                          rows=rows, cols=cols)
    assert np.array_equal(sub, full[np.ix_(rows, cols)])
    assert np.array_equal(oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16,
                                          bias=d["bias"], nthreads=1), full)


# ----------------------------------------------------------------------------------------
# the pass criterion
# ----------------------------------------------------------------------------------------
def pin_ulp_out():
    assert oracle.ulp_out(1.0, OR_F16) == 2.0 ** -10
    assert oracle.ulp_out(65504.0, OR_F16) == 32.0
    assert oracle.ulp_out(0.0, OR_F16) == 2.0 ** -24
    assert oracle.ulp_out(1.0, OR_BF16) == 2.0 ** -7
    assert oracle.ulp_out(0.0, OR_BF16) == 2.0 ** -133
    assert oracle.ulp_out(-3.0, OR_BF16) == 2.0 ** -6
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-60000, 60000, 5000), rng.uniform(-1e-4, 1e-4, 5000)])
    x16 = x.astype(np.float16)
    x16 = x16[np.isfinite(x16) & (x16 != 0)]
    # numpy's spacing of a binary16 value is one ulp at that value (towards larger magnitude)
    assert np.array_equal(oracle.ulp_out(x16.astype(np.float64), OR_F16),
                          np.abs(np.spacing(np.abs(x16))).astype(np.float64))


def pin_check_catches_planted_errors():
    M, N, K = 16, 24, 64
    d = W.generate(W.problem(M, N, K, dtype_out="f16", bias=True, seed=91))
    ref = oracle.gemm_ref(M, N, K, d["A"], OR_ROW, d["B"], OR_ROW, OR_F16, bias=d["bias"],
                          dtype_bias=OR_F16)
    maxA = float(d["A"].abs().max())
    maxB = float(d["B"].abs().max())
    rounded = torch.tensor(ref).to(torch.float16).to(torch.float64).numpy()
    assert oracle.check(rounded, ref, K, maxA, maxB, OR_F16)["passed"]
    no_bias = rounded - _f64(d["bias"])[None, :]
    assert not oracle.check(no_bias, ref, K, maxA, maxB, OR_F16)["passed"]
    assert not oracle.check(-rounded, ref, K, maxA, maxB, OR_F16)["passed"]
    bad = rounded.copy()
    bad[3, 5] = np.nan
    rep = oracle.check(bad, ref, K, maxA, maxB, OR_F16)
    assert not rep["passed"] and rep["n_nonfinite"] == 1
    shifted = np.roll(rounded, 1, axis=1)
    assert not oracle.check(shifted, ref, K, maxA, maxB, OR_F16)["passed"]


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()
