"""Python side of the CPU oracle (test infrastructure only).

``gemm_ref`` calls the plain f64 triple loop in ``gemm_oracle.c`` through
ctypes.  ``check`` applies the pass criterion of the GEMM's accuracy target:

* f32 output:        |C_gpu - C_ref| <= 1e-4 * K * max|A| * max|B|
* f16 / bf16 output: the same bound + one ulp of |C_ref| in the output format

(the accuracy target this library is held to for the dense GEMM C = A*B
with f16/bf16 operands and f32 accumulation that "Optimizing GEMMs using
tcgen05 - Part 2" optimises).  Two readings are added where it is silent:
the bound is multiplied by max(1, |alpha|) (it is stated for alpha = 1), and a
term of 4 f32 ulps of the epilogue's operand magnitude covers the f32
evaluation of alpha*S + beta*C_in + bias, which the statement leaves out and
which matters only when K is 0 or tiny.  The error metrics reported beside it
(largest error / largest entry, relative Frobenius error) are the two used in
"Matrix Multiplication: The Operation Behind Modern AI", section "What the
precision buys, and what it costs".

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from pathlib import Path

import numpy as np

OR_F16, OR_BF16, OR_F32 = 0, 1, 2
OR_E4M3, OR_E5M2 = 3, 4          # 8-bit float inputs (OCP FP8 formats)
OR_ROW, OR_COL = 0, 1

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "gemm_oracle.c"
_LIB = _HERE / "liboracle.so"
_lib = None


def lib_path() -> Path:
    return _LIB


def build(force: bool = False) -> Path:
    """Compile the oracle with the host C compiler (plain -O2, no fast-math)."""
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", str(_SRC), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def configure(lib):
    """Declare the C signatures on a loaded oracle library (also used for test copies)."""
    i64, vp, dbl, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
    lib.oracle_gemm.argtypes = [i64, i64, i64, vp, i64, ci, vp, i64, ci, ci, dbl, dbl,
                                vp, i64, ci, vp, ci, vp, i64, vp, i64, vp, i64, ci]
    lib.oracle_gemm.restype = ci
    lib.oracle_decode_array.argtypes = [vp, ci, i64, vp]
    lib.oracle_decode_array.restype = ci
    lib.oracle_num_cpus.argtypes = []
    lib.oracle_num_cpus.restype = ci
    lib.oracle_f64_to_f16.argtypes = [dbl]
    lib.oracle_f64_to_f16.restype = ctypes.c_uint16
    lib.oracle_q4_0_to_f16.argtypes = [vp, i64, i64, i64, vp, i64]
    lib.oracle_q4_0_to_f16.restype = ci
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = configure(ctypes.CDLL(str(_LIB)))
    return _lib


def num_cpus() -> int:
    """Host cores this process may run on (the oracle's default thread count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return _load().oracle_num_cpus()


def _as_raw(x, dtype_code: int) -> np.ndarray:
    """Return a C-contiguous numpy array holding the stored bits of ``x``.

    ``x`` is a numpy array (uint16 bit patterns for f16/bf16, float32 for f32)
    or a CPU torch tensor of the matching dtype.
    """
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        t = x.detach().contiguous().cpu()
        if dtype_code in (OR_F16, OR_BF16):
            import torch
            return t.view(torch.int16).numpy().view(np.uint16)
        if dtype_code in (OR_E4M3, OR_E5M2):
            import torch
            return t.view(torch.uint8).numpy()
        return t.numpy().astype(np.float32, copy=False)
    a = np.ascontiguousarray(x)
    if dtype_code in (OR_E4M3, OR_E5M2):
        assert a.dtype == np.uint8, "8-bit float inputs are passed as uint8 bit patterns"
    elif dtype_code in (OR_F16, OR_BF16):
        if a.dtype == np.float16:
            a = a.view(np.uint16)
        assert a.dtype == np.uint16, "half inputs are passed as uint16 bit patterns"
    else:
        assert a.dtype == np.float32
    return a


def _decode(x, code: int) -> np.ndarray:
    raw = _as_raw(x, code)
    out = np.empty(raw.shape, dtype=np.float64)
    rc = _load().oracle_decode_array(raw.ctypes.data, code, raw.size, out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_decode_array failed")
    return out


def decode_f16(x) -> np.ndarray:
    return _decode(x, OR_F16)


def decode_bf16(x) -> np.ndarray:
    return _decode(x, OR_BF16)


def decode_f32(x) -> np.ndarray:
    return _decode(x, OR_F32)


def decode(x, code: int) -> np.ndarray:
    return _decode(x, code)


def decode_e4m3(x) -> np.ndarray:
    return _decode(x, OR_E4M3)


def decode_e5m2(x) -> np.ndarray:
    return _decode(x, OR_E5M2)


def gemm_ref(M, N, K, A, layoutA, B, layoutB, dtype_in, *, alpha=1.0, beta=0.0,
             Cin=None, dtype_cin=OR_F32, bias=None, dtype_bias=None,
             rows=None, cols=None, nthreads=0) -> np.ndarray:
    """Unrounded f64 reference of alpha*op(A)*op(B) + beta*C_in + bias.

    Arrays are passed as stored: A ROW (M, lda>=K), A COL (K, lda>=M),
    B ROW (K, ldb>=N), B COL (N, ldb>=K), Cin (M, ldc>=N); the leading dimension
    is each array's second extent.  ``rows`` / ``cols`` select a sub-grid of C
    (None = all).  Returns an f64 array of shape (len(rows), len(cols)).
    """
    lib = _load()
    a = _as_raw(A, dtype_in) if K > 0 else None
    b = _as_raw(B, dtype_in) if K > 0 else None
    lda = a.shape[1] if a is not None else 1
    ldb = b.shape[1] if b is not None else 1
    cin = _as_raw(Cin, dtype_cin) if beta != 0.0 else None
    ldcin = cin.shape[1] if cin is not None else 0
    if bias is not None:
        bias_raw = _as_raw(bias, dtype_bias if dtype_bias is not None else dtype_cin)
        bias_code = dtype_bias if dtype_bias is not None else dtype_cin
    else:
        bias_raw, bias_code = None, 0
    rows_a = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    cols_a = None if cols is None else np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    nr = M if rows_a is None else rows_a.size
    nc = N if cols_a is None else cols_a.size
    out = np.empty((nr, nc), dtype=np.float64)
    ptr = lambda arr: None if arr is None else arr.ctypes.data  # noqa: E731
    rc = lib.oracle_gemm(M, N, K, ptr(a), lda, layoutA, ptr(b), ldb, layoutB, dtype_in,
                         float(alpha), float(beta), ptr(cin), ldcin, dtype_cin,
                         ptr(bias_raw), bias_code,
                         ptr(rows_a), 0 if rows_a is None else rows_a.size,
                         ptr(cols_a), 0 if cols_a is None else cols_a.size,
                         out.ctypes.data, max(nc, 1), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return out


def f64_to_f16_bits(x: float) -> int:
    """binary16 bits of x rounded to nearest, ties to even (the oracle's own encoder)."""
    return int(_load().oracle_f64_to_f16(float(x)))


def q4_0_to_f16(bq, N: int, K: int) -> np.ndarray:
    """Dequantise Q4_0 weights to binary16 bit patterns.

    ``bq``: uint8 array of shape (N, ldbq) holding N rows of K/32 blocks of 18 bytes
    ("02 . 8m/8m(2) -- Tiled wmma f16 prefill GEMM", section 3.2).  Returns (N, K) uint16.
    """
    raw = np.ascontiguousarray(bq if not hasattr(bq, "numpy") else bq.detach().cpu().numpy(), dtype=np.uint8)
    assert raw.ndim == 2 and raw.shape[0] == N
    out = np.empty((N, K), dtype=np.uint16)
    rc = _load().oracle_q4_0_to_f16(raw.ctypes.data if raw.size else None, raw.shape[1], N, K,
                                    out.ctypes.data if out.size else None, K)
    if rc != 0:
        raise ValueError("oracle_q4_0_to_f16 rejected its arguments")
    return out


def gemm_ref_q4_0(M, N, K, A, layoutA, Bq, *, alpha=1.0, beta=0.0, Cin=None, dtype_cin=OR_F32,
                  bias=None, dtype_bias=None, rows=None, cols=None, nthreads=0) -> np.ndarray:
    """Unrounded f64 reference of alpha * A * W^T + beta * C_in + bias, W = dequantised Q4_0
    weights (N x K, f16): the dequantisation followed by the plain GEMM definition."""
    W = q4_0_to_f16(Bq, N, K)
    return gemm_ref(M, N, K, A, layoutA, W, OR_COL, OR_F16, alpha=alpha, beta=beta, Cin=Cin,
                    dtype_cin=dtype_cin, bias=bias, dtype_bias=dtype_bias, rows=rows, cols=cols,
                    nthreads=nthreads)


# --------------------------------------------------------------------------------------
# pass criterion
# --------------------------------------------------------------------------------------
_FMT = {OR_F16: (11, -14), OR_BF16: (8, -126)}  # (precision p, minimum normal exponent)


def ulp_out(x, dtype_out: int) -> np.ndarray:
    """One ulp of |x| in the output format: 2^(max(floor(log2|x|), e_min) - (p-1)).

    ulp_out(0) is the smallest subnormal 2^(e_min - (p-1)).
    """
    p, emin = _FMT[dtype_out]
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(ax)                 # ax = m * 2^e, m in [0.5, 1)  =>  floor(log2 ax) = e - 1
    fl = np.where(ax > 0, e - 1, emin)
    fl = np.maximum(fl, emin)
    return np.ldexp(1.0, (fl - (p - 1)).astype(np.int32))


def tolerance(Cref, K, maxA, maxB, dtype_out, *, alpha=1.0, epi_mag=None) -> np.ndarray:
    """Per-element bound (see module docstring)."""
    Cref = np.asarray(Cref, dtype=np.float64)
    bound = np.full(Cref.shape, 1e-4 * K * maxA * maxB * max(1.0, abs(alpha)))
    mag = np.abs(Cref) if epi_mag is None else epi_mag
    bound = bound + 4.0 * 2.0 ** -24 * mag
    if dtype_out in _FMT:
        bound = bound + ulp_out(Cref, dtype_out)
    return bound


def epilogue_magnitude(Cref, beta=0.0, Cin=None, bias=None) -> np.ndarray:
    """Upper bound of |alpha*S| + |beta*C_in| + |bias| from |C_ref| and the decoded inputs."""
    mag = np.abs(np.asarray(Cref, dtype=np.float64)).copy()
    if beta != 0.0 and Cin is not None:
        mag += 2.0 * np.abs(beta * np.asarray(Cin, dtype=np.float64))
    if bias is not None:
        mag += 2.0 * np.abs(np.asarray(bias, dtype=np.float64))[None, :]
    return mag


def error_metrics(Cgpu, Cref) -> dict:
    Cgpu = np.asarray(Cgpu, dtype=np.float64)
    Cref = np.asarray(Cref, dtype=np.float64)
    err = np.abs(Cgpu - Cref)
    max_ref = float(np.max(np.abs(Cref))) if Cref.size else 0.0
    fro_ref = float(np.linalg.norm(Cref)) if Cref.size else 0.0
    max_err = float(np.max(err)) if err.size else 0.0
    return {
        "max_abs_err": max_err,
        "max_err_over_max_ref": (max_err / max_ref) if max_ref > 0 else max_err,
        "rel_fro": (float(np.linalg.norm(Cgpu - Cref)) / fro_ref) if fro_ref > 0 else max_err,
    }


def check(Cgpu, Cref, K, maxA, maxB, dtype_out, *, alpha=1.0, epi_mag=None) -> dict:
    """Element-by-element pass/fail of a GPU result (already decoded to f64) against Cref."""
    Cgpu = np.asarray(Cgpu, dtype=np.float64)
    Cref = np.asarray(Cref, dtype=np.float64)
    assert Cgpu.shape == Cref.shape, (Cgpu.shape, Cref.shape)
    finite = np.isfinite(Cgpu)
    bound = tolerance(Cref, K, maxA, maxB, dtype_out, alpha=alpha, epi_mag=epi_mag)
    err = np.abs(Cgpu - Cref)
    bad = ~finite | (err > bound)
    rep = error_metrics(np.where(finite, Cgpu, 0.0), Cref)
    rep["n_nonfinite"] = int((~finite).sum())
    rep["n_bad"] = int(bad.sum())
    rep["n"] = int(Cgpu.size)
    ratio = np.where(finite, err / np.maximum(bound, 1e-300), np.inf)
    if ratio.size:
        w = int(np.argmax(ratio))
        rep["worst_index"] = tuple(int(v) for v in np.unravel_index(w, ratio.shape))
        rep["worst_ratio"] = float(ratio.flat[w])
    rep["passed"] = rep["n_bad"] == 0
    return rep


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
