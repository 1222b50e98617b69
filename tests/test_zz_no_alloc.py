"""gemm_run_noalloc against gemm_run, through the C ABI.

gemm_run_noalloc serves callers that cannot allocate device memory (their memory belongs to
another allocator, or cudaMalloc/cudaFree would synchronise a latency-critical loop).  Its
operand repacks go to a fixed file-scope device scratch instead of a handle-owned workspace.
This file is collected last so that a run stopping at the first failure has run every other
test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from bf16_tensor_core_gb300 import gemm as G
from bf16_tensor_core_gb300 import workloads as W
from gpu_cases import OR_CODE, alloc_c, compare, device_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    return G.load_library()


def _ld(t):
    return max(t.stride(0), t.size(1), 1)


def _noalloc(w, dd, C, stream):
    return G.gemm_run_noalloc(w.M, w.N, w.K, dd["A"].data_ptr(), _ld(dd["A"]), dd["B"].data_ptr(), _ld(dd["B"]),
                              C.data_ptr(), _ld(C), G.DTYPE_CODES[w.dtype_in], G.DTYPE_CODES[w.dtype_out],
                              G.LAYOUT_CODES[w.layoutA], G.LAYOUT_CODES[w.layoutB], w.alpha, w.beta,
                              dd["bias"].data_ptr() if dd["bias"] is not None else None, stream)


def _within_tolerance(w, d, got, want):
    """The per-element bound the parity tests use, with gemm_run's output in the place of C_ref."""
    want64 = want[:, : w.N].cpu().to(torch.float64).numpy()
    got64 = got[:, : w.N].cpu().to(torch.float64).numpy()
    cin = d["Cin"].to(torch.float64).numpy() if (d["Cin"] is not None and w.beta != 0.0) else None
    bias = d["bias"].to(torch.float64).numpy() if d["bias"] is not None else None
    mag = oracle.epilogue_magnitude(want64, w.beta, cin, bias)
    return oracle.check(got64, want64, w.K, float(d["A"].abs().max()), float(d["B"].abs().max()),
                        OR_CODE[w.dtype_out], alpha=w.alpha, epi_mag=mag)


def test_noalloc_matches_gemm_run_on_two_calls_in_a_row(lib):
    # Both problems need the scratch: 2050-element (4100-byte) and 1030-element pitches are not
    # multiples of 16 bytes, so their operands are repacked before the product.
    w1 = W.WORKLOADS[4]                                        # 1000 x 3000 x 2050, B stored N x K
    w2 = W.problem(700, 900, 1030, dtype_in="bf16", dtype_out="bf16", layoutA="col", layoutB="row",
                   bias=True, seed=77, name="noalloc_second")   # A stored K x M: lda = 700 (1400 bytes)
    d1, d2 = W.generate(w1), W.generate(w2, ldb=906)            # 906 bf16 = 1812 bytes: repacked
    dd1, dd2 = device_inputs(d1), device_inputs(d2)
    stream = torch.cuda.current_stream().cuda_stream

    with G.Gemm(0) as g:
        ref1, ref2 = alloc_c(w1, d1), alloc_c(w2, d2)
        for w, dd, C in ((w1, dd1, ref1), (w2, dd2, ref2)):
            g.run(dd["A"], dd["B"], C, M=w.M, N=w.N, K=w.K, layoutA=w.layoutA, layoutB=w.layoutB,
                  alpha=w.alpha, beta=w.beta, bias=dd["bias"])
        torch.cuda.synchronize()

    out1, out2 = alloc_c(w1, d1), alloc_c(w2, d2)
    assert _noalloc(w1, dd1, out1, stream) == G.GEMM_OK
    assert _noalloc(w2, dd2, out2, stream) == G.GEMM_OK     # second call reuses the scratch
    assert G.gemm_noalloc_get_device_status(stream) == G.GEMM_OK   # no bounded wait expired
    torch.cuda.synchronize()
    for w, d, got, want in ((w1, d1, out1, ref1), (w2, d2, out2, ref2)):
        rep = compare(w, d, got)                             # every element against the CPU oracle
        assert rep["passed"], (w.name, "oracle", rep)
        rep = _within_tolerance(w, d, got, want)             # and against gemm_run's output
        assert rep["passed"], (w.name, "gemm_run", rep)


def test_noalloc_rejects_repack_beyond_the_scratch(lib):
    # A stored 4100 x 4100 with lda = 4100 f16 (8200-byte pitch) needs 4100 * 4104 * 2 bytes of scratch,
    # more than the 32 MiB the entry point holds.  A, B and C have their full sizes, so the operands a
    # call would read and the output it would write all lie in memory the test owns.
    M, N, K = 4100, 64, 4100
    assert M * 4104 * 2 > (32 << 20)
    A = torch.zeros(M, K, dtype=torch.float16, device="cuda")
    B = torch.zeros(K, N, dtype=torch.float16, device="cuda")
    C = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    st = G.gemm_run_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
                            G.GEMM_F16, G.GEMM_F32, G.GEMM_ROW, G.GEMM_ROW, 1.0, 0.0, None,
                            torch.cuda.current_stream().cuda_stream)
    assert st == G.GEMM_ERR_UNSUPPORTED
    assert G.gemm_noalloc_get_device_status(torch.cuda.current_stream().cuda_stream) == G.GEMM_OK
