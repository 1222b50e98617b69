"""GPU parity at sizes that stress the index arithmetic: outputs of more than 2^31 elements (TMA-store
and direct-store epilogues), a K of 2^18 (many k-tiles, split K), and small-M products over half a
million weight rows (f16 and Q4_0).  Outputs are checked on sampled rows or columns, computed by the
oracle one by one; the samples include the last row and column."""
import numpy as np
import pytest
import torch

import oracle
from bf16_tensor_core_gb300 import gemm as G
from bf16_tensor_core_gb300 import workloads as W
from gpu_cases import OR_CODE, reference, sample_indices

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _check_sampled(w, d, C, rows=None, cols=None):
    """The GPU's rows (all columns) or columns (all rows) of C against the oracle's."""
    ref = reference(w, d, rows, cols)
    if rows is not None:
        got = C[torch.as_tensor(rows, dtype=torch.long, device=C.device), : w.N]
    else:
        got = C[: w.M, torch.as_tensor(cols, dtype=torch.long, device=C.device)]
    got = got.to(torch.float64).cpu().numpy()
    maxA = float(d["A"].float().abs().max())
    maxB = float(d["B"].float().abs().max())
    rep = oracle.check(got, ref, w.K, maxA, maxB, OR_CODE[w.dtype_out], alpha=w.alpha)
    assert rep["passed"], rep


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M,N,dout,pad", [(49152, 49152, "f16", 0),     # TMA-store epilogue
                                          (49152, 49152, "f16", 1),     # odd pitch: direct stores
                                          (46341, 46344, "f32", 0)])    # 2,147,627,304 f32 elements
def test_output_beyond_2_31_elements(M, N, dout, pad):
    _need_gpu()
    assert M * N > 2 ** 31
    w = W.problem(M, N, 64, dtype_out=dout, bias=True, seed=900 + pad)
    d = W.generate(w)
    A, B, bias = d["A"].cuda(), d["B"].cuda(), d["bias"].cuda()
    C = torch.empty(M, N + pad, dtype=W.DTYPES[dout], device="cuda")
    with G.Gemm(0, sync_check=1) as g:
        g.run(A, B, C[:, :N] if pad else C, M=M, N=N, K=64, bias=bias)
        plan = g.last_plan()
    assert plan["tma_store"] == (0 if pad else 1)
    rows = sorted(set(sample_indices(M, 6, 1, 256)) | {M - 1, M - 2})
    cols = sorted(set(sample_indices(N, 6, 2, 256)) | {N - 1})
    _check_sampled(w, d, C, rows=rows)
    _check_sampled(w, d, C, cols=cols)
    del A, B, C
    _free()


def test_k_of_2_18():
    _need_gpu()
    w = W.problem(256, 256, 1 << 18, dtype_out="f32", seed=910)
    d = W.generate(w)
    C = torch.full((256, 256), float("nan"), dtype=torch.float32, device="cuda")
    with G.Gemm(0, sync_check=1) as g:
        g.run(d["A"].cuda(), d["B"].cuda(), C)
        plan = g.last_plan()
    assert plan["stream_k"] == 1
    _check_sampled(w, d, C, rows=list(range(256)))
    _free()


def test_small_m_half_a_million_rows():
    _need_gpu()
    M, N, K = 3, 1 << 19, 512
    w = W.problem(M, N, K, dtype_out="f32", layoutB="col", seed=920)
    d = W.generate(w)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    with G.Gemm(0, sync_check=1) as g:
        g.run(d["A"].cuda(), d["B"].cuda(), C, layoutB="col")
        assert g.last_plan()["gemv"] == 1
    cols = sorted(set(sample_indices(N, 64, 3, 4096)) | {N - 1})
    _check_sampled(w, d, C, cols=cols)
    _free()


def test_q4_0_small_m_half_a_million_rows():
    _need_gpu()
    M, N, K = 2, 1 << 19, 512
    g0 = torch.Generator().manual_seed(930)
    A = (torch.rand(M, K, generator=g0, dtype=torch.float64) * 2 - 1).half()
    bq = W.q4_0_blocks(N, K, 931)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    with G.Gemm(0, sync_check=1) as g:
        g.run_q4_0(A.cuda(), bq.cuda(), C, N=N)
        assert g.last_plan()["gemv"] == 1
    cols = sorted(set(sample_indices(N, 64, 4, 4096)) | {N - 1})
    ref = oracle.gemm_ref_q4_0(M, N, K, A, oracle.OR_ROW, bq.numpy(), cols=cols)
    got = C[:, torch.as_tensor(cols, dtype=torch.long, device="cuda")].double().cpu().numpy()
    Wf = oracle.q4_0_to_f16(bq[torch.as_tensor(cols)].numpy(), len(cols), K).view(np.float16).astype(np.float64)
    rep = oracle.check(got, ref, K, float(A.abs().max()), float(np.abs(Wf).max()), oracle.OR_F32)
    assert rep["passed"], rep
    _free()
