"""GPU parity of 8-bit float inputs (E4M3, E5M2) multiplied by kind::f8f6f4 MMAs with f32
accumulation, against the oracle's exact decoding of the same bytes."""
import pytest
import torch

from bf16_tensor_core_gb300 import gemm as G
from bf16_tensor_core_gb300 import workloads as W
from gpu_cases import alloc_c, compare, device_inputs, run_gpu, sample_indices

pytestmark = pytest.mark.gpu
F8_CONFIGS = [8, 9, 10]


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _check(w, rows=None, cols=None, **opts):
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d)
    with G.Gemm(0, sync_check=1, **opts) as g:
        run_gpu(g, w, dd, C)
        plan = g.last_plan()
    torch.cuda.synchronize()
    rep = compare(w, d, C, rows, cols)
    assert rep["passed"], rep
    return plan


CASES = [
    dict(M=300, N=520, K=640, dtype_in="e4m3", dtype_out="f16", bias=True),
    dict(M=512, N=512, K=1024, dtype_in="e5m2", dtype_out="f32"),
    dict(M=257, N=300, K=2048, dtype_in="e4m3", dtype_out="bf16", alpha=0.5, beta=1.0),
    dict(M=700, N=260, K=96, dtype_in="e5m2", dtype_out="f32", bias=True),      # one partial k-tile
    dict(M=1000, N=1500, K=4096, dtype_in="e4m3", dtype_out="f32"),
]


@pytest.mark.parametrize("cfg", F8_CONFIGS + [-1])
@pytest.mark.parametrize("i", range(len(CASES)))
def test_fp8_parity(cfg, i):
    _need_gpu()
    c = dict(CASES[i])
    w = W.problem(c.pop("M"), c.pop("N"), c.pop("K"), layoutB="col", seed=700 + 10 * i + max(cfg, 0),
                  dist=("normal", 1.0), **c)
    plan = _check(w, config=cfg, skinny=0 if cfg >= 0 else -1)
    assert G.gemm_config_info(plan["config"])[1].in_bytes == 1


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_small_integers_exact(fmt):
    """Integers in [-3, 3] are exact in both formats; every partial sum is an exact f32 integer."""
    _need_gpu()
    M, N, K = 384, 512, 2048
    A = W.small_ints(M, K, fmt, 41)
    B = W.small_ints(N, K, fmt, 42)                       # stored N x K
    ref = (A.float().to(torch.int64) @ B.float().to(torch.int64).t()).to(torch.float32)
    for sk in (0, 1):
        C = torch.empty(M, N, dtype=torch.float32, device="cuda")
        with G.Gemm(0, sync_check=1, stream_k=sk) as g:
            g.run(A.cuda(), B.cuda(), C, layoutB="col")
        torch.cuda.synchronize()
        assert torch.equal(C.cpu(), ref), (fmt, sk)


def test_fp8_skinny_transposed():
    _need_gpu()
    w = W.problem(16, 4096, 4096, dtype_in="e4m3", dtype_out="f16", layoutB="col", bias=True, seed=750,
                  dist=("normal", 1.0))
    plan = _check(w)
    assert plan["transposed"] == 1


def test_fp8_repacked_rows():
    """1000-byte rows are not a multiple of 16 bytes: both operands go through the repack."""
    _need_gpu()
    w = W.problem(300, 300, 1000, dtype_in="e5m2", dtype_out="f32", layoutB="col", seed=760, dist=("normal", 1.0))
    plan = _check(w)
    assert plan["repack_a"] == 1 and plan["repack_b"] == 1


def test_fp8_4096_sampled():
    _need_gpu()
    w = W.WORKLOADS[9]
    rows = sample_indices(w.M, 32, 1, 256)
    cols = sample_indices(w.N, 32, 2, 256)
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d)
    with G.Gemm(0, sync_check=1) as g:
        run_gpu(g, w, dd, C)
    torch.cuda.synchronize()
    for r, c in ((rows, None), (None, cols)):
        rep = compare(w, d, C, r, c)
        assert rep["passed"], rep


def test_fp8_rejects_mn_major_operands():
    _need_gpu()
    A = torch.zeros(256, 256, dtype=torch.float8_e4m3fn, device="cuda")
    C = torch.zeros(256, 256, dtype=torch.float32, device="cuda")
    with G.Gemm(0) as g:
        assert g.run(A, A, C, layoutB="row", check=False) == G.GEMM_ERR_UNSUPPORTED
