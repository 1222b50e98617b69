"""GPU parity of skinny products (few rows of C against many columns), computed as C^T =
op(B)^T op(A)^T so that C's columns fill the long side of the tile ("Matrix Multiplication: The
Operation Behind Modern AI", section "The shape a language model actually runs": an M x 4096 by
4096 x 4096 product with M from 1 to 64)."""
import pytest
import torch

from bf16_tensor_core_gb300 import gemm as G
from bf16_tensor_core_gb300 import workloads as W
from gpu_cases import alloc_c, compare, device_inputs, run_gpu

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _check(w, **opts):
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d)
    with G.Gemm(0, sync_check=1, **opts) as g:
        run_gpu(g, w, dd, C)
        plan = g.last_plan()
    torch.cuda.synchronize()
    rep = compare(w, d, C)
    assert rep["passed"], rep
    return plan, C


CASES = [
    dict(M=1, N=4096, K=4096, dtype_out="f16", layoutB="col"),            # one token, weights N x K
    dict(M=7, N=3000, K=2048, dtype_out="f32", layoutB="row", bias=True),
    dict(M=16, N=4100, K=1000, dtype_out="bf16", dtype_in="bf16", layoutB="col", bias=True),
    dict(M=33, N=1000, K=512, dtype_out="f32", layoutA="col", alpha=0.5, beta=1.0),
    dict(M=64, N=4096, K=4096, dtype_out="f16", layoutB="col"),
    dict(M=64, N=520, K=200, dtype_out="f32", layoutA="col", layoutB="row", bias=True, alpha=-2.0, beta=0.25),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_skinny_parity_automatic(i):
    _need_gpu()
    c = dict(CASES[i])
    w = W.problem(c.pop("M"), c.pop("N"), c.pop("K"), seed=300 + i, **c)
    plan, _ = _check(w)
    # M <= 8 with A row-major and B stored N x K takes the CUDA-core kernel, otherwise C^T
    assert (plan["transposed"] == 1 and plan["tma_store"] == 0) or plan["gemv"] == 1


@pytest.mark.parametrize("i", [1, 3, 5])
def test_skinny_off_gives_the_plain_product(i):
    _need_gpu()
    c = dict(CASES[i])
    w = W.problem(c.pop("M"), c.pop("N"), c.pop("K"), seed=400 + i, **c)
    plan, _ = _check(w, skinny=0)
    assert plan["transposed"] == 0


@pytest.mark.parametrize("cfg", [0, 2, 4, 7])
def test_transposed_product_on_any_shape_and_config(cfg):
    """skinny=1 forces the transposed product (and a config) on an ordinary shape."""
    _need_gpu()
    w = W.problem(300, 260, 700, dtype_out="f32", bias=True, alpha=0.5, beta=1.0, seed=500 + cfg)
    plan, _ = _check(w, skinny=1, config=cfg)
    assert plan["transposed"] == 1 and plan["config"] == cfg


def test_skinny_split_k_and_fixup():
    """64 x 4096 x 4096: 32 tiles of C^T on 152 SMs, so K is split over several CTAs per tile."""
    _need_gpu()
    w = W.problem(64, 4096, 4096, dtype_out="f32", layoutB="col", seed=601)
    plan, _ = _check(w, stream_k=1)
    assert plan["transposed"] == 1 and plan["stream_k"] == 1 and plan["clusters"] > plan["tiles_m"] * plan["tiles_n"]


def test_skinny_split_through_global_partials_without_clusters():
    """A split of 3 parts per tile is not a reduce-scatter (3 does not divide the 8 epilogue warps), so
    the cluster exchange does not take it: the parts hand their partial sums to the tile's head through
    global memory."""
    _need_gpu()
    w = W.problem(48, 640, 4096, dtype_out="f16", layoutB="col", bias=True, seed=602)
    plan, _ = _check(w, stream_k=1, max_clusters=15)        # 5 tiles x 3 parts: not a reduce-scatter
    assert plan["transposed"] == 1 and plan["stream_k"] == 1 and plan["split_cluster"] == 0


@pytest.mark.parametrize("S", [2, 4, 8])
@pytest.mark.parametrize("dout,beta,bias", [("f16", 0.0, False), ("f32", 1.0, True), ("bf16", 0.0, True)])
def test_skinny_split_reduction_is_deterministic(S, dout, beta, bias):
    """40 x 1024 x 4096: 8 tiles of C^T, each split over S CTAs that form one thread-block cluster and
    reduce their partial sums as a reduce-scatter through distributed shared memory.  Each block is
    added up in part order, so every run gives the same bits whichever part finishes first, and the
    result matches the oracle."""
    _need_gpu()
    din = "bf16" if dout == "bf16" else "f16"
    w = W.problem(40, 1024, 4096, dtype_in=din, dtype_out=dout, layoutB="col", bias=bias, alpha=0.75, beta=beta,
                  seed=640 + S)
    d = W.generate(w)
    dd = device_inputs(d)
    C0 = alloc_c(w, d)
    outs = []
    with G.Gemm(0, stream_k=1, max_clusters=8 * S) as g:
        for _ in range(6):
            C = C0.clone()
            run_gpu(g, w, dd, C)
            outs.append(C)
        plan = g.last_plan()
        assert g.status() == G.GEMM_OK
    torch.cuda.synchronize()
    assert plan["transposed"] == 1 and plan["stream_k"] == 1 and plan["clusters"] == 8 * S
    assert plan["split_cluster"] == 1
    rep = compare(w, d, outs[0])
    assert rep["passed"], rep
    for C in outs[1:]:
        assert torch.equal(C, outs[0])


def test_skinny_cluster_split_bounded_wait():
    """The first CTA of the first tile's cluster never receives its second stage: its MMA wait runs out,
    so it never signals its slices free nor sends its blocks, and the other three parts of that cluster
    give up on it after 200 ms.  The timeout is reported, every CTA leaves, and the next call works."""
    _need_gpu()
    w = W.problem(40, 1024, 4096, dtype_out="f16", layoutB="col", seed=650)
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d)
    g = G.Gemm(0, stream_k=1, max_clusters=32, timeout_ms=200, debug_skip_stage=1)
    run_gpu(g, w, dd, C)
    assert g.last_plan()["split_cluster"] == 1 and g.last_plan()["config"] == 7
    st = g.status()
    assert st == G.GEMM_ERR_TIMEOUT, G.gemm_status_string(st)
    assert g.status() == G.GEMM_OK
    g.close()
    C = alloc_c(w, d)
    with G.Gemm(0, stream_k=1, max_clusters=32, sync_check=1) as g2:
        run_gpu(g2, w, dd, C)
        assert g2.last_plan()["split_cluster"] == 1
    torch.cuda.synchronize()
    rep = compare(w, d, C)
    assert rep["passed"], rep


def test_skinny_integers_equal_plain_product():
    """Small integers: the transposed and the plain product are both exact, hence equal."""
    _need_gpu()
    M, N, K = 24, 2048, 1536
    A = W.small_ints(M, K, "f16", 31).cuda()
    B = W.small_ints(N, K, "f16", 32).cuda()               # stored N x K
    ref = (A.cpu().to(torch.int64) @ B.cpu().to(torch.int64).t()).to(torch.float32)
    outs = []
    for skinny in (0, 1):
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        with G.Gemm(0, sync_check=1, skinny=skinny) as g:
            g.run(A, B, C, layoutB="col")
            assert g.last_plan()["transposed"] == skinny
        outs.append(C.cpu())
    assert torch.equal(outs[0], ref) and torch.equal(outs[1], ref)


def test_skinny_ldc_wider_than_n_leaves_padding():
    _need_gpu()
    w = W.problem(5, 700, 256, dtype_out="f16", layoutB="col", seed=602)
    d = W.generate(w)
    dd = device_inputs(d)
    C = torch.full((5, 720), -7.0, dtype=torch.float16, device="cuda")
    for skinny in (1, 2):                                  # the transposed product and the CUDA-core kernel
        C.fill_(-7.0)
        with G.Gemm(0, sync_check=1, skinny=skinny) as g:
            g.run(dd["A"], dd["B"], C, M=5, N=700, K=256, layoutB="col")
            assert g.last_plan()["transposed" if skinny == 1 else "gemv"] == 1
        torch.cuda.synchronize()
        assert torch.all(C[:, 700:].cpu() == -7.0)
        rep = compare(w, d, C[:, :700].contiguous())
        assert rep["passed"], rep


# ------------------------------------------------------------------ CUDA-core kernel, M <= 8
GEMV_CASES = [
    dict(M=1, N=4096, K=4096, dtype_out="f16"),
    dict(M=2, N=4097, K=1000, dtype_out="f32", bias=True),                  # N tail (4-row groups), K = 8 * 125
    dict(M=3, N=300, K=72, dtype_out="bf16", dtype_in="bf16", alpha=0.5, beta=1.0),
    dict(M=5, N=1000, K=2048, dtype_out="f32", bias=True, alpha=-1.5, beta=0.25),
    dict(M=8, N=4096, K=4096, dtype_out="f16", bias=True),
    dict(M=8, N=11008, K=4096, dtype_out="bf16", dtype_in="bf16"),
    dict(M=7, N=65, K=16384, dtype_out="f32"),                               # long K
    dict(M=4, N=151, K=1032, dtype_out="f16", bias=True),                    # fewer rows than SMs, K = 1024 + 8
    dict(M=1, N=20000, K=520, dtype_out="bf16", dtype_in="bf16"),           # many short rows per CTA
]


@pytest.mark.parametrize("M,N,K", [(1, 1, 4096), (3, 2, 8), (8, 17, 5000), (2, 5, 1024)])
def test_small_m_forced_tiny_n(M, N, K):
    """skinny 2 takes the CUDA-core kernel for any N: a row's pieces spread over many warps."""
    _need_gpu()
    w = W.problem(M, N, K, dtype_out="f32", layoutB="col", bias=True, seed=850 + M + N)
    plan, _ = _check(w, skinny=2)
    assert plan["gemv"] == 1


@pytest.mark.parametrize("i", range(len(GEMV_CASES)))
def test_small_m_cuda_core_parity(i):
    _need_gpu()
    c = dict(GEMV_CASES[i])
    w = W.problem(c.pop("M"), c.pop("N"), c.pop("K"), layoutB="col", seed=800 + i, **c)
    plan, _ = _check(w)
    assert plan["gemv"] == 1


def test_small_m_with_a_stored_k_by_m_takes_the_transposed_product():
    _need_gpu()
    w = W.problem(5, 1000, 2048, dtype_out="f32", layoutA="col", layoutB="col", bias=True, seed=820)
    plan, _ = _check(w)
    assert plan["gemv"] == 0 and plan["transposed"] == 1


def test_small_m_padded_pitches():
    """B rows at a pitch wider than K (16-byte multiple), C with ldc > N: padding never touched."""
    _need_gpu()
    M, N, K = 6, 700, 512
    g0 = torch.Generator().manual_seed(77)
    A = (torch.rand(M, K, generator=g0, dtype=torch.float64) * 2 - 1).half()
    Bs = (torch.rand(N, K + 24, generator=g0, dtype=torch.float64) * 2 - 1).half()
    Bs[:, K:] = float("nan")                                                # must never be read
    C = torch.full((M, N + 9), -3.0, dtype=torch.float32, device="cuda")
    with G.Gemm(0, sync_check=1) as g:
        g.run(A.cuda(), Bs.cuda(), C, M=M, N=N, K=K, layoutB="col")
        assert g.last_plan()["gemv"] == 1
    torch.cuda.synchronize()
    ref = A.double() @ Bs[:, :K].double().t()
    got = C[:, :N].cpu().double()
    assert torch.all(C[:, N:].cpu() == -3.0)
    assert float((got - ref).abs().max()) <= 1e-4 * K


def test_small_m_integers_equal_tensor_core_paths():
    _need_gpu()
    M, N, K = 8, 3000, 2048
    A = W.small_ints(M, K, "f16", 51).cuda()
    B = W.small_ints(N, K, "f16", 52).cuda()                                # stored N x K
    ref = (A.cpu().to(torch.int64) @ B.cpu().to(torch.int64).t()).to(torch.float32)
    for skinny in (2, 1, 0):
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        with G.Gemm(0, sync_check=1, skinny=skinny) as g:
            g.run(A, B, C, layoutB="col")
            plan = g.last_plan()
        assert plan["gemv"] == (1 if skinny == 2 else 0)
        torch.cuda.synchronize()
        assert torch.equal(C.cpu(), ref), skinny


def test_small_m_forced_where_it_does_not_apply():
    _need_gpu()
    A = torch.zeros(4, 4096, dtype=torch.float16, device="cuda")
    B = torch.zeros(4096, 4096, dtype=torch.float16, device="cuda")
    C = torch.zeros(4, 4096, dtype=torch.float32, device="cuda")
    with G.Gemm(0, skinny=2) as g:
        assert g.run(A, B, C, layoutB="row", check=False) == G.GEMM_ERR_UNSUPPORTED   # B stored K x N
        A16 = torch.zeros(16, 4096, dtype=torch.float16, device="cuda")
        C16 = torch.zeros(16, 4096, dtype=torch.float32, device="cuda")
        assert g.run(A16, B, C16, layoutB="col", check=False) == G.GEMM_ERR_UNSUPPORTED  # M > 8


@pytest.mark.parametrize("wid", [7, 8])
def test_decode_workloads_full_check(wid):
    """The benchmark's decode workloads (1 x 4096 x 4096 on the CUDA-core kernel, 64 x 4096 x 4096 on the transposed
    split product) with the benchmark's own inputs and handle options, every element against the oracle."""
    _need_gpu()
    w = W.WORKLOADS[wid]
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d)
    with G.Gemm(0, sync_check=1) as g:
        run_gpu(g, w, dd, C)
        plan = g.last_plan()
        assert plan["gemv"] == (1 if wid == 7 else 0) and plan["transposed"] == (0 if wid == 7 else 1)
    torch.cuda.synchronize()
    rep = compare(w, d, C)
    assert rep["passed"], rep
