"""GPU parity of the Q4_0 weight path: the separate dequantisation kernel (bit-exact against the
oracle's decode) and the three routes of gemm_run_q4_0 -- the GEMM whose kernel dequantises B in
shared memory, the CUDA-core kernel for M <= 8, and the separate pass followed by the f16 GEMM --
against the oracle's dequantise-then-GEMM reference (and, where the arithmetic is the same, bit for
bit against the plain GEMM on the dequantised weights)."""
import numpy as np
import pytest
import torch

import oracle
from bf16_tensor_core_gb300 import gemm as G
from bf16_tensor_core_gb300 import workloads as W
from gpu_cases import OR_CODE, sample_indices

pytestmark = pytest.mark.gpu
Q4_CONFIG = 6


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _blocks(N, K, seed, ldbq=None, scale=0.02):
    return W.q4_0_blocks(N, K, seed, ldbq=ldbq, scale=scale)


def _special_block_rows(K):
    """Rows of hand-made blocks: subnormal scales, a rounding case, every nibble, negative scale."""
    assert K % 32 == 0
    rows = []
    for d_bits in (0x0003, 0x03FF, 0x3C01, 0xB800, 0x3C00, 0x1400):
        r = bytearray()
        for b in range(K // 32):
            r += bytes([d_bits & 0xff, d_bits >> 8]) + bytes([(i * 17 + b * 5) & 0xff for i in range(16)])
        rows.append(np.frombuffer(bytes(r), np.uint8))
    return torch.from_numpy(np.stack(rows))


# ------------------------------------------------------------------ separate dequantisation
@pytest.mark.parametrize("N,K,ldbq,ldo", [(7, 64, None, None), (70, 256, 148, 260), (33, 1024, None, 1025),
                                          (300, 4096, None, None), (45, 1056, 608, 1064), (3, 32, 32, 40),
                                          (129, 8192, 4624, None)])
def test_dequant_bit_exact(N, K, ldbq, ldo):
    _need_gpu()
    bq = _blocks(N, K, seed=N + K, ldbq=ldbq)
    ref = oracle.q4_0_to_f16(bq.numpy(), N, K)
    ldo = ldo or K
    out = torch.full((N, ldo), -1.0, dtype=torch.float16, device="cuda")
    st = G.gemm_dequant_q4_0(bq.cuda().data_ptr(), bq.size(1), N, K, out.data_ptr(), ldo,
                             torch.cuda.current_stream().cuda_stream)
    assert st == G.GEMM_OK
    torch.cuda.synchronize()
    got = out[:, :K].cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    if ldo > K:
        assert torch.all(out[:, K:].cpu() == -1.0)          # padding untouched


def test_dequant_special_blocks_bit_exact():
    _need_gpu()
    bq = _special_block_rows(128)
    ref = oracle.q4_0_to_f16(bq.numpy(), bq.size(0), 128)
    out = torch.empty(bq.size(0), 128, dtype=torch.float16, device="cuda")
    assert G.gemm_dequant_q4_0(bq.cuda().data_ptr(), bq.size(1), bq.size(0), 128, out.data_ptr(), 128, None) == 0
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), ref)


def test_dequant_rejects_bad_arguments():
    _need_gpu()
    bq = _blocks(4, 64, 1).cuda()
    out = torch.empty(4, 64, dtype=torch.float16, device="cuda")
    assert G.gemm_dequant_q4_0(bq.data_ptr(), 36, 4, 48, out.data_ptr(), 64, None) == G.GEMM_ERR_INVALID_ARG
    assert G.gemm_dequant_q4_0(bq.data_ptr(), 35, 4, 64, out.data_ptr(), 64, None) == G.GEMM_ERR_INVALID_ARG
    assert G.gemm_dequant_q4_0(bq.data_ptr() + 1, 36, 4, 64, out.data_ptr(), 64, None) == G.GEMM_ERR_ALIGNMENT


# ------------------------------------------------------------------ fused dequant-in-GEMM
def _case(M, N, K, seed, *, dout="f16", layoutA="row", alpha=1.0, beta=0.0, bias=False, ldbq=None, scale=0.02):
    g = torch.Generator().manual_seed(seed)
    A_st = (torch.rand((M, K) if layoutA == "row" else (K, M), generator=g, dtype=torch.float64) * 2 - 1).half()
    bq = _blocks(N, K, seed + 1, ldbq=ldbq, scale=scale)
    b = (torch.rand(N, generator=g, dtype=torch.float64) * 2 - 1).to(W.DTYPES[dout]) if bias else None
    cin = (torch.rand((M, N), generator=g, dtype=torch.float64) * 2 - 1).to(W.DTYPES[dout]) if beta != 0 else None
    return dict(M=M, N=N, K=K, A=A_st, bq=bq, bias=b, Cin=cin, dout=dout, layoutA=layoutA, alpha=alpha, beta=beta)


def _run(g, c, C=None):
    A, bq = c["A"].cuda(), c["bq"].cuda()
    if C is None:
        C = (c["Cin"].cuda().clone() if c["Cin"] is not None
             else torch.full((c["M"], c["N"]), float("nan"), dtype=W.DTYPES[c["dout"]], device="cuda"))
    g.run_q4_0(A, bq, C, N=c["N"], K=c["K"], M=c["M"], layoutA=c["layoutA"], alpha=c["alpha"], beta=c["beta"],
               bias=c["bias"].cuda() if c["bias"] is not None else None)
    torch.cuda.synchronize()
    return C


def _check(c, C, rows=None, cols=None):
    ref = oracle.gemm_ref_q4_0(c["M"], c["N"], c["K"], c["A"], oracle.OR_ROW if c["layoutA"] == "row" else oracle.OR_COL,
                               c["bq"].numpy(), alpha=c["alpha"], beta=c["beta"], Cin=c["Cin"],
                               dtype_cin=OR_CODE[c["dout"]], bias=c["bias"], dtype_bias=OR_CODE[c["dout"]],
                               rows=rows, cols=cols)
    got = C.cpu()
    if rows is not None:
        got = got[torch.as_tensor(rows)]
    if cols is not None:
        got = got[:, torch.as_tensor(cols)]
    got = got.double().numpy()
    Wf = oracle.q4_0_to_f16(c["bq"].numpy(), c["N"], c["K"]).view(np.float16).astype(np.float64)
    maxA, maxB = float(c["A"].abs().max()), float(np.abs(Wf).max())
    cin = None
    if c["Cin"] is not None:
        cin = c["Cin"].double()
        if rows is not None:
            cin = cin[torch.as_tensor(rows)]
        if cols is not None:
            cin = cin[:, torch.as_tensor(cols)]
        cin = cin.numpy()
    bias = c["bias"].double().numpy() if c["bias"] is not None else None
    if bias is not None and cols is not None:
        bias = bias[np.asarray(cols)]
    mag = oracle.epilogue_magnitude(ref, c["beta"], cin, bias)
    rep = oracle.check(got, ref, c["K"], maxA, maxB, OR_CODE[c["dout"]], alpha=c["alpha"], epi_mag=mag)
    assert rep["passed"], rep
    return rep


FUSED_CASES = [
    dict(M=300, N=520, K=640, dout="f16", bias=True),                       # ragged tiles, K tail of 128
    dict(M=512, N=768, K=1024, dout="f32"),
    dict(M=257, N=300, K=2048, dout="bf16", layoutA="col"),
    dict(M=700, N=260, K=96, dout="f32", alpha=0.5, beta=1.0),               # one partial k-tile
    dict(M=128, N=1000, K=4096, dout="f16", ldbq=2320),                      # padded weight rows
    dict(M=200, N=300, K=128, dout="f32", ldbq=74),                          # pitch 2 mod 4: rows repacked
]


@pytest.mark.parametrize("i", range(len(FUSED_CASES)))
def test_fused_parity(i):
    _need_gpu()
    c = _case(seed=50 + i, **FUSED_CASES[i])
    with G.Gemm(0, sync_check=1, config=Q4_CONFIG) as g:
        C = _run(g, c)
        assert g.last_plan()["config"] == Q4_CONFIG
    _check(c, C)


@pytest.mark.parametrize("sk", [0, 1])
def test_fused_equals_plain_gemm_on_dequantised_weights(sk):
    """Same tiles, same k order, same MMAs: only where B comes from differs, so the outputs agree
    bit for bit with the plain GEMM (config 4, the same tile shape) on the dequantised f16 weights."""
    _need_gpu()
    c = _case(1000, 1500, 2048, seed=70, dout="f32", bias=True)
    # 24 tiles on at most 48 clusters: both configs take the same split whatever their time models say.
    with G.Gemm(0, sync_check=1, stream_k=sk, config=Q4_CONFIG, max_clusters=48) as g:
        C1 = _run(g, c)
        plan = g.last_plan()
    Wd = torch.empty(c["N"], c["K"], dtype=torch.float16, device="cuda")
    bq = c["bq"].cuda()
    assert G.gemm_dequant_q4_0(bq.data_ptr(), bq.size(1), c["N"], c["K"], Wd.data_ptr(), c["K"], None) == 0
    C2 = torch.full_like(C1, float("nan"))
    with G.Gemm(0, config=4, sync_check=1, stream_k=sk, max_clusters=48) as g:
        g.run(c["A"].cuda(), Wd, C2, layoutB="col", bias=c["bias"].cuda())
        p2 = g.last_plan()
        assert (p2["stream_k"], p2["clusters"], p2["dp_tiles"]) == (plan["stream_k"], plan["clusters"], plan["dp_tiles"])
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


def test_fused_rows_two_bytes_past_alignment():
    """Weights whose rows start 2 bytes past a 4-byte boundary are repacked first; same result."""
    _need_gpu()
    c = _case(256, 384, 1024, seed=60, dout="f32")
    N, pitch = c["N"], c["bq"].size(1)                    # 576 bytes per row
    store = torch.zeros(N, pitch + 4, dtype=torch.uint8)
    store[:, 2:2 + pitch] = c["bq"]
    dev = store.cuda()
    view = dev[:, 2:2 + pitch]                            # data_ptr % 4 == 2, row stride pitch + 4
    C = torch.full((c["M"], N), float("nan"), dtype=torch.float32, device="cuda")
    with G.Gemm(0, sync_check=1, config=Q4_CONFIG) as g:
        n0 = g.launches
        st = G.gemm_run_q4_0(g.h, c["M"], N, c["K"], c["A"].cuda().data_ptr(), c["K"], 0, view.data_ptr(),
                             pitch + 4, C.data_ptr(), N, 2, 1.0, 0.0, None, torch.cuda.current_stream().cuda_stream)
        assert st == G.GEMM_OK, g.last_error()
        assert g.last_plan()["repack_b"] == 1 and g.launches - n0 == 2
    torch.cuda.synchronize()
    _check(c, C)


def test_fused_integers_exact():
    """d = 1 and small-integer activations: every product and partial sum is an integer < 2^24."""
    _need_gpu()
    M, N, K = 384, 640, 1024
    A = W.small_ints(M, K, "f16", 9)
    g0 = torch.Generator().manual_seed(10)
    q = torch.randint(0, 256, (N, K // 32, 16), generator=g0, dtype=torch.int64).to(torch.uint8)
    blocks = torch.zeros(N, K // 32, 18, dtype=torch.uint8)
    blocks[:, :, 0], blocks[:, :, 1] = 0x00, 0x3C          # d = 1.0
    blocks[:, :, 2:] = q
    bq = blocks.reshape(N, -1)
    Wint = oracle.q4_0_to_f16(bq.numpy(), N, K).view(np.float16).astype(np.int64)
    ref = torch.from_numpy(A.to(torch.int64).numpy() @ Wint.T).to(torch.float32)
    for sk in (0, 1):
        C = torch.empty(M, N, dtype=torch.float32, device="cuda")
        with G.Gemm(0, sync_check=1, stream_k=sk, config=Q4_CONFIG) as g:
            g.run_q4_0(A.cuda(), bq.cuda(), C, N=N)
        torch.cuda.synchronize()
        assert torch.equal(C.cpu(), ref), sk


def test_fused_split_k_parity():
    """Few output tiles and long K: the schedule splits K over several clusters."""
    _need_gpu()
    c = _case(200, 500, 8192, seed=80, dout="f32")
    with G.Gemm(0, sync_check=1, stream_k=1, config=Q4_CONFIG) as g:
        C = _run(g, c)
        plan = g.last_plan()
    assert plan["stream_k"] == 1 and plan["clusters"] > plan["tiles_m"] * plan["tiles_n"]
    _check(c, C)


def test_fused_split_k_reduce_scatter_parity():
    """Two tiles split four ways each (eight clusters): the four epilogue warps of a tile are shared out
    among its parts, one each."""
    _need_gpu()
    c = _case(256, 512, 4096, seed=81, dout="f16", bias=True)
    with G.Gemm(0, sync_check=1, stream_k=1, config=Q4_CONFIG, max_clusters=8) as g:
        C = _run(g, c)
        plan = g.last_plan()
    assert plan["stream_k"] == 1 and plan["dp_tiles"] == 0
    assert plan["clusters"] == 4 * plan["tiles_m"] * plan["tiles_n"] == 8
    _check(c, C)


def test_fused_special_blocks():
    _need_gpu()
    M, K = 256, 128
    bq = _special_block_rows(K)
    A = (torch.rand(M, K, generator=torch.Generator().manual_seed(4), dtype=torch.float64) * 2 - 1).half()
    c = dict(M=M, N=bq.size(0), K=K, A=A, bq=bq, bias=None, Cin=None, dout="f32", layoutA="row", alpha=1.0,
             beta=0.0)
    with G.Gemm(0, sync_check=1, config=Q4_CONFIG) as g:
        C = _run(g, c)
    _check(c, C)


def test_fused_prefill_shape_sampled():
    """The 2048 x 11008 x 4096 prefill projection with Q4_0 weights, sampled rows and columns."""
    _need_gpu()
    c = _case(2048, 11008, 4096, seed=90, dout="bf16", bias=True)
    with G.Gemm(0, sync_check=1, config=Q4_CONFIG) as g:
        C = _run(g, c)
    rows = sample_indices(2048, 24, 1, 256)
    cols = sample_indices(11008, 24, 2, 256)
    _check(c, C, rows=rows)
    _check(c, C, cols=cols)


def test_fused_rejects_bad_arguments():
    _need_gpu()
    A = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    bq = _blocks(64, 64, 3).cuda()
    C = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    with G.Gemm(0) as g:
        s = torch.cuda.current_stream().cuda_stream
        assert G.gemm_run_q4_0(g.h, 64, 64, 48, A.data_ptr(), 64, 0, bq.data_ptr(), 36, C.data_ptr(), 64, 2,
                               1.0, 0.0, None, s) == G.GEMM_ERR_INVALID_ARG        # K not whole blocks
        assert G.gemm_run_q4_0(g.h, 64, 64, 64, A.data_ptr(), 64, 0, bq.data_ptr(), 35, C.data_ptr(), 64, 2,
                               1.0, 0.0, None, s) == G.GEMM_ERR_INVALID_ARG        # odd pitch
        assert G.gemm_run_q4_0(g.h, 64, 64, 64, A.data_ptr(), 64, 0, bq.data_ptr() + 1, 36, C.data_ptr(), 64, 2,
                               1.0, 0.0, None, s) == G.GEMM_ERR_ALIGNMENT
    with G.Gemm(0, skinny=2) as g:                                                 # small-M kernel, M > 8
        assert G.gemm_run_q4_0(g.h, 64, 64, 64, A.data_ptr(), 64, 0, bq.data_ptr(), 36, C.data_ptr(), 64, 2,
                               1.0, 0.0, None, torch.cuda.current_stream().cuda_stream) == G.GEMM_ERR_UNSUPPORTED
    with G.Gemm(0, config=Q4_CONFIG) as g:                                         # plain B on the Q4_0 config
        assert g.run(A, A, C, check=False) == G.GEMM_ERR_UNSUPPORTED


def test_fused_bounded_wait_expires_and_reports():
    """Cluster 0's producer never issues the A copy of stage 3: the MMA issuer's wait runs out after
    200 ms, the dequantisation warps leave their loop together (their per-stage barrier ANDs the
    wait outcomes), the kernel records the timeout and returns; the next call works."""
    _need_gpu()
    c = _case(256, 256, 1024, seed=95, dout="f32")
    with G.Gemm(0, timeout_ms=200, debug_skip_stage=3, config=Q4_CONFIG, stream_k=0) as g:   # 8 stages per tile
        _run(g, c)
        st = g.status()
        assert st == G.GEMM_ERR_TIMEOUT, G.gemm_status_string(st)
        assert g.status() == G.GEMM_OK
    with G.Gemm(0, sync_check=1) as g:
        C = _run(g, c)
    _check(c, C)


# ------------------------------------------------------------------ CUDA-core kernel, M <= 8
GEMV_CASES = [
    dict(M=1, N=4096, K=4096, dout="f16"),
    dict(M=1, N=11008, K=4096, dout="bf16", bias=True),
    dict(M=2, N=37, K=32, dout="f32"),                                      # one block per row
    dict(M=3, N=1001, K=11008, dout="f32", alpha=0.5, beta=1.0),            # several blocks per thread
    dict(M=5, N=6, K=96, dout="f16", bias=True),
    dict(M=7, N=130, K=4128, dout="bf16", ldbq=2330),                       # pitch 2 mod 4: rows alternate alignment
    dict(M=8, N=515, K=2048, dout="f32", bias=True, alpha=2.0, beta=-1.0),
    dict(M=4, N=64, K=640, dout="f16", layoutA="row"),
    dict(M=1, N=3, K=8192, dout="f32"),                                     # two pieces per row, few rows
    dict(M=2, N=2000, K=4096, dout="f16", ldbq=2320, bias=True),            # padded 16-byte pitch
    dict(M=6, N=777, K=12288, dout="bf16", alpha=0.25, beta=0.5),
]


@pytest.mark.parametrize("i", range(len(GEMV_CASES)))
def test_small_m_parity(i):
    _need_gpu()
    c = _case(seed=200 + i, **GEMV_CASES[i])
    with G.Gemm(0, sync_check=1) as g:
        n0 = g.launches
        C = _run(g, c)
        plan = g.last_plan()
        assert plan["gemv"] == 1 and plan["config"] == -1 and g.launches - n0 == 1
    _check(c, C)


def test_small_m_rows_two_bytes_past_alignment():
    """The CUDA-core kernel reads blocks at any 2-byte alignment (no repack)."""
    _need_gpu()
    c = _case(3, 300, 1024, seed=210, dout="f32")
    N, pitch = c["N"], c["bq"].size(1)
    store = torch.zeros(N, pitch + 4, dtype=torch.uint8)
    store[:, 2:2 + pitch] = c["bq"]
    view = store.cuda()[:, 2:2 + pitch]
    C = torch.full((c["M"], N), float("nan"), dtype=torch.float32, device="cuda")
    with G.Gemm(0, sync_check=1) as g:
        n0 = g.launches
        st = G.gemm_run_q4_0(g.h, c["M"], N, c["K"], c["A"].cuda().data_ptr(), c["K"], 0, view.data_ptr(),
                             pitch + 4, C.data_ptr(), N, 2, 1.0, 0.0, None, torch.cuda.current_stream().cuda_stream)
        assert st == G.GEMM_OK, g.last_error()
        assert g.last_plan()["gemv"] == 1 and g.launches - n0 == 1
    torch.cuda.synchronize()
    _check(c, C)


def test_small_m_integers_exact():
    """d = 1, small-integer activations: every product and f32 partial sum is an exact integer."""
    _need_gpu()
    M, N, K = 8, 333, 2048
    A = W.small_ints(M, K, "f16", 19)
    g0 = torch.Generator().manual_seed(20)
    q = torch.randint(0, 256, (N, K // 32, 16), generator=g0, dtype=torch.int64).to(torch.uint8)
    blocks = torch.zeros(N, K // 32, 18, dtype=torch.uint8)
    blocks[:, :, 0], blocks[:, :, 1] = 0x00, 0x3C
    blocks[:, :, 2:] = q
    bq = blocks.reshape(N, -1)
    Wint = oracle.q4_0_to_f16(bq.numpy(), N, K).view(np.float16).astype(np.int64)
    ref = torch.from_numpy(A.to(torch.int64).numpy() @ Wint.T).to(torch.float32)
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    with G.Gemm(0, sync_check=1) as g:
        g.run_q4_0(A.cuda(), bq.cuda(), C, N=N)
        assert g.last_plan()["gemv"] == 1
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), ref)


def test_small_m_special_blocks():
    _need_gpu()
    K = 128
    bq = _special_block_rows(K)
    A = (torch.rand(4, K, generator=torch.Generator().manual_seed(21), dtype=torch.float64) * 2 - 1).half()
    c = dict(M=4, N=bq.size(0), K=K, A=A, bq=bq, bias=None, Cin=None, dout="f32", layoutA="row", alpha=1.0,
             beta=0.0)
    with G.Gemm(0, sync_check=1) as g:
        C = _run(g, c)
        assert g.last_plan()["gemv"] == 1
    _check(c, C)


def test_small_m_column_major_a_takes_the_fused_kernel():
    """The CUDA-core kernel wants row-major activations; a column-major A goes to the fused kernel."""
    _need_gpu()
    c = _case(4, 300, 512, seed=220, dout="f32", layoutA="col")
    with G.Gemm(0, sync_check=1) as g:
        C = _run(g, c)
        assert g.last_plan()["gemv"] == 0 and g.last_plan()["config"] == Q4_CONFIG
    _check(c, C)


# ------------------------------------------------------------------ separate pass + f16 GEMM
def test_separate_pass_route_chosen_for_the_prefill_shape():
    _need_gpu()
    c = _case(2048, 11008, 4096, seed=230, dout="bf16", bias=True)
    with G.Gemm(0, sync_check=1) as g:
        n0 = g.launches
        C = _run(g, c)
        plan = g.last_plan()
        assert plan["q4_dequant"] == 1 and plan["config"] != Q4_CONFIG and g.launches - n0 == 2
    _check(c, C, rows=sample_indices(2048, 24, 3, 256))
    _check(c, C, cols=sample_indices(11008, 24, 4, 256))


@pytest.mark.parametrize("cfg", [1, 4])
def test_separate_pass_equals_plain_gemm_on_dequantised_weights(cfg):
    """A config without Q4_0 weights asks for the separate pass: the result is the plain GEMM on the
    dequantised weights with that config, bit for bit."""
    _need_gpu()
    c = _case(700, 900, 1024, seed=240, dout="f32", bias=True, alpha=0.75, beta=0.5)
    with G.Gemm(0, sync_check=1, config=cfg) as g:
        C1 = _run(g, c)
        assert g.last_plan()["q4_dequant"] == 1 and g.last_plan()["config"] == cfg
    Wd = torch.empty(c["N"], c["K"], dtype=torch.float16, device="cuda")
    bq = c["bq"].cuda()
    assert G.gemm_dequant_q4_0(bq.data_ptr(), bq.size(1), c["N"], c["K"], Wd.data_ptr(), c["K"], None) == 0
    C2 = c["Cin"].cuda().clone()
    with G.Gemm(0, sync_check=1, config=cfg) as g:
        g.run(c["A"].cuda(), Wd, C2, layoutB="col", bias=c["bias"].cuda(), alpha=c["alpha"], beta=c["beta"])
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    _check(c, C1)


def test_decode_workload_q4_0_full_check():
    """The benchmark's Q4_0 decode workload (1 x 4096 x 4096) with the benchmark's own inputs and handle options,
    every element against the oracle."""
    _need_gpu()
    w = W.WORKLOADS[10]
    d = W.generate(w)
    c = dict(M=w.M, N=w.N, K=w.K, A=d["A"], bq=d["B"], bias=d["bias"], Cin=d["Cin"], dout=w.dtype_out,
             layoutA=w.layoutA, alpha=w.alpha, beta=w.beta)
    with G.Gemm(0, sync_check=1) as g:
        C = _run(g, c)
        assert g.last_plan()["config"] == -1          # the CUDA-core small-M route
    _check(c, C)
