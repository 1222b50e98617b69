"""GPU parity tests: the CUDA path (through the C ABI) against the CPU oracle, element by element.

Tolerance (per element): 1e-4 * K * max|A| * max|B| for f32 output, plus one output ulp of
|C_ref| for f16/bf16 output, plus 4 f32 ulps of the epilogue operands (see oracle.check).
Integer-valued inputs whose partial sums stay below 2^24 must match bit for bit.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from bf16_tensor_core_gb300 import gemm as G
from bf16_tensor_core_gb300 import workloads as W
from gpu_cases import alloc_c, compare, device_inputs, run_gpu, sample_indices

pytestmark = pytest.mark.gpu

CONFIGS = [0, 1, 2, 3, 4, 5]


@pytest.fixture(scope="module")
def handles():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    hs = {c: G.Gemm(0, config=c, sync_check=1) for c in CONFIGS}
    hs["auto"] = G.Gemm(0, sync_check=1)
    yield hs
    for h in hs.values():
        h.close()


def _run_check(h, w, *, ldc=None, rows=None, cols=None):
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d, ldc)
    run_gpu(h, w, dd, C)
    torch.cuda.synchronize()
    rep = compare(w, d, C, rows, cols)
    assert rep["passed"], rep
    return rep, C, d


# ------------------------------------------------------------------------------ the five workloads
@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("wid", [1, 4])
def test_small_workloads_full_check(handles, cfg, wid):
    """512^3 and the ragged 1000x3000x2050 case checked on every element, on every config."""
    _run_check(handles[cfg], W.WORKLOADS[wid])


@pytest.mark.parametrize("wid", [2, 3, 5])
def test_large_workloads_sampled(handles, wid):
    """Full-size 4096^3, the 2048x11008x4096 prefill projection and 8192^3 with the automatic
    config (the one the benchmark times): sampled rows x all columns and all rows x sampled columns,
    including every tile boundary."""
    w = W.WORKLOADS[wid]
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d)
    run_gpu(handles["auto"], w, dd, C)
    torch.cuda.synchronize()
    rows = sample_indices(w.M, 48, seed=wid, tile=128)
    cols = sample_indices(w.N, 48, seed=wid + 100, tile=64)
    rep_r = compare(w, d, C, rows=rows)
    assert rep_r["passed"], rep_r
    rep_c = compare(w, d, C, cols=cols)
    assert rep_c["passed"], rep_c


@pytest.mark.parametrize("cfg", CONFIGS)
def test_prefill_shape_reduced_on_every_config(handles, cfg):
    w = W.with_changes(W.WORKLOADS[3], M=384, N=1000, K=640, name="prefill_reduced")
    _run_check(handles[cfg], w)


# ------------------------------------------------------------------------------ tails and layouts
TAIL_SHAPES = [(1, 1, 1), (1, 300, 70), (17, 33, 16), (127, 129, 64), (128, 128, 128), (129, 255, 65),
               (255, 257, 129), (257, 127, 200), (300, 520, 1), (33, 600, 333), (640, 64, 8)]


@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("shape", TAIL_SHAPES)
def test_tail_shapes(handles, cfg, shape):
    M, N, K = shape
    w = W.problem(M, N, K, dtype_in="f16", dtype_out="f32", seed=M * 7 + N * 3 + K)
    _run_check(handles[cfg], w)


@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("la,lb", [("row", "row"), ("row", "col"), ("col", "row"), ("col", "col")])
@pytest.mark.parametrize("din,dout", [("f16", "f32"), ("bf16", "bf16"), ("f16", "f16"), ("bf16", "f32")])
def test_layouts_and_dtypes(handles, cfg, la, lb, din, dout):
    w = W.problem(300, 392, 200, dtype_in=din, dtype_out=dout, layoutA=la, layoutB=lb, bias=True,
                  seed=len(la) * 97 + len(lb) * 31 + len(din) * 7 + len(dout))
    _run_check(handles[cfg], w)


@pytest.mark.parametrize("cfg", CONFIGS)
def test_alpha_beta_bias(handles, cfg):
    for (alpha, beta, dout) in [(0.5, 1.0, "f32"), (-2.0, 0.25, "f16"), (1.0, -1.0, "bf16"), (0.0, 2.0, "f32")]:
        w = W.problem(260, 300, 150, dtype_out=dout, alpha=alpha, beta=beta, bias=True, seed=int(abs(alpha * 10)))
        _run_check(handles[cfg], w)


# ------------------------------------------------------------------------------ exactness
@pytest.mark.parametrize("cfg", CONFIGS)
def test_small_integers_bit_exact(handles, cfg):
    """Integers in [-3, 3]: every partial sum is an integer below 2^24, so f32 accumulation is exact."""
    M, N, K = 320, 384, 1100
    for dt in ("f16", "bf16"):
        A = W.small_ints(M, K, dt, 1)
        B = W.small_ints(K, N, dt, 2)
        C = torch.empty(M, N, dtype=torch.float32, device="cuda")
        handles[cfg].run(A.cuda(), B.cuda(), C)
        torch.cuda.synchronize()
        ref = A.to(torch.int64) @ B.to(torch.int64)
        assert torch.equal(C.cpu(), ref.to(torch.float32)), dt


@pytest.mark.parametrize("cfg", CONFIGS)
def test_identity_and_permutation_exact(handles, cfg):
    n, N = 384, 200
    B = W.generate(W.problem(n, N, n, seed=3))["B"]          # n x N
    I = W.identity(n, n, "f16")
    C = torch.empty(n, N, dtype=torch.float32, device="cuda")
    handles[cfg].run(I.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), B.to(torch.float32))
    perm = W.permutation(n, 4)
    P = W.permutation_matrix(perm, "f16")
    handles[cfg].run(P.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), B.to(torch.float32)[perm])
    ones_a = W.ones(n, n, "f16")
    handles[cfg].run(ones_a.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    col_sums = oracle.gemm_ref(n, N, n, ones_a, oracle.OR_ROW, B, oracle.OR_ROW, oracle.OR_F16)
    rep = oracle.check(C.cpu().double().numpy(), col_sums, n, 1.0, float(B.abs().max()), oracle.OR_F32)
    assert rep["passed"], rep


# ------------------------------------------------------------------------------ edge cases
def test_beta_zero_does_not_read_c(handles):
    w = W.problem(200, 300, 100, dtype_out="f32", seed=5)
    d = W.generate(w)
    C = torch.full((w.M, w.N), float("nan"), device="cuda")
    handles["auto"].run(d["A"].cuda(), d["B"].cuda(), C)
    torch.cuda.synchronize()
    assert torch.isfinite(C).all()
    assert compare(w, d, C)["passed"]


@pytest.mark.parametrize("dout", ["f32", "f16", "bf16"])
def test_k_zero(handles, dout):
    w = W.problem(70, 90, 0, dtype_out=dout, beta=0.5, bias=True, seed=9)
    d = W.generate(w)
    C = d["Cin"].cuda().clone()
    A = torch.empty(70, 8, dtype=torch.float16, device="cuda")
    B = torch.empty(8, 90, dtype=torch.float16, device="cuda")
    handles["auto"].run(A, B, C, M=70, N=90, K=0, beta=0.5, bias=d["bias"].cuda())
    torch.cuda.synchronize()
    rep = compare(w, d, C)
    assert rep["passed"], rep


def test_m_or_n_zero_is_noop(handles):
    C = torch.full((4, 4), 7.0, device="cuda")
    A = torch.ones(4, 8, dtype=torch.float16, device="cuda")
    B = torch.ones(8, 4, dtype=torch.float16, device="cuda")
    handles["auto"].run(A, B, C, M=0, N=4, K=8)
    handles["auto"].run(A, B, C, M=4, N=0, K=8)
    torch.cuda.synchronize()
    assert (C == 7.0).all()


def test_unaligned_operand_is_rejected(handles):
    A = torch.zeros(64 * 64 + 8, dtype=torch.float16, device="cuda")
    B = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    C = torch.zeros(64, 64, device="cuda")
    Ash = A[1:1 + 64 * 64].view(64, 64)                        # 2-byte offset
    st = handles["auto"].run(Ash, B, C, check=False)
    assert st == G.GEMM_ERR_ALIGNMENT


@pytest.mark.parametrize("cfg", CONFIGS)
def test_guard_band_untouched(handles, cfg):
    """C inside a larger buffer: padding columns (ldc > N) and rows after M keep their sentinel."""
    for dout in ("f32", "f16"):
        w = W.problem(300, 200, 96, dtype_out=dout, bias=True, seed=11)
        d = W.generate(w)
        ldc = 264
        buf = torch.full((w.M + 7, ldc), 12345.0, dtype=W.DTYPES[dout], device="cuda")
        C = buf[: w.M]
        handles[cfg].run(d["A"].cuda(), d["B"].cuda(), C, M=w.M, N=w.N, K=w.K, bias=d["bias"].cuda())
        torch.cuda.synchronize()
        assert (buf[:, w.N:] == 12345.0).all()
        assert (buf[w.M:] == 12345.0).all()
        assert compare(w, d, C)["passed"]


def test_unaligned_ldc_uses_direct_stores(handles):
    w = W.problem(130, 63, 70, dtype_out="f16", seed=13)
    d = W.generate(w)
    buf = torch.full((w.M, 63), float("nan"), dtype=torch.float16, device="cuda")
    handles["auto"].run(d["A"].cuda(), d["B"].cuda(), buf)
    torch.cuda.synchronize()
    assert compare(w, d, buf)["passed"]


def test_non_default_stream(handles):
    w = W.problem(500, 700, 300, dtype_out="bf16", dtype_in="bf16", seed=17)
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        handles["auto"].run(dd["A"], dd["B"], C, stream=s.cuda_stream)
    s.synchronize()
    assert compare(w, d, C)["passed"]


def test_launch_count(handles):
    g = G.Gemm(0)
    w = W.WORKLOADS[4]
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d)
    n0 = g.launches
    run_gpu(g, w, dd, C)
    assert g.launches - n0 == 2            # one repack launch for both operands + the GEMM
    A = torch.zeros(128, 128, dtype=torch.float16, device="cuda")
    C2 = torch.zeros(128, 128, device="cuda")
    n1 = g.launches
    g.run(A, A, C2)
    assert g.launches - n1 == 1
    torch.cuda.synchronize()
    g.close()


# ------------------------------------------------------------------------------ failure detection
@pytest.mark.parametrize("site,status", [("tmap", G.GEMM_ERR_CUDA), ("launch", G.GEMM_ERR_CUDA),
                                         ("alloc", G.GEMM_ERR_OOM)])
def test_host_fault_injection(handles, site, status, monkeypatch):
    monkeypatch.setenv("GEMM_TEST_FAIL", site)
    g = G.Gemm(0)
    monkeypatch.delenv("GEMM_TEST_FAIL")
    w = W.WORKLOADS[4] if site == "alloc" else W.problem(64, 64, 64, seed=1)
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d)
    st = g.run(dd["A"], dd["B"], C, M=w.M, N=w.N, K=w.K, layoutA=w.layoutA, layoutB=w.layoutB,
               alpha=w.alpha, beta=w.beta, check=False)
    assert st == status
    assert "forced failure" in g.last_error()
    g.close()
    # the process and the device stay usable
    _run_check(handles["auto"], W.problem(64, 64, 64, seed=2))


def test_optin_fault_fails_create(monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    monkeypatch.setenv("GEMM_TEST_FAIL", "optin")
    st, h = G.gemm_create(0)
    assert st == G.GEMM_ERR_CUDA and not h.value


@pytest.mark.parametrize("cfg", CONFIGS)
def test_bounded_wait_expires_and_reports(handles, cfg):
    """The producer of cluster 0 never issues stage 3, so the MMA issuer's wait runs out after
    200 ms; the kernel records the timeout, frees its TMEM and returns; the next call works.  (No
    split: with K split over clusters, cluster 0 might not reach stage 3.)"""
    g = G.Gemm(0, config=cfg, timeout_ms=200, debug_skip_stage=3, stream_k=0)
    w = W.problem(256, 256, 1024, seed=21)
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d)
    run_gpu(g, w, dd, C)
    st = g.status()
    assert st == G.GEMM_ERR_TIMEOUT, G.gemm_status_string(st)
    assert "mma" in g.last_error() or "producer" in g.last_error() or "epilogue" in g.last_error()
    assert g.status() == G.GEMM_OK       # the word was cleared
    g.close()
    _run_check(handles[cfg], W.problem(256, 256, 1024, seed=22))


# ------------------------------------------------------------------------------ stream-K tail
SK_CASES = {
    0: dict(M=2126, N=2460, K=300, dtype_out="f16", bias=True),               # 17 x 10 = 170 tiles > 152
    1: dict(M=2274, N=2300, K=700, dtype_out="bf16", dtype_in="bf16"),       # 9 x 9 = 81 tiles > 76
    2: dict(M=1650, N=1640, K=200, dtype_out="f32", alpha=0.5, beta=1.0),   # 13 x 13 = 169 > 152
    3: dict(M=2250, N=1250, K=450, dtype_out="f32", layoutB="col"),         # 9 x 10 = 90 > 76
    4: dict(M=2274, N=2300, K=700, dtype_out="f32", layoutA="col"),         # 81 tiles > 76, 6 k-tiles of 128
    5: dict(M=2250, N=4500, K=320, dtype_out="f16", bias=True, layoutB="col"),  # 9 x 9 = 81 tiles > 76
}


@pytest.mark.parametrize("cfg", CONFIGS)
def test_stream_k_tail_parity(cfg):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    c = dict(SK_CASES[cfg])
    w = W.problem(c.pop("M"), c.pop("N"), c.pop("K"), seed=100 + cfg, **c)
    st, plan = G.gemm_plan(w.M, w.N, w.K, w.K if w.layoutA == "row" else w.M, w.N if w.layoutB == "row" else w.K,
                           w.N, G.DTYPE_CODES[w.dtype_in], G.DTYPE_CODES[w.dtype_out], G.LAYOUT_CODES[w.layoutA],
                           G.LAYOUT_CODES[w.layoutB], w.beta, torch.cuda.get_device_properties(0).multi_processor_count,
                           0, cfg, 1)
    assert st == G.GEMM_OK and plan.stream_k == 1
    with G.Gemm(0, config=cfg, stream_k=1, sync_check=1) as g:
        for _ in range(2):                          # the second launch runs with the next epoch
            _run_check(g, w)


def test_stream_k_matches_data_parallel_on_integers():
    """Split tiles add two partial sums; with small integers both schedules are exact and equal."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    M, N, K = 2304, 2304, 1280                      # 81 tiles of 256 x 256 on 76 clusters
    A = W.small_ints(M, K, "f16", 5).cuda()
    B = W.small_ints(K, N, "f16", 6).cuda()
    outs = []
    for sk in (0, 1):
        C = torch.empty(M, N, dtype=torch.float32, device="cuda")
        with G.Gemm(0, config=1, stream_k=sk, sync_check=1) as g:
            g.run(A, B, C)
        outs.append(C)
    torch.cuda.synchronize()
    ref = (A.cpu().to(torch.int64) @ B.cpu().to(torch.int64)).to(torch.float32)
    assert torch.equal(outs[0].cpu(), ref)
    assert torch.equal(outs[1].cpu(), ref)


@pytest.mark.parametrize("group", [0, 1, 3, 16, 40])
def test_raster_groups_cover_every_tile_once(group):
    """Any raster group (the planner's, 1, one that does not divide the tile rows, or more rows than
    there are) visits every tile exactly once: small integers give the exact product, and the plan
    reports the group the kernel ran with."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    M, N, K = 4352, 1280, 512                       # 17 x 5 tiles of 256 x 256 on 76 clusters
    A = W.small_ints(M, K, "f16", 7).cuda()
    B = W.small_ints(K, N, "f16", 8).cuda()
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    with G.Gemm(0, config=4, raster_group=group, sync_check=1) as g:
        g.run(A, B, C)
        plan = g.last_plan()
    torch.cuda.synchronize()
    assert plan["tiles_m"] == 17
    assert plan["raster_group"] == (min(group, 17) if group > 0 else 9)   # 17 rows: two groups of 9
    ref = (A.cpu().to(torch.int64) @ B.cpu().to(torch.int64)).to(torch.float32)
    assert torch.equal(C.cpu(), ref)


# Fewer tiles than clusters: each tile's K range is split over several clusters and the head adds
# every following cluster's partial (split-K).  K is long enough for several sources per tile.
SPLIT_CASES = {
    0: dict(M=300, N=500, K=3000, dtype_out="f16", bias=True),               # 3 x 2 tiles, 47 k-tiles
    1: dict(M=500, N=300, K=4100, dtype_out="bf16", dtype_in="bf16"),        # 2 x 2 tiles
    2: dict(M=250, N=250, K=2500, dtype_out="f32", alpha=0.5, beta=1.0),     # 2 x 2 tiles
    3: dict(M=700, N=250, K=1500, dtype_out="f32", layoutB="col"),           # 3 x 2 tiles
    4: dict(M=600, N=700, K=3000, dtype_out="f32", layoutA="col"),           # 3 x 3 tiles, 24 k-tiles of 128
    5: dict(M=300, N=1000, K=2000, dtype_out="f16", bias=True, layoutA="col"),
}


def _plan_for(w, cfg, sk):
    return G.gemm_plan(w.M, w.N, w.K, w.K if w.layoutA == "row" else w.M, w.N if w.layoutB == "row" else w.K,
                       w.N, G.DTYPE_CODES[w.dtype_in], G.DTYPE_CODES[w.dtype_out], G.LAYOUT_CODES[w.layoutA],
                       G.LAYOUT_CODES[w.layoutB], w.beta, torch.cuda.get_device_properties(0).multi_processor_count,
                       0, cfg, sk)


@pytest.mark.parametrize("dout,cfg", [("bf16", 4), ("f32", 7), ("f16", 2)])
def test_bias_unaligned_matches_aligned(dout, cfg):
    """A bias one element past a 16-byte boundary takes the scalar loads, an aligned one the 16-byte
    vector loads; both add the same values, so C is bit-identical and matches the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    w = W.problem(300, 520, 256, dtype_in="bf16" if dout == "bf16" else "f16", dtype_out=dout, bias=True,
                  seed=280 + cfg)
    d = W.generate(w)
    dd = device_inputs(d)
    store = torch.empty(w.N + 8, dtype=W.DTYPES[dout], device="cuda")
    store[1:w.N + 1].copy_(dd["bias"])
    outs = []
    for bias in (dd["bias"], store[1:w.N + 1]):
        C = alloc_c(w, d)
        with G.Gemm(0, config=cfg, sync_check=1) as g:
            g.run(dd["A"], dd["B"], C, M=w.M, N=w.N, K=w.K, bias=bias)
        torch.cuda.synchronize()
        rep = compare(w, d, C)
        assert rep["passed"], rep
        outs.append(C)
    assert torch.equal(outs[0], outs[1])


# Every tile split over the same number S of consecutive clusters with equal k ranges: the partials
# meet as a reduce-scatter, each part finishing 1/S of the tile's epilogue blocks (S = 2, 4, 8).
RS_CASES = [
    (7, 0, dict(M=300, N=200, K=2048, dtype_out="f16", bias=True)),                       # S = 4, ragged tiles
    (7, 0, dict(M=1000, N=130, K=4096, dtype_out="f32", layoutB="col", alpha=0.5, beta=1.0)),   # S = 4, C_in
    (7, 0, dict(M=520, N=264, K=1536, dtype_out="bf16", dtype_in="bf16")),                # S = 4
    (7, 0, dict(M=1000, N=128, K=8192, dtype_out="f32", layoutB="col", beta=1.0)),        # S = 8, C_in
    (2, 0, dict(M=256, N=256, K=4096, dtype_out="f32", bias=True, layoutA="col")),        # S = 8
    (4, 12, dict(M=640, N=512, K=2048, dtype_out="f16", bias=True)),                      # 2-SM pairs, S = 2
    (4, 24, dict(M=640, N=512, K=2048, dtype_out="f32", beta=1.0)),                       # 2-SM pairs, S = 4
    (4, 0, dict(M=600, N=700, K=3000, dtype_out="bf16", dtype_in="bf16", layoutA="col")),  # S = 4, K tail
    (10, 0, dict(M=256, N=256, K=8192, dtype_in="e4m3", layoutB="col", dtype_out="f16")),  # FP8, S = 8
]


def _rs_plan(w, cfg, mc):
    st, plan = G.gemm_plan(w.M, w.N, w.K, w.K if w.layoutA == "row" else w.M, w.N if w.layoutB == "row" else w.K,
                           w.N, G.DTYPE_CODES[w.dtype_in], G.DTYPE_CODES[w.dtype_out], G.LAYOUT_CODES[w.layoutA],
                           G.LAYOUT_CODES[w.layoutB], w.beta, torch.cuda.get_device_properties(0).multi_processor_count,
                           mc, cfg, 1)
    assert st == G.GEMM_OK
    tiles = plan.tiles_m * plan.tiles_n
    k_tiles = -(-w.K // plan.block_k)
    split = plan.clusters // tiles
    assert plan.stream_k == 1 and plan.dp_tiles == 0 and plan.clusters == tiles * split
    assert split in (2, 4, 8) and k_tiles % split == 0, (split, k_tiles)
    return plan


@pytest.mark.parametrize("i", range(len(RS_CASES)))
def test_split_k_reduce_scatter_parity(i):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    cfg, mc, c = RS_CASES[i]
    c = dict(c)
    w = W.problem(c.pop("M"), c.pop("N"), c.pop("K"), seed=260 + i, **c)
    _rs_plan(w, cfg, mc)
    with G.Gemm(0, config=cfg, stream_k=1, max_clusters=mc, sync_check=1) as g:
        for _ in range(2):                                      # the second launch runs with the next epoch
            _run_check(g, w)


@pytest.mark.parametrize("cfg,mc,M,N,K", [(7, 0, 300, 200, 2048), (4, 24, 640, 512, 2048), (2, 0, 256, 256, 4096)])
def test_split_k_reduce_scatter_integers_exact(cfg, mc, M, N, K):
    """Small integers: every part's sum and their total are exact, in any order of addition."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    _rs_plan(W.problem(M, N, K), cfg, mc)
    A = W.small_ints(M, K, "f16", 40 + cfg).cuda()
    B = W.small_ints(K, N, "f16", 41 + cfg).cuda()
    ref = (A.cpu().to(torch.int64) @ B.cpu().to(torch.int64)).to(torch.float32)
    for sk in (1, 0):
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        with G.Gemm(0, config=cfg, stream_k=sk, max_clusters=mc, sync_check=1) as g:
            g.run(A, B, C)
        torch.cuda.synchronize()
        assert torch.equal(C.cpu(), ref), sk


def test_split_k_reduce_scatter_bounded_wait():
    """Cluster 0 (part 0 of tile 0) never receives its second stage: its MMA wait runs out, so its
    partials are never written, and the owning warps of tile 0's other three parts give up on their
    flags after 200 ms.  The timeout is reported and the next call works."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    w = W.problem(300, 200, 2048, dtype_out="f16", bias=True, seed=270)
    _rs_plan(w, 7, 0)
    d = W.generate(w)
    dd = device_inputs(d)
    C = alloc_c(w, d)
    g = G.Gemm(0, config=7, stream_k=1, timeout_ms=200, debug_skip_stage=1)
    run_gpu(g, w, dd, C)
    st = g.status()
    assert st == G.GEMM_ERR_TIMEOUT, G.gemm_status_string(st)
    assert g.status() == G.GEMM_OK
    g.close()
    with G.Gemm(0, config=7, stream_k=1, sync_check=1) as g2:
        _run_check(g2, w)


@pytest.mark.parametrize("cfg", CONFIGS)
def test_split_k_parity(cfg):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    c = dict(SPLIT_CASES[cfg])
    w = W.problem(c.pop("M"), c.pop("N"), c.pop("K"), seed=200 + cfg, **c)
    st, plan = _plan_for(w, cfg, 1)
    assert st == G.GEMM_OK and plan.stream_k == 1 and plan.dp_tiles == 0
    assert plan.clusters > plan.tiles_m * plan.tiles_n          # a tile spans several clusters
    with G.Gemm(0, config=cfg, stream_k=1, sync_check=1) as g:
        outs = []
        for _ in range(2):                                      # the second launch runs with the next epoch
            _, C, _ = _run_check(g, w)
            outs.append(C.clone())
        assert g.last_plan()["clusters"] == plan.clusters
    assert torch.equal(outs[0], outs[1])                        # partials are added in a fixed order


@pytest.mark.parametrize("cfg", [0, 2, 4])
def test_split_k_matches_data_parallel_on_integers(cfg):
    """Several partial sums per tile; with small integers every schedule is exact."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    M, N, K = 384, 512, 6144
    A = W.small_ints(M, K, "f16", 15 + cfg).cuda()
    B = W.small_ints(K, N, "f16", 16 + cfg).cuda()
    ref = (A.cpu().to(torch.int64) @ B.cpu().to(torch.int64)).to(torch.float32)
    for sk in (0, 1):
        C = torch.empty(M, N, dtype=torch.float32, device="cuda")
        with G.Gemm(0, config=cfg, stream_k=sk, sync_check=1) as g:
            g.run(A, B, C)
            torch.cuda.synchronize()
            plan = g.last_plan()
        assert plan["stream_k"] == sk
        assert torch.equal(C.cpu(), ref), (cfg, sk)


def test_three_d_and_two_d_tensor_maps_agree(monkeypatch):
    """Where the extents allow a 3-D operand map (one box per stage) the result must equal the
    one-box-per-slab 2-D path bit for bit: same data in the same shared-memory layout."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    for (la, lb, cfg) in [("row", "row", 4), ("col", "col", 1), ("row", "col", 0), ("col", "row", 4)]:
        w = W.problem(640, 768, 512, dtype_in="bf16", dtype_out="f32", layoutA=la, layoutB=lb, bias=True,
                      seed=len(la) + 3 * len(lb) + cfg)
        d = W.generate(w)
        dd = device_inputs(d)
        outs = []
        for rank in ("2", "3"):
            monkeypatch.setenv("GEMM_TMA_RANK", rank)
            with G.Gemm(0, config=cfg, sync_check=1) as g:
                C = alloc_c(w, d)
                run_gpu(g, w, dd, C)
                torch.cuda.synchronize()
                outs.append(C.cpu())
        assert torch.equal(outs[0], outs[1]), (la, lb, cfg)
        assert compare(w, d, outs[1].cuda())["passed"]


def test_last_plan_reports_the_run():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    with G.Gemm(0, config=4) as g:
        assert g.last_plan() == {}
        w = W.problem(600, 700, 256, seed=3)
        d = W.generate(w)
        dd = device_inputs(d)
        C = alloc_c(w, d)
        run_gpu(g, w, dd, C)
        p = g.last_plan()
        assert p["config"] == 4 and p["block_k"] == 128 and p["tiles_m"] == 3 and p["tiles_n"] == 3
        assert 1 <= p["clusters"] <= 9


@pytest.mark.parametrize("cfg,mc,c", [
    (4, 0, dict(M=2274, N=2300, K=700, dtype_out="f32", layoutA="col")),             # stream-K heads
    (4, 24, dict(M=640, N=512, K=2048, dtype_out="f32", beta=1.0)),                  # reduce-scatter, S = 4
    (7, 0, dict(M=300, N=200, K=2048, dtype_out="f16", bias=True)),                  # reduce-scatter, S = 4
    (7, 32, dict(M=40, N=1024, K=4096, dtype_out="f32", layoutB="col", beta=1.0)),  # C^T, reduce-scatter, S = 4
])
def test_graph_replay_with_stream_k_hand_off(cfg, mc, c):
    """A captured call replayed several times, with new A each time, matches the oracle every time: the
    hand-off flags are reset by their consumer, so a replay (same epoch) never reads a stale partial."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    c = dict(c)
    w = W.problem(c.pop("M"), c.pop("N"), c.pop("K"), seed=900 + cfg + mc, **c)
    ds = [W.generate(w)] + [W.generate(W.problem(w.M, w.N, w.K, seed=901 + i + cfg + mc, **c)) for i in range(3)]
    dd = device_inputs(ds[0])
    C = alloc_c(w, ds[0])
    Cin = C.clone()
    g = G.Gemm(0, config=cfg, stream_k=1, max_clusters=mc)
    try:
        run_gpu(g, w, dd, C)                                  # warm-up: the partial buffers are allocated here
        torch.cuda.synchronize()
        assert g.last_plan()["stream_k"] == 1
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run_gpu(g, w, dd, C)
        for d in ds[1:]:
            A = d["A"]
            dd["A"].copy_(A.cuda())                           # new A in the captured buffer
            C.copy_(Cin)
            graph.replay()
            torch.cuda.synchronize()
            want = dict(ds[0], A=A)
            rep = compare(w, want, C)
            assert rep["passed"], rep
        assert g.status() == G.GEMM_OK
    finally:
        g.close()
