"""C-ABI boundary checks that need no GPU: the library loads, exports every declared symbol,
validates arguments and plans calls (config choice, grid, repack, workspace) on the host."""
import ctypes
import os
import subprocess
import sys

import pytest

from bf16_tensor_core_gb300 import gemm as G


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    from bf16_tensor_core_gb300 import build
    build.build()
    return G.load_library()


def test_exports_every_declared_symbol(lib):
    names = G.header_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/gemm.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", str(G.LIB_PATH)], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    assert set(names) <= exported


def _header_prototypes():
    """Each declared function's parameter types, parsed from include/gemm.h (comments removed)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", G.HEADER.read_text(), flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(gemm_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = " ".join(m.group(2).split())
        protos[m.group(1)] = [] if params in ("", "void") else [q.strip() for q in params.split(",")]
    return protos


def _ctypes_kind(param: str):
    """The ctypes type a C parameter must be marshalled as (pointers and handles as void*)."""
    if "*" in param or param.startswith("gemm_handle_t"):
        return "ptr"
    if param.startswith("int64_t"):
        return ctypes.c_int64
    if param.startswith("float"):
        return ctypes.c_float
    return ctypes.c_int    # int and the enums


def test_bindings_match_the_header(lib):
    protos = _header_prototypes()
    assert set(protos) == set(G.header_functions())
    for name, params in protos.items():
        argtypes = getattr(lib, name).argtypes
        assert argtypes is not None and len(argtypes) == len(params), name
        for param, t in zip(params, argtypes):
            want = _ctypes_kind(param)
            if want == "ptr":
                assert t is ctypes.c_void_p or hasattr(t, "_type_") and issubclass(t, ctypes._Pointer), (name, param)
            else:
                assert t is want, (name, param, t)


def test_status_strings(lib):
    for code, name in [(0, "GEMM_OK"), (1, "GEMM_ERR_INVALID_ARG"), (2, "GEMM_ERR_UNSUPPORTED"),
                       (3, "GEMM_ERR_ALIGNMENT"), (4, "GEMM_ERR_CUDA"), (5, "GEMM_ERR_TIMEOUT"),
                       (6, "GEMM_ERR_OOM")]:
        assert G.gemm_status_string(code) == name
    assert G.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"


def test_options_default(lib):
    o = G.gemm_options_default()
    assert o.struct_size == ctypes.sizeof(G.gemm_options_t)
    assert o.config == -1 and o.timeout_ms == 2000 and o.debug_skip_stage == -1


def test_config_table(lib):
    n = G.gemm_num_configs()
    assert n == 11
    seen = set()
    for i in range(n):
        st, c = G.gemm_config_info(i)
        assert st == G.GEMM_OK and c.id == i
        assert c.block_m == 128 * c.cta_group and c.block_k in (64, 128, 256)
        assert c.block_n in (64, 128, 256, 512) and c.smem_bytes <= 232448
        assert c.threads == (448 if c.b_q4_0 else 320)        # Q4_0: 8 more dequantisation warps, 4 fewer epilogue
        stage = (128 + c.block_n // c.cta_group) * c.block_k * c.in_bytes
        assert c.block_k * c.in_bytes in (128, 256)                  # one or two 128-byte swizzle spans of K
        assert c.smem_bytes >= c.stages * stage
        seen.add((c.cta_group, c.block_n, c.block_k, c.b_q4_0, c.in_bytes))
    assert seen == {(1, 128, 64, 0, 2), (1, 256, 64, 0, 2), (2, 128, 64, 0, 2), (2, 256, 64, 0, 2),
                    (2, 256, 128, 0, 2), (2, 512, 64, 0, 2), (2, 256, 128, 1, 2), (1, 64, 128, 0, 2),
                    (2, 256, 256, 0, 1), (1, 64, 256, 0, 1), (1, 128, 128, 0, 1)}
    assert G.gemm_config_info(n)[0] == G.GEMM_ERR_UNSUPPORTED


def test_null_handle_and_create_without_gpu(lib):
    assert G.gemm_destroy(None) == G.GEMM_OK
    assert lib.gemm_run(None, 1, 1, 1, None, 1, None, 1, None, 1, 0, 0, 0, 0, 1.0, 0.0, None, None) == \
        G.GEMM_ERR_INVALID_ARG
    assert lib.gemm_create(None, 0, None) == G.GEMM_ERR_INVALID_ARG
    import torch
    if not torch.cuda.is_available():
        st, h = G.gemm_create(0)
        assert st in (G.GEMM_ERR_CUDA, G.GEMM_ERR_INVALID_ARG) and not h.value


def plan(M, N, K, lda=None, ldb=None, ldc=None, din=0, dout=2, la=0, lb=0, beta=0.0, config=-1, sms=152, sk=-1):
    lda = lda if lda is not None else (K if la == 0 else M)
    ldb = ldb if ldb is not None else (N if lb == 0 else K)
    ldc = ldc if ldc is not None else N
    return G.gemm_plan(M, N, K, max(lda, 1), max(ldb, 1), max(ldc, 1), din, dout, la, lb, beta, sms, 0, config, sk)


@pytest.mark.parametrize("args,status", [
    (dict(M=-1, N=4, K=4), G.GEMM_ERR_INVALID_ARG),
    (dict(M=4, N=-1, K=4), G.GEMM_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=-1), G.GEMM_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4, din=2), G.GEMM_ERR_INVALID_ARG),      # f32 operands are not a kind::f16 input
    (dict(M=4, N=4, K=4, dout=7), G.GEMM_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4, la=2), G.GEMM_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=8, lda=7), G.GEMM_ERR_INVALID_ARG),      # lda < K for row-major A
    (dict(M=9, N=4, K=8, la=1, lda=8), G.GEMM_ERR_INVALID_ARG),  # lda < M for column-major A
    (dict(M=4, N=9, K=8, ldb=8), G.GEMM_ERR_INVALID_ARG),      # ldb < N for row-major B
    (dict(M=4, N=9, K=8, lb=1, ldb=7), G.GEMM_ERR_INVALID_ARG),  # ldb < K for B stored N x K
    (dict(M=4, N=9, K=8, ldc=8), G.GEMM_ERR_INVALID_ARG),
    (dict(M=2 ** 31, N=4, K=4), G.GEMM_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4, config=11), G.GEMM_ERR_UNSUPPORTED),
    (dict(M=4, N=4, K=4, sms=0), G.GEMM_ERR_INVALID_ARG),
    (dict(M=4, N=4, K=4), G.GEMM_OK),
])
def test_plan_validation(lib, args, status):
    st, _ = plan(**args)
    assert st == status


def test_plan_degenerate(lib):
    st, p = plan(0, 100, 100)
    assert st == G.GEMM_OK and p.kernels == 0
    st, p = plan(100, 0, 100)
    assert st == G.GEMM_OK and p.kernels == 0
    st, p = plan(100, 100, 0)
    assert st == G.GEMM_OK and p.kernels == 1


def test_q4_0_config_is_not_a_plain_gemm_config(lib):
    q4 = [i for i in range(G.gemm_num_configs()) if G.gemm_config_info(i)[1].b_q4_0]
    assert q4 == [6]
    st, p = plan(4096, 4096, 4096, dout=0, config=6)       # f16 B cannot use the Q4_0 kernel
    assert st == G.GEMM_ERR_UNSUPPORTED
    for shape in [(512, 512, 512), (4096, 4096, 4096), (64, 4096, 4096), (1000, 3000, 2048)]:
        st, p = plan(*shape, dout=0)
        assert st == G.GEMM_OK and p.config != 6


def plan_q4(M, N, K, *, lda=None, la=0, ldbq=None, dout=2, config=-1, sk=-1, sms=152):
    lda = lda if lda is not None else (K if la == 0 else M)
    ldbq = ldbq if ldbq is not None else K // 32 * 18
    return G.gemm_plan_q4_0(M, N, K, max(lda, 1), la, ldbq, max(N, 1), dout, 0.0, sms, 0, config, sk)


def test_q4_0_routes(lib):
    """gemm_run_q4_0: the CUDA-core kernel for M <= 8 (row-major A), the fused kernel for a few
    output-tile rows, the separate pass + f16 GEMM once the fused kernel would dequantise B for
    many tile rows (it does so once per row of output tiles)."""
    for M in (1, 8):
        st, p = plan_q4(M, 4096, 4096)
        assert st == G.GEMM_OK and p.gemv == 1 and p.q4_dequant == 0 and p.config == -1 and p.kernels == 1
    st, p = plan_q4(4, 4096, 4096, la=1)                   # column-major A: not the CUDA-core kernel
    assert st == G.GEMM_OK and p.gemv == 0 and p.config == 6
    for M in (9, 64, 256):
        st, p = plan_q4(M, 11008, 4096)
        assert st == G.GEMM_OK and p.gemv == 0 and p.q4_dequant == 0 and p.config == 6 and p.kernels == 1
    for M in (1024, 2048, 8192):
        st, p = plan_q4(M, 11008, 4096, dout=1)
        assert st == G.GEMM_OK and p.q4_dequant == 1 and p.config not in (-1, 6) and p.kernels == 2
        assert p.workspace_bytes >= 11008 * 4096 * 2


def test_q4_0_route_by_config(lib):
    st, p = plan_q4(2048, 11008, 4096, config=6)            # the fused kernel on request
    assert st == G.GEMM_OK and p.config == 6 and p.q4_dequant == 0
    st, p = plan_q4(64, 4096, 4096, config=4)               # a plain config: separate pass + that config
    assert st == G.GEMM_OK and p.config == 4 and p.q4_dequant == 1 and p.kernels == 2
    st, p = plan_q4(1, 4096, 4096, config=6)                # an explicit config overrides the small-M kernel
    assert st == G.GEMM_OK and p.config == 6 and p.gemv == 0


@pytest.mark.parametrize("kw,status", [
    (dict(M=64, N=64, K=48), G.GEMM_ERR_INVALID_ARG),                 # K not whole blocks
    (dict(M=64, N=64, K=64, ldbq=35), G.GEMM_ERR_INVALID_ARG),        # odd pitch
    (dict(M=64, N=64, K=64, ldbq=34), G.GEMM_ERR_INVALID_ARG),        # pitch below K/32*18
    (dict(M=64, N=64, K=64, config=99), G.GEMM_ERR_UNSUPPORTED),
    (dict(M=0, N=64, K=64), G.GEMM_OK),
])
def test_q4_0_plan_validation(lib, kw, status):
    st, _ = plan_q4(**kw)
    assert st == status


def test_plan_few_rows_use_the_cuda_core_kernel(lib):
    # M <= 8, B stored N x K with a 16-byte pitch, K a multiple of 8: the CUDA-core kernel.
    for M in (1, 5, 8):
        st, p = plan(M, 4096, 4096, dout=0, lb=1)
        assert st == G.GEMM_OK and p.gemv == 1 and p.config == -1 and p.kernels == 1
    assert plan(9, 4096, 4096, dout=0, lb=1)[1].gemv == 0                 # 9 rows: tensor cores
    assert plan(4, 4096, 4096, dout=0, lb=0)[1].gemv == 0                 # B stored K x N
    assert plan(4, 4096, 4100, dout=0, lb=1)[1].gemv == 0                 # K not a multiple of 8
    assert plan(4, 4096, 4096, dout=0, lb=1, ldb=4100)[1].gemv == 0       # pitch not 16-byte aligned
    assert plan(4, 4096, 4096, din=G.GEMM_E4M3, dout=0, lb=1)[1].gemv == 0   # 8-bit inputs: tensor cores
    assert plan(4, 4096, 4096, dout=0, lb=1, config=7)[1].gemv == 0       # a forced config


def test_plan_skinny_products_are_transposed(lib):
    # A few rows of C against many columns: the kernel computes C^T with C's columns as its rows.
    for M in (1, 16, 64):
        st, p = plan(M, 4096, 4096, dout=0)
        assert st == G.GEMM_OK and p.transposed == 1
        assert p.tiles_m == 4096 // p.block_m and p.tiles_n == 1 and p.tma_store == 0
    st, p = plan(65, 4096, 4096, dout=0)                  # more rows: the plain product
    assert p.transposed == 0
    st, p = plan(16, 64, 4096, dout=0)                    # nothing to gain with 64 columns
    assert p.transposed == 0
    st, p = plan(16, 4096, 4096, dout=0, config=4)        # a forced config keeps the plain product
    assert p.transposed == 0 and p.config == 4
    # operand checks still refer to the caller's arrays
    st, p = plan(16, 4096, 4096, ldb=100)
    assert st == G.GEMM_ERR_INVALID_ARG


def test_plan_8bit_inputs(lib):
    E4M3, E5M2 = G.GEMM_E4M3, G.GEMM_E5M2
    st, p = plan(4096, 4096, 4096, din=E4M3, dout=0, lb=1)
    assert st == G.GEMM_OK and G.gemm_config_info(p.config)[1].in_bytes == 1 and p.block_k == 256
    st, p = plan(4096, 4096, 4096, din=E5M2, dout=2, lb=1)
    assert st == G.GEMM_OK and G.gemm_config_info(p.config)[1].in_bytes == 1
    assert plan(256, 256, 256, din=E4M3, lb=0)[0] == G.GEMM_ERR_UNSUPPORTED      # B must be K-major
    assert plan(256, 256, 256, din=E4M3, la=1, lb=1)[0] == G.GEMM_ERR_UNSUPPORTED
    assert plan(256, 256, 256, din=E4M3, lb=1, config=4)[0] == G.GEMM_ERR_UNSUPPORTED   # 16-bit config
    assert plan(256, 256, 256, din=0, lb=1, config=8)[0] == G.GEMM_ERR_UNSUPPORTED     # 8-bit config
    st, p = plan(300, 300, 1000, din=E4M3, lb=1, lda=1000, ldb=1000)   # 1000-byte rows: repacked as pairs
    assert st == G.GEMM_OK and p.repack_a == 1 and p.repack_b == 1
    assert plan(300, 300, 999, din=E4M3, lb=1, lda=999, ldb=999)[0] == G.GEMM_ERR_UNSUPPORTED  # odd rows
    st, p = plan(16, 4096, 4096, din=E4M3, lb=1)                       # skinny 8-bit: transposed, K-major
    assert st == G.GEMM_OK and p.transposed == 1 and G.gemm_config_info(p.config)[1].in_bytes == 1


def test_plan_tiles_and_grid(lib):
    for cfg in range(G.gemm_num_configs()):
        st, c = G.gemm_config_info(cfg)
        if c.b_q4_0 or c.in_bytes != 2:
            continue
        st, p = plan(4096, 4096, 4096, dout=0, config=cfg)
        assert st == G.GEMM_OK and p.config == cfg
        assert p.tiles_m == 4096 // c.block_m and p.tiles_n == 4096 // c.block_n
        slots = 152 // c.cta_group
        assert p.clusters == min(p.tiles_m * p.tiles_n, slots)
        # f16 output: TMA stores need each epilogue warp to drain whole 128-byte rows (64 columns)
        assert p.tma_store == (1 if c.block_n // 2 >= 64 else 0) and p.kernels == 1
        assert p.workspace_bytes == p.sk_partial_bytes
    st, p = plan(1000, 3000, 2050, config=1)
    assert (p.tiles_m, p.tiles_n) == (4, 12)           # partial last tiles: 1000 = 3*256 + 232, 3000 = 11*256 + 184
    st, p = plan(1, 1, 1, config=0)
    assert (p.tiles_m, p.tiles_n, p.clusters) == (1, 1, 1)


def test_plan_repack_and_workspace(lib):
    # 2050 halves = 4100 bytes is not a multiple of 16: both operands go through the workspace
    st, p = plan(1000, 3000, 2050, lda=2050, ldb=2050, la=0, lb=1, beta=1.0)
    assert st == G.GEMM_OK
    assert p.repack_a == 1 and p.repack_b == 1 and p.kernels == 2
    a_bytes = -(-1000 * 2056 * 2 // 256) * 256
    b_bytes = -(-3000 * 2056 * 2 // 256) * 256
    assert p.workspace_bytes == a_bytes + b_bytes + p.sk_partial_bytes
    assert p.tma_store == 1                             # 12000-byte rows: C_in loaded and C stored by TMA
    st, p = plan(64, 64, 64, lda=72, ldb=64)
    assert p.repack_a == 0 and p.repack_b == 0 and p.workspace_bytes == 0
    st, p = plan(64, 63, 64, ldc=63, dout=0)            # 126-byte rows: TMA cannot store C
    assert p.tma_store == 0
    st, p = plan(64, 60, 64, ldc=60, dout=2)            # 240-byte rows: TMA store is fine
    assert p.tma_store == 1


def test_plan_auto_choice_is_a_valid_config(lib):
    for (M, N, K) in [(512, 512, 512), (4096, 4096, 4096), (2048, 11008, 4096), (1000, 3000, 2050),
                      (8192, 8192, 8192), (1, 4096, 4096), (128, 128, 64)]:
        st, p = plan(M, N, K, dout=0)
        assert st == G.GEMM_OK and 0 <= p.config < G.gemm_num_configs()
        assert p.clusters >= 1 and p.raster_group >= 1 and p.raster_group <= p.tiles_m


@pytest.mark.parametrize("M,N,K,cfg,group", [
    (4096, 4096, 4096, 4, 8),        # 16 tile rows of 256: two groups of 8
    (1024, 4096, 4096, 4, 4),        # 4 tile rows: one group
    (8192, 8192, 8192, 4, 16),       # 32 tile rows: two groups of 16 (A panels 64 MiB per group)
    (6144, 6144, 4096, 4, 12),       # 24 tile rows: two groups of 12
    (8192, 8192, 16384, 4, 8),       # a group of 16 would hold 128 MiB of A panels: groups of 8
    (8192, 4096, 4096, 0, 16),       # 64 tile rows of 128: four groups of 16
])
def test_plan_raster_group(lib, M, N, K, cfg, group):
    """Tall products are rastered in as few groups of at most 16 tile rows as cover them (each group
    re-reads every B panel), unless a group's A panels would outgrow half the L2."""
    st, p = plan(M, N, K, dout=0, config=cfg)
    assert st == G.GEMM_OK and p.config == cfg
    assert p.raster_group == group, (M, N, K, p.tiles_m, p.raster_group)


def test_python_binding_fails_loudly_without_library(tmp_path):
    code = ("import sys; sys.path.insert(0, %r)\n"
            "from bf16_tensor_core_gb300 import gemm\n"
            "try:\n    gemm.load_library(%r)\nexcept OSError as e:\n    print('LOUD', e)\n") % (
        os.path.dirname(os.path.dirname(os.path.abspath(__file__))), str(tmp_path / "missing.so"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert "LOUD" in r.stdout


# ------------------------------------------------------------------------------ stream-K tail
def test_plan_stream_k(lib):
    st, p = plan(4096, 4096, 4096, dout=0, config=1)            # 256 tiles over 76 clusters: 3.37 waves
    assert st == G.GEMM_OK and p.stream_k == 1 and p.clusters == 76
    assert p.dp_tiles == (256 // 76 - 1) * 76
    assert p.sk_partial_bytes == 76 * 2 * 128 * 256 * 4
    st, p = plan(4096, 4096, 4096, dout=0, config=1, sk=0)
    assert p.stream_k == 0 and p.sk_partial_bytes == 0 and p.workspace_bytes == 0
    st, p = plan(256 * 19, 256 * 8, 1024, config=1)              # 152 tiles = 2 whole waves
    assert p.stream_k == 0
    st, p = plan(1024, 1024, 1024, config=1, sk=0)               # 16 tiles < 76 clusters, split-K off
    assert p.stream_k == 0 and p.clusters == 16
    st, p = plan(1024, 1024, 1024, config=1, sk=1)               # split-K: each tile over several clusters
    assert p.stream_k == 1 and p.dp_tiles == 0 and 16 < p.clusters <= 76
    st, p = plan(256 * 9, 256 * 9, 512, config=1, sk=1)          # 81 tiles: forced on
    assert p.stream_k == 1 and p.dp_tiles == 0
    st, p = plan(256 * 16, 256 * 19, 512, config=1)              # 304 tiles = 4.0 waves exactly
    assert p.stream_k == 0
    st, p = plan(256 * 11, 256 * 14, 4096, config=1)             # 154 tiles = 2.03 waves: last wave 3% full
    assert p.stream_k == 1 and p.dp_tiles == 76


def sk_units(T, P, KT, dp_tiles, cluster):
    """Python model of the kernel's per-cluster unit sequence (UnitIter)."""
    total = (T - dp_tiles) * KT
    base, extra = total // P, total % P
    out = [(t, 0, KT, "full") for t in range(cluster, dp_tiles, P)]
    it = cluster * base + min(cluster, extra)
    end = it + base + (1 if cluster < extra else 0)
    while it < end:
        rel, k0 = divmod(it, KT)
        seg_end = min((rel + 1) * KT, end)
        k1 = k0 + seg_end - it
        kind = "full" if (k0 == 0 and k1 == KT) else ("head" if k0 == 0 else "tail")
        out.append((dp_tiles + rel, k0, k1, kind))
        it = seg_end
    return out


def sk_sources(T, P, KT, dp_tiles, cluster, tile):
    """Clusters whose partials the head of `tile` adds: the following ranges that start before the tile ends."""
    total = (T - dp_tiles) * KT
    base, extra = total // P, total % P
    tile_end = (tile - dp_tiles + 1) * KT
    out = []
    src = cluster + 1
    while src < P and src * base + min(src, extra) < tile_end:
        out.append(src)
        src += 1
    return out


SCHEDULES = [(256, 76, 64, None), (1024, 76, 128, None), (344, 76, 64, None), (81, 76, 5, None),
             (170, 152, 8, None), (77, 76, 1, None), (151, 76, 3, None), (100, 7, 13, None),
             # fewer tiles than clusters: tiles split K-wise over several clusters
             (48, 76, 17, 0), (6, 48, 47, 0), (4, 32, 128, 0), (16, 128, 33, 0), (1, 8, 9, 0), (5, 37, 11, 0)]


@pytest.mark.parametrize("T,P,KT,dp", SCHEDULES)
def test_stream_k_schedule_covers_every_k_iteration_once(T, P, KT, dp):
    dp_tiles = (T // P - 1) * P if dp is None else dp
    cover = {}
    for c in range(P):
        units = sk_units(T, P, KT, dp_tiles, c)
        assert sum(1 for u in units if u[3] == "tail") <= 1           # one partial slot per cluster
        tails = [i for i, u in enumerate(units) if u[3] == "tail"]
        heads = [i for i, u in enumerate(units) if u[3] == "head"]
        n_dp = sum(1 for u in units if u[0] < dp_tiles)
        assert not tails or tails == [n_dp]                           # the tail segment comes first
        assert not heads or heads == [len(units) - 1]                 # the head segment comes last
        for (t, k0, k1, kind) in units:
            assert 0 <= t < T and 0 <= k0 < k1 <= KT
            for k in range(k0, k1):
                assert (t, k) not in cover
                cover[(t, k)] = (c, kind)
            if kind == "head":
                # The rest of the tile is exactly the first units of the source clusters, in order.
                srcs = sk_sources(T, P, KT, dp_tiles, c, t)
                assert srcs and srcs == list(range(c + 1, c + 1 + len(srcs)))
                k = k1
                for s in srcs:
                    first = sk_units(T, P, KT, dp_tiles, s)[sum(1 for u in sk_units(T, P, KT, dp_tiles, s)
                                                                if u[0] < dp_tiles)]
                    assert first[0] == t and first[1] == k and first[3] == "tail"
                    k = first[2]
                assert k == KT
            if kind == "tail":
                assert c > 0
    assert len(cover) == T * KT


# The plan of every bench workload on a 152-SM GB300, as the measurements and profiles quote it:
# (config, stream_k, dp_tiles, clusters, transposed, gemv, q4_dequant, kernels).
WORKLOAD_PLANS = {
    1: (7, 0, 0, 32, 0, 0, 0, 1),        # 512^3: 128 x 64 tiles on single SMs
    2: (4, 1, 152, 76, 0, 0, 0, 1),      # 4096^3: two whole waves, then the wave and a half split K-wise
    3: (4, 0, 0, 76, 0, 0, 0, 1),        # prefill bf16 + bias: data-parallel
    4: (4, 0, 0, 48, 0, 0, 0, 2),        # ragged: both operands repacked to 16-byte pitches, then the product
    5: (4, 1, 988, 76, 0, 0, 0, 1),      # 8192^3: only the partial last wave split
    6: (4, 0, 0, 76, 0, 0, 1, 2),        # prefill Q4_0: the separate dequantisation pass, then config 4
    7: (-1, 0, 0, 0, 0, 1, 0, 1),        # decode M = 1: the CUDA-core kernel
    8: (7, 1, 0, 128, 1, 0, 0, 1),       # decode M = 64: transposed product, split-K over 128 SMs
    9: (8, 1, 152, 76, 0, 0, 0, 1),      # 4096^3 E4M3
    10: (-1, 0, 0, 0, 0, 1, 0, 1),       # decode M = 1 with Q4_0 weights: the CUDA-core kernel
}


@pytest.mark.parametrize("wid", sorted(WORKLOAD_PLANS))
def test_bench_workload_plans(lib, wid):
    from bf16_tensor_core_gb300 import workloads as W
    w = W.WORKLOADS[wid]
    la = G.LAYOUT_CODES[w.layoutA]
    lda = w.K if w.layoutA == "row" else w.M
    if w.layoutB == "q4_0":
        st, p = G.gemm_plan_q4_0(w.M, w.N, w.K, lda, la, w.K // 32 * 18, w.N, G.DTYPE_CODES[w.dtype_out], beta=w.beta)
    else:
        ldb = w.N if w.layoutB == "row" else w.K
        st, p = G.gemm_plan(w.M, w.N, w.K, lda, ldb, w.N, G.DTYPE_CODES[w.dtype_in], G.DTYPE_CODES[w.dtype_out],
                            la, G.LAYOUT_CODES[w.layoutB], beta=w.beta)
    assert st == G.GEMM_OK
    got = (p.config, p.stream_k, p.dp_tiles, p.clusters, p.transposed, p.gemv, p.q4_dequant, p.kernels)
    assert got == WORKLOAD_PLANS[wid], (w.name, got)
    assert (p.repack_a, p.repack_b) == ((1, 1) if wid == 4 else (0, 0))


C_CLIENT = r"""
#include <stdio.h>
#include "gemm.h"

int main(void) {
    gemm_options_t o;
    gemm_plan_t p;
    gemm_config_info_t info;
    int n = gemm_num_configs();
    gemm_options_default(&o);
    if (o.config != -1) return 1;
    if (gemm_config_info(n - 1, &info) != GEMM_OK) return 2;
    if (gemm_plan(4096, 4096, 4096, 4096, 4096, 4096, GEMM_F16, GEMM_F16, GEMM_ROW, GEMM_ROW, 0.0f, 152, 0, -1, -1,
                  &p) != GEMM_OK) return 3;
    printf("configs %d plan %d tiles %d x %d status %s\n", n, p.config, p.tiles_m, p.tiles_n,
           gemm_status_string(GEMM_ERR_ALIGNMENT));
    return 0;
}
"""


def test_header_compiles_as_c_and_links(lib, tmp_path):
    """include/gemm.h is a plain C header: a C99 client built with gcc -Werror links against the
    library and gets the same plan as the Python binding, using host-only entry points."""
    import shutil
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(lib._name)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(root, "include"), str(src),
                        "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(lib._name), "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    st, p = plan(4096, 4096, 4096, dout=0)
    assert r.stdout.split()[:7] == ["configs", str(G.gemm_num_configs()), "plan", str(p.config), "tiles",
                                    str(p.tiles_m), "x"], r.stdout


def test_warp_specialised_kernel_uses_barriers_that_allow_diverged_warps():
    """The tensor-core kernel's roles reach its block- and cluster-wide barriers with lane 0 of the producer and
    MMA warps still working alone.  The .aligned forms (bar.sync / __syncthreads(), barrier.cluster.*.aligned,
    bar.red) need converged warps and were measured to release early there; only the forms that count each thread
    as it arrives may appear in the kernel and its PTX wrappers."""
    import re
    src = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bf16_tensor_core_gb300", "csrc")
    kernel = open(os.path.join(src, "gemm_kernel.cuh")).read()
    ptx = open(os.path.join(src, "ptx_sm103.cuh")).read()
    code = "\n".join(l for l in (kernel + ptx).splitlines() if not l.lstrip().startswith("//"))
    assert "__syncthreads" not in code
    assert not re.search(r"\bbar\.(sync|red|arrive)\b", code)
    assert not re.search(r"barrier\.cluster\.(arrive|wait)[.\w]*\.aligned", code)
    assert "barrier.sync 0" in code and "barrier.cluster.arrive.release;" in code
