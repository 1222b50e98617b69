"""ctypes binding of the C ABI in include/gemm.h (argument marshalling only).

Every function named like the C entry point forwards to it unchanged.  ``Gemm`` is a small
convenience wrapper that takes torch CUDA tensors and passes their device pointers, leading
dimensions and the current stream.  There is no fallback: if ``libgemm_gb300.so`` cannot be
loaded, importing the library raises.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libgemm_gb300.so"
HEADER = _PKG.parent / "include" / "gemm.h"

GEMM_F16, GEMM_BF16, GEMM_F32, GEMM_E4M3, GEMM_E5M2 = 0, 1, 2, 3, 4
GEMM_ROW, GEMM_COL = 0, 1
GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED, GEMM_ERR_ALIGNMENT = 0, 1, 2, 3
GEMM_ERR_CUDA, GEMM_ERR_TIMEOUT, GEMM_ERR_OOM = 4, 5, 6

DTYPE_CODES = {"f16": GEMM_F16, "bf16": GEMM_BF16, "f32": GEMM_F32, "e4m3": GEMM_E4M3, "e5m2": GEMM_E5M2}
LAYOUT_CODES = {"row": GEMM_ROW, "col": GEMM_COL}


class gemm_options_t(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_int), ("config", ctypes.c_int), ("timeout_ms", ctypes.c_int),
                ("sync_check", ctypes.c_int), ("raster_group", ctypes.c_int), ("max_clusters", ctypes.c_int),
                ("debug_skip_stage", ctypes.c_int), ("stream_k", ctypes.c_int), ("skinny", ctypes.c_int),
                ("pdl", ctypes.c_int)]


class gemm_config_info_t(ctypes.Structure):
    _fields_ = [("id", ctypes.c_int), ("cta_group", ctypes.c_int), ("block_m", ctypes.c_int),
                ("block_n", ctypes.c_int), ("block_k", ctypes.c_int), ("stages", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("threads", ctypes.c_int), ("b_q4_0", ctypes.c_int),
                ("in_bytes", ctypes.c_int)]


class gemm_plan_t(ctypes.Structure):
    _fields_ = [("config", ctypes.c_int), ("cta_group", ctypes.c_int), ("block_m", ctypes.c_int),
                ("block_n", ctypes.c_int), ("block_k", ctypes.c_int), ("stages", ctypes.c_int),
                ("tiles_m", ctypes.c_int), ("tiles_n", ctypes.c_int), ("clusters", ctypes.c_int),
                ("raster_group", ctypes.c_int), ("tma_store", ctypes.c_int), ("repack_a", ctypes.c_int),
                ("repack_b", ctypes.c_int), ("workspace_bytes", ctypes.c_int64), ("kernels", ctypes.c_int),
                ("stream_k", ctypes.c_int), ("dp_tiles", ctypes.c_int), ("sk_partial_bytes", ctypes.c_int64),
                ("transposed", ctypes.c_int), ("gemv", ctypes.c_int), ("q4_dequant", ctypes.c_int),
                ("split_cluster", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


class GemmError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} [{status}]")
        self.status = status


_lib = None


def load_library(path: Path | str | None = None):
    """Load libgemm_gb300.so (raises OSError if it is missing: there is no other implementation)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path else LIB_PATH
    if not p.exists():
        raise OSError(f"{p} not found: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(str(p))
    vp, i64, ci, cf = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.gemm_options_default.argtypes = [ctypes.POINTER(gemm_options_t)]
    lib.gemm_options_default.restype = None
    lib.gemm_create.argtypes = [ctypes.POINTER(vp), ci, ctypes.POINTER(gemm_options_t)]
    lib.gemm_create.restype = ci
    lib.gemm_run.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, ci, ci, ci, ci, cf, cf, vp, vp]
    lib.gemm_run.restype = ci
    lib.gemm_destroy.argtypes = [vp]
    lib.gemm_destroy.restype = ci
    lib.gemm_status_string.argtypes = [ci]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_last_error.argtypes = [vp]
    lib.gemm_last_error.restype = ctypes.c_char_p
    lib.gemm_get_device_status.argtypes = [vp, vp]
    lib.gemm_get_device_status.restype = ci
    lib.gemm_plan.argtypes = [i64, i64, i64, i64, i64, i64, ci, ci, ci, ci, cf, ci, ci, ci, ci,
                              ctypes.POINTER(gemm_plan_t)]
    lib.gemm_plan.restype = ci
    lib.gemm_plan_q4_0.argtypes = [i64, i64, i64, i64, ci, i64, i64, ci, cf, ci, ci, ci, ci,
                                   ctypes.POINTER(gemm_plan_t)]
    lib.gemm_plan_q4_0.restype = ci
    lib.gemm_num_configs.argtypes = []
    lib.gemm_num_configs.restype = ci
    lib.gemm_config_info.argtypes = [ci, ctypes.POINTER(gemm_config_info_t)]
    lib.gemm_config_info.restype = ci
    lib.gemm_launch_count.argtypes = [vp]
    lib.gemm_launch_count.restype = i64
    lib.gemm_last_plan.argtypes = [vp, ctypes.POINTER(gemm_plan_t)]
    lib.gemm_last_plan.restype = ci
    lib.gemm_run_noalloc.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ci, ci, ci, ci, cf, cf, vp, vp]
    lib.gemm_run_noalloc.restype = ci
    lib.gemm_noalloc_get_device_status.argtypes = [vp]
    lib.gemm_noalloc_get_device_status.restype = ci
    lib.gemm_run_q4_0.argtypes = [vp, i64, i64, i64, vp, i64, ci, vp, i64, vp, i64, ci, cf, cf, vp, vp]
    lib.gemm_run_q4_0.restype = ci
    lib.gemm_dequant_q4_0.argtypes = [vp, i64, i64, i64, vp, i64, vp]
    lib.gemm_dequant_q4_0.restype = ci
    if path is None:
        _lib = lib
    return lib


def header_functions() -> list[str]:
    """Names of the functions declared in include/gemm.h."""
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_[a-z0-9_]+)\s*\(", text)))


# ------------------------------------------------------------------ one-to-one forwarders
def gemm_options_default() -> gemm_options_t:
    o = gemm_options_t()
    load_library().gemm_options_default(ctypes.byref(o))
    return o


def gemm_create(device: int = 0, opt: gemm_options_t | None = None) -> tuple[int, ctypes.c_void_p]:
    h = ctypes.c_void_p()
    st = load_library().gemm_create(ctypes.byref(h), device, ctypes.byref(opt) if opt is not None else None)
    return st, h


def gemm_run(h, M, N, K, A, lda, B, ldb, C, ldc, dtype_in, dtype_out, layoutA, layoutB,
             alpha, beta, bias, stream) -> int:
    return load_library().gemm_run(h, M, N, K, A, lda, B, ldb, C, ldc, dtype_in, dtype_out, layoutA, layoutB,
                                   alpha, beta, bias, stream)


def gemm_destroy(h) -> int:
    return load_library().gemm_destroy(h)


def gemm_status_string(s: int) -> str:
    return load_library().gemm_status_string(s).decode()


def gemm_last_error(h) -> str:
    return load_library().gemm_last_error(h).decode()


def gemm_get_device_status(h, stream=None) -> int:
    return load_library().gemm_get_device_status(h, stream)


def gemm_plan(M, N, K, lda, ldb, ldc, dtype_in, dtype_out, layoutA, layoutB, beta=0.0, num_sms=152,
              max_clusters=0, config=-1, stream_k=-1) -> tuple[int, gemm_plan_t]:
    p = gemm_plan_t()
    st = load_library().gemm_plan(M, N, K, lda, ldb, ldc, dtype_in, dtype_out, layoutA, layoutB, beta, num_sms,
                                  max_clusters, config, stream_k, ctypes.byref(p))
    return st, p


def gemm_plan_q4_0(M, N, K, lda, layoutA, ldbq, ldc, dtype_out, beta=0.0, num_sms=152, max_clusters=0, config=-1,
                   stream_k=-1) -> tuple[int, gemm_plan_t]:
    p = gemm_plan_t()
    st = load_library().gemm_plan_q4_0(M, N, K, lda, layoutA, ldbq, ldc, dtype_out, beta, num_sms, max_clusters, config,
                                       stream_k, ctypes.byref(p))
    return st, p


def gemm_num_configs() -> int:
    return load_library().gemm_num_configs()


def gemm_config_info(i: int) -> tuple[int, gemm_config_info_t]:
    c = gemm_config_info_t()
    return load_library().gemm_config_info(i, ctypes.byref(c)), c


def gemm_launch_count(h) -> int:
    return load_library().gemm_launch_count(h)


def gemm_last_plan(h) -> tuple[int, gemm_plan_t]:
    p = gemm_plan_t()
    return load_library().gemm_last_plan(h, ctypes.byref(p)), p


def gemm_run_noalloc(M, N, K, A, lda, B, ldb, C, ldc, dtype_in, dtype_out, layoutA, layoutB,
                     alpha, beta, bias, stream) -> int:
    return load_library().gemm_run_noalloc(M, N, K, A, lda, B, ldb, C, ldc, dtype_in, dtype_out, layoutA,
                                           layoutB, alpha, beta, bias, stream)


def gemm_noalloc_get_device_status(stream=None) -> int:
    return load_library().gemm_noalloc_get_device_status(stream)


def gemm_run_q4_0(h, M, N, K, A, lda, layoutA, Bq, ldbq, C, ldc, dtype_out, alpha, beta, bias, stream) -> int:
    return load_library().gemm_run_q4_0(h, M, N, K, A, lda, layoutA, Bq, ldbq, C, ldc, dtype_out, alpha, beta,
                                        bias, stream)


def gemm_dequant_q4_0(Bq, ldbq, N, K, out, ldo, stream) -> int:
    return load_library().gemm_dequant_q4_0(Bq, ldbq, N, K, out, ldo, stream)


# ------------------------------------------------------------------ torch convenience wrapper
def _torch_code(t) -> int:
    import torch
    return {torch.float16: GEMM_F16, torch.bfloat16: GEMM_BF16, torch.float32: GEMM_F32,
            torch.float8_e4m3fn: GEMM_E4M3, torch.float8_e5m2: GEMM_E5M2}[t.dtype]


def _ld(t) -> int:
    """Leading dimension (elements) of a 2-D tensor with unit inner stride."""
    assert t.dim() == 2 and (t.stride(1) == 1 or t.size(1) <= 1), "inner dimension must be contiguous"
    return max(t.stride(0), t.size(1), 1)


class Gemm:
    """Owns one handle; ``run`` enqueues C <- alpha*op(A)*op(B) + beta*C + bias on the current stream."""

    def __init__(self, device: int = 0, **options):
        opt = gemm_options_default()
        for k, v in options.items():
            setattr(opt, k, int(v))
        st, h = gemm_create(device, opt)
        if st != GEMM_OK:
            raise GemmError(st, f"gemm_create failed: {gemm_status_string(st)}")
        self.h = h
        self.device = device

    def close(self):
        if self.h:
            gemm_destroy(self.h)
            self.h = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def launches(self) -> int:
        return gemm_launch_count(self.h)

    def last_plan(self) -> dict:
        st, p = gemm_last_plan(self.h)
        return p.as_dict() if st == GEMM_OK else {}

    def run(self, A, B, C, *, M=None, N=None, K=None, layoutA="row", layoutB="row", alpha=1.0, beta=0.0,
            bias=None, stream=None, check=True) -> int:
        """A, B, C: 2-D CUDA tensors in their STORED layout (see include/gemm.h)."""
        import torch
        la, lb = LAYOUT_CODES[layoutA], LAYOUT_CODES[layoutB]
        if M is None:
            M = A.size(0) if la == GEMM_ROW else A.size(1)
        if K is None:
            K = A.size(1) if la == GEMM_ROW else A.size(0)
        if N is None:
            N = B.size(1) if lb == GEMM_ROW else B.size(0)
        s = stream if stream is not None else torch.cuda.current_stream(C.device).cuda_stream
        st = gemm_run(self.h, M, N, K, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), C.data_ptr(), _ld(C),
                      _torch_code(A), _torch_code(C), la, lb, float(alpha), float(beta),
                      bias.data_ptr() if bias is not None else None, s)
        if check and st != GEMM_OK:
            raise GemmError(st, f"gemm_run: {gemm_status_string(st)}: {gemm_last_error(self.h)}")
        return st

    def run_q4_0(self, A, Bq, C, *, N, K=None, M=None, layoutA="row", alpha=1.0, beta=0.0, bias=None,
                 stream=None, check=True) -> int:
        """A: f16 activations (stored layout); Bq: uint8 tensor (N, ldbq) of Q4_0 blocks."""
        import torch
        la = LAYOUT_CODES[layoutA]
        if M is None:
            M = A.size(0) if la == GEMM_ROW else A.size(1)
        if K is None:
            K = A.size(1) if la == GEMM_ROW else A.size(0)
        s = stream if stream is not None else torch.cuda.current_stream(C.device).cuda_stream
        st = gemm_run_q4_0(self.h, M, N, K, A.data_ptr(), _ld(A), la, Bq.data_ptr(), _ld(Bq), C.data_ptr(), _ld(C),
                           _torch_code(C), float(alpha), float(beta), bias.data_ptr() if bias is not None else None, s)
        if check and st != GEMM_OK:
            raise GemmError(st, f"gemm_run_q4_0: {gemm_status_string(st)}: {gemm_last_error(self.h)}")
        return st

    def status(self, stream=None) -> int:
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        return gemm_get_device_status(self.h, s)

    def last_error(self) -> str:
        return gemm_last_error(self.h)
