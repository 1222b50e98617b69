"""CPU oracle for the dense GEMM (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.
"""
from .oracle import (  # noqa: F401
    OR_F16, OR_BF16, OR_F32, OR_E4M3, OR_E5M2, OR_ROW, OR_COL, decode_e4m3, decode_e5m2,
    build, lib_path, decode_f16, decode_bf16, decode_f32,
    gemm_ref, ulp_out, tolerance, check, error_metrics, epilogue_magnitude, num_cpus, decode,
    f64_to_f16_bits, q4_0_to_f16, gemm_ref_q4_0,
)
