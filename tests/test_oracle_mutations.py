"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each one.

Every mutant is compiled from an edited copy of ``oracle/gemm_oracle.c`` in a
temporary directory (the oracle itself is untouched) and the pins run against it
in a child process, so a mutant that reads out of bounds and crashes cannot take
the test session down (a crash counts as caught).
"""
import os
import subprocess
import sys
from pathlib import Path

import pytest

import oracle.oracle as oracle_mod

SRC = Path(oracle_mod.__file__).with_name("gemm_oracle.c")
TESTS = Path(__file__).resolve().parent

RUNNER = r"""
import ctypes, sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle.oracle as om
import test_oracle_pins as P
import test_oracle_q4_0 as Q
import test_oracle_fp8 as F8
om._lib = om.configure(ctypes.CDLL({lib!r}))
caught = []
for pin in P.PINS + Q.PINS + F8.PINS:
    try:
        pin()
    except Exception:
        caught.append(pin.__name__)
for shape in [(2, 3, 7), (7, 16, 17)]:
    try:
        P.test_brute_force_exact_rational(*shape)
    except Exception:
        caught.append("brute_force" + str(shape))
print("CAUGHT", ",".join(caught))
"""

MUTANTS = {
    "f16_exponent_bias": ("(int)expo - 25)", "(int)expo - 24)"),
    "bf16_subnormal_scale": ("ldexp((double)frac, -133)", "ldexp((double)frac, -132)"),
    "dropped_bias": ("if (j->biasd) v += j->biasd[col];", "(void)col;"),
    "beta_sign": ("v += j->beta * load_elem", "v -= j->beta * load_elem"),
    "bias_scaled_by_alpha": ("v += j->biasd[col];", "v += j->alpha * j->biasd[col];"),
    "transposed_a_row": ("layout == OR_ROW ? i * lda + k : k * lda + i",
                         "layout == OR_ROW ? k * lda + i : k * lda + i"),
    "transposed_b_col": ("layout == OR_ROW ? k * ldb + j : j * ldb + k",
                         "layout == OR_ROW ? k * ldb + j : k * ldb + j"),
    "dropped_last_k": ("for (int64_t k = 0; k < j->K; ++k) {\n            const double a",
                       "for (int64_t k = 0; k + 1 < j->K; ++k) {\n            const double a"),
    "cin_read_when_beta_zero": ("if (j->beta != 0.0) v +=", "if (1) v +="),
    "sign_dropped_f16": ("return sign ? -v : v;\n}\n\n/* bfloat16", "return v;\n}\n\n/* bfloat16"),
    # Q4_0 dequantisation and the binary16 encoder
    "q4_nibbles_swapped": ("const int lo = blk[2 + i] & 0x0f, hi = blk[2 + i] >> 4;",
                           "const int hi = blk[2 + i] & 0x0f, lo = blk[2 + i] >> 4;"),
    "q4_offset_7": ("d * (double)(lo - 8)", "d * (double)(lo - 7)"),
    "q4_scale_big_endian": ("(uint16_t)(blk[0] | (blk[1] << 8))", "(uint16_t)(blk[1] | (blk[0] << 8))"),
    "q4_block_stride_16": ("bq + n * ldbq + b * 18", "bq + n * ldbq + b * 16"),
    "f16_truncates": ("if (r > 0.5) return f + 1.0;", "if (r > 2.0) return f + 1.0;"),
    "f16_ties_away": ("return fmod(f, 2.0) == 0.0 ? f : f + 1.0;", "return f + 1.0;"),
    "f16_subnormal_scale": ("rne(ldexp(a, 24))", "rne(ldexp(a, 23))"),
    "f16_exponent_bias_enc": ("(((e + 15) << 10)", "(((e + 14) << 10)"),
    # 8-bit floats
    "e4m3_bias_8": ("(int)expo - 10);             /* (8 + frac)", "(int)expo - 11);             /* (8 + frac)"),
    "e4m3_no_nan": ("if (expo == 0xf && frac == 0x7) return NAN;", "(void)0;"),
    "e4m3_subnormal_scale": ("ldexp((double)frac, -9);", "ldexp((double)frac, -10);"),
    "e5m2_frac_bits": ("const unsigned frac = b & 0x3u;", "const unsigned frac = b & 0x7u;"),
    "e5m2_no_inf": ("else if (expo == 0x1f) v = frac ? NAN : INFINITY;", "else if (expo == 0x1f) v = NAN;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = SRC.read_text()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib_file = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", str(mutated),
                    "-o", str(lib_file), "-lm"], check=True)
    code = RUNNER.format(root=str(TESTS.parent), tests=str(TESTS), lib=str(lib_file))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, PYTHONDONTWRITEBYTECODE="1"))
    if r.returncode < 0:
        return  # the mutant crashed on the pins' inputs: caught
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("CAUGHT")][-1]
    caught = [c for c in line[len("CAUGHT"):].strip().split(",") if c]
    assert caught, f"no pin caught mutant {name}"
